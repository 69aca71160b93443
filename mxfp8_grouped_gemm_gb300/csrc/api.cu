// C-ABI entry points: argument validation, the layout of the caller-owned
// saved/workspace buffers, and the launch sequence of the forward and backward
// passes.  Nothing here allocates or synchronises; every call only enqueues
// work on the caller's stream.
#include <atomic>
#include <climits>
#include <cstring>

#include "common.cuh"
#include "api_common.h"
#include "kernels.h"

namespace mxg {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

using namespace api;

// CTA-pair GEMM tiles (256 x 256 over two SMs) for the MLP's GEMMs whose
// output width is a multiple of 256.  Measured on GB300 (Mixtral layer): the
// fwd+bwd step drops from 16.0 to 15.5 ms against single-SM 128 x 256 tiles,
// the extra row padding (groups 256-aligned) included.
constexpr bool kUsePairTiles = true;
// The MLP's per-expert row layout: every group starts on a multiple of the
// GEMM tile height (256 rows with CTA pairs, else 128), so
// sum_e roundup(m_e, A) <= roundup(T*k, A) + A*E.
constexpr int kMlpAlign = kUsePairTiles ? 256 : 128;
inline int64_t row_cap(int64_t T, int64_t k, int64_t E) { return align_up(T * k, kMlpAlign) + kMlpAlign * E; }
// The standalone grouped quantiser's group count limit (its padding kernel is
// one block of 1024 threads, each taking a run of groups).
constexpr int kMaxQuantGroups = 1 << 20;

// Whether a bf16-output GEMM with contraction length K sums each token's k
// rows in its epilogue (the tile that stores a token's last row reads the other
// k - 1 back through L2) instead of leaving that to the combine kernel.  The
// reads wait on L2 one after another, which a long mainloop hides and a short
// one does not.  Measured on GB300: Mixtral (k = 2, K = 14336 and 28672) fused
// saves ~0.07 ms per step; 64 experts top-8 (K = 1024 and 2048) fused ran the
// down GEMM at 0.13 of peak.  Rule: fuse when the tile has at least 32 K steps
// of 128 per extra row (k = 1 is a plain scatter: always fused), or when the
// layer routes at most 4096 rows: such a step is bound by its launches (the
// 256-token, top-2 shape runs 0.39 ms fused against 0.47 ms with the kernel).
inline bool fuse_combine(int64_t k, int64_t K, int64_t R) {
  return k == 1 || K / 128 >= 32 * (k - 1) || R <= 4096;
}


// Byte offsets of every buffer inside `saved` and `workspace`.
struct Plan {
  int64_t T, H, I, E, k, R, Rc;
  // saved (forward -> backward)
  int64_t poff, prow_src, prow_of_src, probs_perm, gu, xc, sxc, hc, shc, wguT, swguT, wdT, swdT, saved_bytes,
      saved_cached_bytes;
  // forward scratch
  int64_t counts, bases, offsets, xq, sxq, hq, shq, wgu, swgu, wd, swd, yperm, cmb_cnt, fwd_bytes;
  // backward scratch
  int64_t dyq, sdyq, dyc, sdyc, dguq, sdguq, dguc, sdguc, dxperm, dp, cmb_cnt_b, bwd_bytes;
  int64_t dp_ld;

  Plan(int64_t T_, int64_t H_, int64_t I_, int64_t E_, int64_t k_) : T(T_), H(H_), I(I_), E(E_), k(k_) {
    R = T * k;
    Rc = row_cap(T, k, E);
    Carver s;
    poff = s.take(4 * (E + 1));
    prow_src = s.take(4 * Rc);
    prow_of_src = s.take(4 * R);
    probs_perm = s.take(4 * Rc);
    gu = s.take(2 * Rc * 2 * I);
    xc = s.take(H * Rc);
    sxc = s.take(H * Rc / 32);
    hc = s.take(I * Rc);
    shc = s.take(I * Rc / 32);
    wguT = s.take(E * H * 2 * I);
    swguT = s.take(E * H * 2 * I / 32);
    wdT = s.take(E * I * H);
    swdT = s.take(E * I * H / 32);
    saved_bytes = s.off;
    saved_cached_bytes = wguT;   // the transposed weights are the last part of `saved`

    Carver f;
    const int64_t nblk = permute_num_blocks(static_cast<int>(R));
    counts = f.take(4 * nblk * E);
    bases = f.take(4 * nblk * E);
    offsets = f.take(4 * (E + 1));
    xq = f.take(Rc * H);
    sxq = f.take(Rc * H / 32);
    hq = f.take(Rc * I);
    shq = f.take(Rc * I / 32);
    wgu = f.take(E * 2 * I * H);
    swgu = f.take(E * 2 * I * H / 32);
    wd = f.take(E * H * I);
    swd = f.take(E * H * I / 32);
    yperm = f.take(2 * Rc * H);
    cmb_cnt = f.take(4 * T * (H / 128) * 2);
    fwd_bytes = f.off;

    Carver b;
    dp_ld = dswiglu_partials(static_cast<int>(I));
    dyq = b.take(Rc * H);
    sdyq = b.take(Rc * H / 32);
    dyc = b.take(H * Rc);
    sdyc = b.take(H * Rc / 32);
    dguq = b.take(Rc * 2 * I);
    sdguq = b.take(Rc * 2 * I / 32);
    dguc = b.take(2 * I * Rc);
    sdguc = b.take(2 * I * Rc / 32);
    dxperm = b.take(2 * Rc * H);
    dp = b.take(4 * Rc * dp_ld);
    cmb_cnt_b = b.take(4 * T * (H / 128) * 2);
    bwd_bytes = b.off;
  }
  int64_t ws_bytes() const { return fwd_bytes > bwd_bytes ? fwd_bytes : bwd_bytes; }
};

// Byte offsets inside a weight cache: the four MXFP8 weight tensors (codes,
// then tensor-core scales) in the order the forward and backward read them.
struct WPlan {
  int64_t wgu, swgu, wd, swd, wguT, swguT, wdT, swdT, bytes;
  WPlan(int64_t H, int64_t I, int64_t E) {
    Carver c;
    wgu = c.take(E * 2 * I * H);
    swgu = c.take(E * 2 * I * H / 32);
    wd = c.take(E * H * I);
    swd = c.take(E * H * I / 32);
    wguT = c.take(E * H * 2 * I);
    swguT = c.take(E * H * 2 * I / 32);
    wdT = c.take(E * I * H);
    swdT = c.take(E * I * H / 32);
    bytes = c.off;
  }
};




bool mlp_shape_ok(int T, int H, int I, int E, int k) {
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return false;
  if (H % 128 || I % 128) return false;
  if (k > E || E > 256 || k > 32) return false;
  // padded row indices are int32: T*k rows plus up to 256 padding rows per group
  if (static_cast<int64_t>(T) * k + 256 * (static_cast<int64_t>(E) + 1) > INT32_MAX) return false;
  return true;
}

// F4: W_gate_up and W_down, both orientations in one pass each: row-wise (the
// forward GEMMs' B, MX along H / I) and column-wise (the dgrad GEMMs' B, MX
// along 2I / H; skipped when q_guT is null).
cudaError_t launch_weight_quant(const uint16_t* w_gate_up, const uint16_t* w_down, int64_t H, int64_t I, int64_t E,
                                uint8_t* q_gu, uint8_t* s_gu, uint8_t* q_guT, uint8_t* s_guT, uint8_t* q_d,
                                uint8_t* s_d, uint8_t* q_dT, uint8_t* s_dT, cudaStream_t s) {
  QuantParams wq{};
  wq.x = w_gate_up;
  wq.ld_x = H;
  wq.x_batch_stride = 2 * I * H;
  wq.src_div = 1;
  wq.rows = static_cast<int32_t>(2 * I);
  wq.cols = static_cast<int32_t>(H);
  wq.batch = static_cast<int32_t>(E);
  wq.q_row = q_gu;
  wq.s_row = s_gu;
  wq.sf_row_rows = E * 2 * I;
  if (q_guT != nullptr) {
    wq.q_col = q_guT;
    wq.s_col = s_guT;
    wq.ld_col = 2 * I;
    wq.sf_col_rows = E * H;
  }
  wq.layout = MXG_LAYOUT_MMA;
  QuantParams dq = wq;
  dq.x = w_down;
  dq.ld_x = I;
  dq.x_batch_stride = H * I;
  dq.rows = static_cast<int32_t>(H);
  dq.cols = static_cast<int32_t>(I);
  dq.q_row = q_d;
  dq.s_row = s_d;
  dq.sf_row_rows = E * H;
  if (q_dT != nullptr) {
    dq.q_col = q_dT;
    dq.s_col = s_dT;
    dq.ld_col = H;
    dq.sf_col_rows = E * I;
  }
  return launch_quant2(wq, dq, s);
}

}  // namespace
}  // namespace mxg

using namespace mxg;

extern "C" {

const char* mxg_status_string(int status) {
  switch (status) {
    case MXG_OK: return "ok";
    case MXG_ERR_ARG: return "invalid argument (null pointer, non-positive size or bad enum)";
    case MXG_ERR_SHAPE: return "shape violates the call's divisibility rules";
    case MXG_ERR_ALIGN: return "device pointer not 32-byte aligned";
    case MXG_ERR_ARCH: return "device is not sm_103 (GB300)";
    case MXG_ERR_WORKSPACE: return "scratch or saved buffer too small";
    case MXG_ERR_CUDA: return "CUDA runtime error or kernel launch failure";
    case MXG_ERR_EXPERT_ID: return "expert id outside [0, E)";
    case MXG_ERR_OFFSETS: return "group offsets not monotone, not 128-aligned or beyond capacity";
    case MXG_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case MXG_ERR_INDEX: return "a row index outside the buffer it indexes";
    default: return "unknown status";
  }
}

int mxg_device_supported(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return 0;
  return (major == 10 && minor == 3) ? 1 : 0;
}

uint64_t mxg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int mxg_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs, void* stream) {
  NvtxRange nvtx("mxg.route_topk");
  if (!logits || !ids || !probs) return MXG_ERR_ARG;
  if (T <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (k > E || E > 256 || k > 32) return MXG_ERR_SHAPE;
  if (!aligned32(logits) || !aligned32(ids) || !aligned32(probs)) return MXG_ERR_ALIGN;
  return cuda_status(launch_topk(logits, T, E, k, ids, probs, static_cast<cudaStream_t>(stream)));
}

size_t mxg_route_permute_workspace_bytes(int T, int k, int E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  const int64_t R = static_cast<int64_t>(T) * k;     // routed entries; must fit the kernels' int32 indices
  if (R > INT32_MAX) return 0;
  const int64_t nblk = permute_num_blocks(static_cast<int>(R));
  return static_cast<size_t>(align_up(4 * nblk * E, kAlign) * 2 + align_up(4 * (E + 1), kAlign));
}

int mxg_route_permute(const int32_t* ids, int T, int k, int E, int32_t* split_sizes, int32_t* src_of_row,
                      int32_t* row_of_src, int32_t* padded_offsets, void* ws, size_t ws_bytes,
                      int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.route_permute");
  if (!ids || !split_sizes || !src_of_row || !row_of_src || !padded_offsets || !ws || !dev_status)
    return MXG_ERR_ARG;
  if (T <= 0 || k <= 0 || E <= 0) return MXG_ERR_ARG;
  if (k > E || E > 256) return MXG_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(T) * k;
  if (R > INT32_MAX) return MXG_ERR_SHAPE;           // row indices are int32
  if (!aligned32(ids) || !aligned32(split_sizes) || !aligned32(src_of_row) || !aligned32(row_of_src) ||
      !aligned32(padded_offsets) || !aligned32(ws))
    return MXG_ERR_ALIGN;
  if (ws_bytes < mxg_route_permute_workspace_bytes(T, k, E)) return MXG_ERR_WORKSPACE;
  const int64_t nblk = permute_num_blocks(static_cast<int>(R));
  PermuteParams p{};
  p.ids = ids;
  p.R = static_cast<int32_t>(R);
  p.E = E;
  p.counts = at<int32_t>(ws, 0);
  p.bases = at<int32_t>(ws, align_up(4 * nblk * E, kAlign));
  p.offsets = at<int32_t>(ws, 2 * align_up(4 * nblk * E, kAlign));
  p.padded_offsets = padded_offsets;
  p.pad = 128;
  p.split_sizes = split_sizes;
  p.src_of_row = src_of_row;
  p.row_of_src = row_of_src;
  p.status = dev_status;
  return cuda_status(launch_permute(p, static_cast<cudaStream_t>(stream)));
}

int mxg_mxfp8_quantize(const uint16_t* x, int rows, int cols, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                       uint8_t* s_col, int layout, void* stream) {
  NvtxRange nvtx("mxg.mxfp8_quantize");
  if (!x || rows <= 0 || cols <= 0) return MXG_ERR_ARG;
  if (layout != MXG_LAYOUT_CANONICAL && layout != MXG_LAYOUT_MMA) return MXG_ERR_ARG;
  if ((q_row == nullptr) != (s_row == nullptr) || (q_col == nullptr) != (s_col == nullptr)) return MXG_ERR_ARG;
  if (!q_row && !q_col) return MXG_ERR_ARG;
  // the kernel tiles 32 rows x 128 columns
  if (rows % 32 || cols % 128) return MXG_ERR_SHAPE;
  if (layout == MXG_LAYOUT_MMA && rows % 128) return MXG_ERR_SHAPE;
  if (!aligned32(x) || (q_row && !aligned32(q_row)) || (q_col && !aligned32(q_col))) return MXG_ERR_ALIGN;
  QuantParams p{};
  p.x = x;
  p.ld_x = cols;
  p.x_batch_stride = 0;
  p.src_div = 1;
  p.rows = rows;
  p.cols = cols;
  p.batch = 1;
  p.q_row = q_row;
  p.s_row = s_row;
  p.sf_row_rows = rows;
  p.q_col = q_col;
  p.s_col = s_col;
  p.ld_col = rows;
  p.sf_col_rows = cols;
  p.layout = layout;
  return cuda_status(launch_quant(p, static_cast<cudaStream_t>(stream)));
}

size_t mxg_mxfp8_grouped_rows_capacity(int rows, int groups, int layout) {
  if (rows <= 0 || groups <= 0 || groups > kMaxQuantGroups) return 0;
  if (layout != MXG_LAYOUT_CANONICAL && layout != MXG_LAYOUT_MMA) return 0;
  const int64_t al = layout == MXG_LAYOUT_MMA ? 128 : 32;
  const int64_t cap = align_up(rows, al) + al * groups;
  return cap > INT32_MAX ? 0 : static_cast<size_t>(cap);
}

int mxg_mxfp8_quantize_grouped(const uint16_t* x, int rows, int cols, const int32_t* group_offsets, int groups,
                               int32_t* padded_offsets, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                               uint8_t* s_col, int layout, int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.mxfp8_quantize_grouped");
  if (!x || !group_offsets || !padded_offsets || !dev_status || rows <= 0 || cols <= 0 || groups <= 0)
    return MXG_ERR_ARG;
  if (layout != MXG_LAYOUT_CANONICAL && layout != MXG_LAYOUT_MMA) return MXG_ERR_ARG;
  if ((q_row == nullptr) != (s_row == nullptr) || (q_col == nullptr) != (s_col == nullptr)) return MXG_ERR_ARG;
  if (!q_row && !q_col) return MXG_ERR_ARG;
  if (cols % 128 || groups > kMaxQuantGroups) return MXG_ERR_SHAPE;
  const int64_t cap = static_cast<int64_t>(mxg_mxfp8_grouped_rows_capacity(rows, groups, layout));
  if (cap == 0) return MXG_ERR_SHAPE;
  if (!aligned32(x) || !aligned32(group_offsets) || !aligned32(padded_offsets) || (q_row && !aligned32(q_row)) ||
      (q_col && !aligned32(q_col)))
    return MXG_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int al = layout == MXG_LAYOUT_MMA ? 128 : 32;
  MXG_TRY(launch_group_pad(group_offsets, groups, rows, al, cap, padded_offsets, dev_status, s));
  QuantParams p{};
  p.x = x;
  p.ld_x = cols;
  p.src_div = 1;
  p.rows = static_cast<int32_t>(cap);
  p.cols = cols;
  p.batch = 1;
  p.rows_valid = padded_offsets + groups;
  p.grp_off = group_offsets;
  p.grp_poff = padded_offsets;
  p.groups = groups;
  p.q_row = q_row;
  p.s_row = s_row;
  p.sf_row_rows = cap;
  p.q_col = q_col;
  p.s_col = s_col;
  p.ld_col = cap;
  p.sf_col_rows = cols;
  p.layout = layout;
  return cuda_status(launch_quant(p, s));
}

int mxg_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes, const int32_t* index, int div,
                    int64_t rows, void* dst, int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.gather_rows");
  if (!src || !index || !dst || !dev_status || src_rows <= 0 || row_bytes <= 0 || div <= 0 || rows <= 0)
    return MXG_ERR_ARG;
  if (row_bytes % 4) return MXG_ERR_SHAPE;
  if (src_rows > static_cast<int64_t>(INT32_MAX) * div || rows > INT32_MAX) return MXG_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(index) |
       reinterpret_cast<uintptr_t>(dev_status)) & 3u)
    return MXG_ERR_ALIGN;
  return cuda_status(launch_gather_rows(src, src_rows, row_bytes, index, div, rows, dst, dev_status,
                                        static_cast<cudaStream_t>(stream)));
}

int mxg_combine(const uint16_t* rows, int64_t src_rows, const int32_t* row_of_src, int T, int k, int H, uint16_t* y,
                int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.combine");
  if (!rows || !row_of_src || !y || !dev_status || src_rows <= 0 || T <= 0 || k <= 0 || H <= 0) return MXG_ERR_ARG;
  if (H % 8 || k > 32) return MXG_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(y)) & 15u) return MXG_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(row_of_src) | reinterpret_cast<uintptr_t>(dev_status)) & 3u) return MXG_ERR_ALIGN;
  return cuda_status(launch_combine(rows, row_of_src, T, k, H, y, static_cast<cudaStream_t>(stream), src_rows,
                                    dev_status));
}

int mxg_grouped_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                     const int32_t* padded_offsets, int E, int m_cap, int N, int K, uint16_t* d,
                     int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.grouped_gemm");
  if (!a || !sa || !b || !sb || !padded_offsets || !d || !dev_status) return MXG_ERR_ARG;
  if (E <= 0 || m_cap <= 0 || N <= 0 || K <= 0) return MXG_ERR_ARG;
  if (E > 256 || K % 128 || N % 128 || m_cap % 128) return MXG_ERR_SHAPE;
  if (!aligned32(a) || !aligned32(sa) || !aligned32(b) || !aligned32(sb) || !aligned32(d) ||
      !aligned32(padded_offsets))
    return MXG_ERR_ALIGN;
  GemmArgs g{};
  g.epi = EPI_BF16;
  g.kgroup = false;
  g.a = a;
  g.sa = sa;
  g.a_rows = m_cap;
  g.a_cols = K;
  g.b = b;
  g.sb = sb;
  g.b_rows = static_cast<int64_t>(E) * N;
  g.b_cols = K;
  g.poff = padded_offsets;
  g.E = E;
  g.M = m_cap;
  g.N = N;
  g.K = K;
  g.b_rows_per_expert = N;
  g.d = d;
  g.ldd = N;
  g.status = dev_status;
  g.tiles_upper = static_cast<int64_t>(m_cap / 128) * (N / gemm_pick_bn(EPI_BF16, N));
  return cuda_status(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

int mxg_debug_grouped_gemm_stall(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                  const int32_t* padded_offsets, int E, int m_cap, int N, int K, uint16_t* d,
                                  uint64_t wait_limit_ns, int32_t* dev_status, void* stream) {
  if (!a || !sa || !b || !sb || !padded_offsets || !d || !dev_status) return MXG_ERR_ARG;
  if (E <= 0 || m_cap <= 0 || N <= 0 || K <= 0 || wait_limit_ns == 0) return MXG_ERR_ARG;
  if (E > 256 || K % 128 || N % 128 || m_cap % 128) return MXG_ERR_SHAPE;
  if (!aligned32(a) || !aligned32(sa) || !aligned32(b) || !aligned32(sb) || !aligned32(d) ||
      !aligned32(padded_offsets))
    return MXG_ERR_ALIGN;
  GemmArgs g{};
  g.epi = EPI_BF16;
  g.a = a;
  g.sa = sa;
  g.a_rows = m_cap;
  g.a_cols = K;
  g.b = b;
  g.sb = sb;
  g.b_rows = static_cast<int64_t>(E) * N;
  g.b_cols = K;
  g.poff = padded_offsets;
  g.E = E;
  g.M = m_cap;
  g.N = N;
  g.K = K;
  g.b_rows_per_expert = N;
  g.d = d;
  g.ldd = N;
  g.status = dev_status;
  g.tiles_upper = static_cast<int64_t>(m_cap / 128) * (N / gemm_pick_bn(EPI_BF16, N));
  g.wait_limit_ns = wait_limit_ns;
  g.debug_stall = 1;
  return cuda_status(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

int mxg_grouped_gemm_wgrad(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                           const int32_t* padded_offsets, int E, int M, int N, int t_cap, uint16_t* d,
                           int32_t* dev_status, void* stream) {
  NvtxRange nvtx("mxg.grouped_gemm_wgrad");
  if (!a || !sa || !b || !sb || !padded_offsets || !d || !dev_status) return MXG_ERR_ARG;
  if (E <= 0 || M <= 0 || N <= 0 || t_cap <= 0) return MXG_ERR_ARG;
  if (E > 256 || M % 128 || N % 128 || t_cap % 128) return MXG_ERR_SHAPE;
  if (!aligned32(a) || !aligned32(sa) || !aligned32(b) || !aligned32(sb) || !aligned32(d) ||
      !aligned32(padded_offsets))
    return MXG_ERR_ALIGN;
  GemmArgs g{};
  g.epi = EPI_BF16;
  g.kgroup = true;
  g.a = a;
  g.sa = sa;
  g.a_rows = M;
  g.a_cols = t_cap;
  g.b = b;
  g.sb = sb;
  g.b_rows = N;
  g.b_cols = t_cap;
  g.poff = padded_offsets;
  g.E = E;
  g.M = M;
  g.N = N;
  g.d = d;
  g.ldd = N;
  g.status = dev_status;
  g.tiles_upper = static_cast<int64_t>(E) * (M / 128) * (N / gemm_pick_bn(EPI_BF16, N));
  return cuda_status(launch_gemm(g, static_cast<cudaStream_t>(stream)));
}

int mxg_mlp_group_align(void) { return kMlpAlign; }

size_t mxg_mlp_row_capacity(int T, int k, int E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  return static_cast<size_t>(row_cap(T, k, E));
}

size_t mxg_mlp_saved_bytes(int T, int H, int I, int E, int k) {
  if (!mlp_shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(Plan(T, H, I, E, k).saved_bytes);
}

size_t mxg_mlp_workspace_bytes(int T, int H, int I, int E, int k) {
  if (!mlp_shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(Plan(T, H, I, E, k).ws_bytes());
}

size_t mxg_mlp_saved_bytes_cached(int T, int H, int I, int E, int k) {
  if (!mlp_shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(Plan(T, H, I, E, k).saved_cached_bytes);
}

size_t mxg_mlp_weight_cache_bytes(int H, int I, int E) {
  if (!mlp_shape_ok(1, H, I, E, 1)) return 0;
  return static_cast<size_t>(WPlan(H, I, E).bytes);
}

const void* mxg_mlp_weight_cache_view(const void* cache, int H, int I, int E, int which) {
  if (!cache || !mlp_shape_ok(1, H, I, E, 1)) return nullptr;
  const WPlan wp(H, I, E);
  switch (which) {
    case 0: return at<uint8_t>(cache, wp.wgu);
    case 1: return at<uint8_t>(cache, wp.swgu);
    case 2: return at<uint8_t>(cache, wp.wd);
    case 3: return at<uint8_t>(cache, wp.swd);
    case 4: return at<uint8_t>(cache, wp.wguT);
    case 5: return at<uint8_t>(cache, wp.swguT);
    case 6: return at<uint8_t>(cache, wp.wdT);
    case 7: return at<uint8_t>(cache, wp.swdT);
    default: return nullptr;
  }
}

int mxg_mlp_quantize_weights(const uint16_t* w_gate_up, const uint16_t* w_down, int H, int I, int E, void* cache,
                             size_t cache_bytes, void* stream) {
  NvtxRange nvtx("mxg.quantize_weights");
  if (!w_gate_up || !w_down || !cache) return MXG_ERR_ARG;
  if (H <= 0 || I <= 0 || E <= 0) return MXG_ERR_ARG;
  if (!mlp_shape_ok(1, H, I, E, 1)) return MXG_ERR_SHAPE;
  if (!aligned32(w_gate_up) || !aligned32(w_down) || !aligned32(cache)) return MXG_ERR_ALIGN;
  const WPlan wp(H, I, E);
  if (cache_bytes < static_cast<size_t>(wp.bytes)) return MXG_ERR_WORKSPACE;
  return cuda_status(launch_weight_quant(w_gate_up, w_down, H, I, E, at<uint8_t>(cache, wp.wgu),
                                         at<uint8_t>(cache, wp.swgu), at<uint8_t>(cache, wp.wguT),
                                         at<uint8_t>(cache, wp.swguT), at<uint8_t>(cache, wp.wd),
                                         at<uint8_t>(cache, wp.swd), at<uint8_t>(cache, wp.wdT),
                                         at<uint8_t>(cache, wp.swdT), static_cast<cudaStream_t>(stream)));
}

const void* mxg_mlp_saved_view(const void* saved, int T, int H, int I, int E, int k, int which) {
  if (!saved || !mlp_shape_ok(T, H, I, E, k)) return nullptr;
  const Plan pl(T, H, I, E, k);
  switch (which) {
    case 0: return at<uint8_t>(saved, pl.gu);
    case 1: return at<uint8_t>(saved, pl.poff);
    case 2: return at<uint8_t>(saved, pl.prow_of_src);
    case 3: return at<uint8_t>(saved, pl.xc);
    case 4: return at<uint8_t>(saved, pl.sxc);
    case 5: return at<uint8_t>(saved, pl.hc);
    case 6: return at<uint8_t>(saved, pl.shc);
    default: return nullptr;
  }
}

const void* mxg_mlp_workspace_view(const void* workspace, int T, int H, int I, int E, int k, int which) {
  if (!workspace || !mlp_shape_ok(T, H, I, E, k)) return nullptr;
  const Plan pl(T, H, I, E, k);
  switch (which) {
    case 0: return at<uint8_t>(workspace, pl.dguq);
    case 1: return at<uint8_t>(workspace, pl.sdguq);
    case 2: return at<uint8_t>(workspace, pl.dguc);
    case 3: return at<uint8_t>(workspace, pl.sdguc);
    case 4: return at<uint8_t>(workspace, pl.yperm);
    case 5: return at<uint8_t>(workspace, pl.dxperm);
    default: return nullptr;
  }
}

// xq_pre / xs_pre (nullable): x already quantised row-wise (codes [T][H] and
// canonical scales [T][H/32], one row per token; used with k = 1); the x stage
// then places those rows into the padded layout instead of quantising
// (inference only: no token-column codes of x exist for a backward).
static int fwd_impl(const mxg_mlp_fwd_args* A, int stage, void* stream, const uint8_t* xq_pre = nullptr,
                    const uint8_t* xs_pre = nullptr) {
  if (!A) return MXG_ERR_ARG;
  const int T = A->T, H = A->H, I = A->I, E = A->E, k = A->k;
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!mlp_shape_ok(T, H, I, E, k)) return MXG_ERR_SHAPE;
  const bool cached = A->weight_cache != nullptr;
  const bool pre = xq_pre != nullptr;
  if (pre && (xs_pre == nullptr || A->save_for_backward != 0)) return MXG_ERR_ARG;
  if ((!A->x && !pre) || !A->ids || !A->probs || (!cached && (!A->w_gate_up || !A->w_down)) || !A->y || !A->split_sizes ||
      !A->saved || !A->workspace || !A->dev_status)
    return MXG_ERR_ARG;
  if (!aligned32(A->x) || !aligned32(A->ids) || !aligned32(A->probs) || !aligned32(A->w_gate_up) ||
      !aligned32(A->w_down) || !aligned32(A->y) || !aligned32(A->split_sizes) || !aligned32(A->saved) ||
      !aligned32(A->workspace) || !aligned32(A->weight_cache))
    return MXG_ERR_ALIGN;
  const Plan pl(T, H, I, E, k);
  const WPlan wp(H, I, E);
  if (A->saved_bytes < static_cast<uint64_t>(cached ? pl.saved_cached_bytes : pl.saved_bytes) ||
      A->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes()) ||
      (cached && A->weight_cache_bytes < static_cast<uint64_t>(wp.bytes)))
    return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* sv = A->saved;
  void* ws = A->workspace;
  const bool save = A->save_for_backward != 0;
  int32_t* st = A->dev_status;
  const int32_t* poff = at<int32_t>(sv, pl.poff);
  auto run = [stage](int id) { return stage < 0 || stage == id; };
  // the forward GEMMs' MXFP8 weights: from the cache, or quantised below into the workspace
  const uint8_t* wgu = cached ? at<uint8_t>(A->weight_cache, wp.wgu) : at<uint8_t>(ws, pl.wgu);
  const uint8_t* swgu = cached ? at<uint8_t>(A->weight_cache, wp.swgu) : at<uint8_t>(ws, pl.swgu);
  const uint8_t* wd = cached ? at<uint8_t>(A->weight_cache, wp.wd) : at<uint8_t>(ws, pl.wd);
  const uint8_t* swd = cached ? at<uint8_t>(A->weight_cache, wp.swd) : at<uint8_t>(ws, pl.swd);

  // F2: permute (histogram -> scan -> stable scatter) into the padded layout
  if (run(MXG_FWD_PERMUTE)) {
  NvtxRange nvtx("mxg.fwd.permute");
  MXG_TRY(cudaMemsetAsync(at<int32_t>(sv, pl.prow_src), 0xFF, 4 * pl.Rc, s));
  PermuteParams pp{};
  pp.ids = A->ids;
  pp.R = static_cast<int32_t>(pl.R);
  pp.E = E;
  pp.counts = at<int32_t>(ws, pl.counts);
  pp.bases = at<int32_t>(ws, pl.bases);
  pp.offsets = at<int32_t>(ws, pl.offsets);
  pp.padded_offsets = at<int32_t>(sv, pl.poff);
  pp.pad = kMlpAlign;
  pp.split_sizes = A->split_sizes;
  pp.prow_src = at<int32_t>(sv, pl.prow_src);
  pp.prow_of_src = at<int32_t>(sv, pl.prow_of_src);
  pp.status = st;
  MXG_TRY(launch_permute(pp, s));
  }

  // F4: weights, both orientations in one pass (the transposed ones only for
  // backward); nothing to do with a weight cache
  if (run(MXG_FWD_QUANT_WEIGHTS) && !cached) {
    NvtxRange nvtx("mxg.fwd.quant_weights");
    MXG_TRY(launch_weight_quant(A->w_gate_up, A->w_down, H, I, E, at<uint8_t>(ws, pl.wgu), at<uint8_t>(ws, pl.swgu),
                                save ? at<uint8_t>(sv, pl.wguT) : nullptr, at<uint8_t>(sv, pl.swguT),
                                at<uint8_t>(ws, pl.wd), at<uint8_t>(ws, pl.swd),
                                save ? at<uint8_t>(sv, pl.wdT) : nullptr, at<uint8_t>(sv, pl.swdT), s));
  }

  // F3: gather x into the padded per-expert layout and quantise (row-wise along
  // H for the gate-up GEMM; token-column-wise for the gate-up weight gradient)
  if (run(MXG_FWD_QUANT_X) && pre) {
    NvtxRange nvtx("mxg.fwd.place_x");
    MXG_TRY(launch_place_rows(xq_pre, xs_pre, static_cast<int64_t>(T) * k, at<int32_t>(sv, pl.prow_src), pl.Rc,
                              poff + E, H, at<uint8_t>(ws, pl.xq), at<uint8_t>(ws, pl.sxq), pl.Rc, A->probs,
                              at<float>(sv, pl.probs_perm), st, s));
  }
  if (run(MXG_FWD_QUANT_X) && !pre) {
  NvtxRange nvtx("mxg.fwd.quant_x");
  QuantParams xq{};
  xq.x = A->x;
  xq.ld_x = H;
  xq.src_rows = at<int32_t>(sv, pl.prow_src);
  xq.src_div = k;
  xq.probs = A->probs;
  xq.probs_perm = at<float>(sv, pl.probs_perm);
  xq.rows = static_cast<int32_t>(pl.Rc);
  xq.cols = H;
  xq.batch = 1;
  xq.rows_valid = poff + E;
  xq.q_row = at<uint8_t>(ws, pl.xq);
  xq.s_row = at<uint8_t>(ws, pl.sxq);
  xq.sf_row_rows = pl.Rc;
  if (save) {
    xq.q_col = at<uint8_t>(sv, pl.xc);
    xq.s_col = at<uint8_t>(sv, pl.sxc);
    xq.ld_col = pl.Rc;
    xq.sf_col_rows = H;
  }
  xq.layout = MXG_LAYOUT_MMA;
  MXG_TRY(launch_quant(xq, s));
  }

  // F5: gate-up grouped GEMM + ScaledSwiGLU + MXFP8 re-quantisation of h
  if (run(MXG_FWD_GATE_UP)) {
  NvtxRange nvtx("mxg.fwd.gate_up");
  GemmArgs g{};
  g.epi = EPI_SWIGLU;
  g.pair = kUsePairTiles;
  g.a = at<uint8_t>(ws, pl.xq);
  g.sa = at<uint8_t>(ws, pl.sxq);
  g.a_rows = pl.Rc;
  g.a_cols = H;
  g.b = wgu;
  g.sb = swgu;
  g.b_rows = pl.E * 2 * I;
  g.b_cols = H;
  g.poff = poff;
  g.E = E;
  g.M = static_cast<int32_t>(pl.Rc);
  g.N = 2 * I;
  g.K = H;
  g.b_rows_per_expert = 2 * I;
  g.I = I;
  g.probs_perm = at<float>(sv, pl.probs_perm);
  g.gu_save = save ? at<uint16_t>(sv, pl.gu) : nullptr;
  g.q_out = at<uint8_t>(ws, pl.hq);
  g.s_out = at<uint8_t>(ws, pl.shq);
  g.q_out_ld = I;
  g.s_out_rows = pl.Rc;
  if (save) {
    g.qc_out = at<uint8_t>(sv, pl.hc);
    g.sc_out = at<uint8_t>(sv, pl.shc);
    g.qc_ld = pl.Rc;
    g.sc_rows = I;
  }
  g.status = st;
  g.tiles_upper = (pl.Rc / kMlpAlign) * (I / 128);
  MXG_TRY(launch_gemm(g, s));
  }

  // F6: down grouped GEMM
  if (run(MXG_FWD_DOWN)) {
  NvtxRange nvtx("mxg.fwd.down");
  GemmArgs d{};
  d.epi = EPI_BF16;
  d.pair = kUsePairTiles && H % 256 == 0;
  d.a = at<uint8_t>(ws, pl.hq);
  d.sa = at<uint8_t>(ws, pl.shq);
  d.a_rows = pl.Rc;
  d.a_cols = I;
  d.b = wd;
  d.sb = swd;
  d.b_rows = pl.E * H;
  d.b_cols = I;
  d.poff = poff;
  d.E = E;
  d.M = static_cast<int32_t>(pl.Rc);
  d.N = H;
  d.K = I;
  d.b_rows_per_expert = H;
  d.d = at<uint16_t>(ws, pl.yperm);
  d.ldd = H;
  if (fuse_combine(k, I, pl.R)) {
    // F7 fused: the thread that stores the last of a token's k rows sums them into y
    MXG_TRY(cudaMemsetAsync(at<int32_t>(ws, pl.cmb_cnt), 0, 4 * pl.T * (H / 128) * 2, s));
    d.cmb_out = A->y;
    d.cmb_prow_src = at<int32_t>(sv, pl.prow_src);
    d.cmb_prow_of_src = at<int32_t>(sv, pl.prow_of_src);
    d.cmb_count = at<int32_t>(ws, pl.cmb_cnt);
    d.cmb_k = k;
  }
  d.status = st;
  d.tiles_upper = d.pair ? (pl.Rc / 256) * (H / 256) : (pl.Rc / 128) * (H / gemm_pick_bn(EPI_BF16, H));
  MXG_TRY(launch_gemm(d, s));
  }

  // F7: y[t] = sum_j Y[row(t, j)] (fused into the down GEMM above for long contractions)
  if (run(MXG_FWD_COMBINE) && !fuse_combine(k, I, pl.R)) {
    NvtxRange nvtx("mxg.fwd.combine");
    MXG_TRY(launch_combine(at<uint16_t>(ws, pl.yperm), at<int32_t>(sv, pl.prow_of_src), static_cast<int>(pl.T),
                           static_cast<int>(k), static_cast<int>(H), A->y, s));
  }
  return MXG_OK;
}

int mxg_grouped_mlp_fwd(const mxg_mlp_fwd_args* A, void* stream) { return fwd_impl(A, -1, stream); }

int mxg_grouped_mlp_fwd_stage(const mxg_mlp_fwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_FWD_NUM_STAGES) return MXG_ERR_ARG;
  return fwd_impl(A, stage, stream);
}

static int bwd_impl(const mxg_mlp_bwd_args* A, int stage, void* stream) {
  if (!A) return MXG_ERR_ARG;
  const int T = A->T, H = A->H, I = A->I, E = A->E, k = A->k;
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!mlp_shape_ok(T, H, I, E, k)) return MXG_ERR_SHAPE;
  const bool cached = A->weight_cache != nullptr;
  const bool main_grad = A->main_grad_gate_up != nullptr || A->main_grad_down != nullptr;
  if (main_grad && (!A->main_grad_gate_up || !A->main_grad_down)) return MXG_ERR_ARG;
  if (!A->dy || !A->saved || !A->dx || (!main_grad && (!A->dw_gate_up || !A->dw_down)) || !A->dprobs ||
      !A->workspace || !A->dev_status)
    return MXG_ERR_ARG;
  if (!aligned32(A->dy) || !aligned32(A->saved) || !aligned32(A->dx) || !aligned32(A->dw_gate_up) ||
      !aligned32(A->dw_down) || !aligned32(A->dprobs) || !aligned32(A->workspace) || !aligned32(A->weight_cache) ||
      !aligned32(A->main_grad_gate_up) || !aligned32(A->main_grad_down))
    return MXG_ERR_ALIGN;
  const Plan pl(T, H, I, E, k);
  const WPlan wp(H, I, E);
  if (A->saved_bytes < static_cast<uint64_t>(cached ? pl.saved_cached_bytes : pl.saved_bytes) ||
      A->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes()) ||
      (cached && A->weight_cache_bytes < static_cast<uint64_t>(wp.bytes)))
    return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* sv = A->saved;
  void* ws = A->workspace;
  int32_t* st = A->dev_status;
  const int32_t* poff = at<int32_t>(sv, pl.poff);
  auto run = [stage](int id) { return stage < 0 || stage == id; };
  // the dgrad GEMMs' MXFP8 weights (MX along the contraction of the backward)
  const void* wsrc = cached ? A->weight_cache : sv;
  const uint8_t* wguT = at<uint8_t>(wsrc, cached ? wp.wguT : pl.wguT);
  const uint8_t* swguT = at<uint8_t>(wsrc, cached ? wp.swguT : pl.swguT);
  const uint8_t* wdT = at<uint8_t>(wsrc, cached ? wp.wdT : pl.wdT);
  const uint8_t* swdT = at<uint8_t>(wsrc, cached ? wp.swdT : pl.swdT);

  // B1: gather dy and quantise (row-wise along H for dgrad, token-column-wise for wgrad)
  if (run(MXG_BWD_QUANT_DY)) {
  NvtxRange nvtx("mxg.bwd.quant_dy");
  QuantParams yq{};
  yq.x = A->dy;
  yq.ld_x = H;
  yq.src_rows = at<int32_t>(sv, pl.prow_src);
  yq.src_div = k;
  yq.rows = static_cast<int32_t>(pl.Rc);
  yq.cols = H;
  yq.batch = 1;
  yq.rows_valid = poff + E;
  yq.q_row = at<uint8_t>(ws, pl.dyq);
  yq.s_row = at<uint8_t>(ws, pl.sdyq);
  yq.sf_row_rows = pl.Rc;
  yq.q_col = at<uint8_t>(ws, pl.dyc);
  yq.s_col = at<uint8_t>(ws, pl.sdyc);
  yq.ld_col = pl.Rc;
  yq.sf_col_rows = H;
  yq.layout = MXG_LAYOUT_MMA;
  MXG_TRY(launch_quant(yq, s));
  }

  // B2: dH = dY W_down (MX along H) with fused dSwiGLU -> dGU (both orientations), d(prob) partials
  if (run(MXG_BWD_DGRAD_DOWN)) {
  NvtxRange nvtx("mxg.bwd.dgrad_down");
  GemmArgs g{};
  g.epi = EPI_DSWIGLU;
  g.pair = kUsePairTiles && I % 256 == 0;
  g.a = at<uint8_t>(ws, pl.dyq);
  g.sa = at<uint8_t>(ws, pl.sdyq);
  g.a_rows = pl.Rc;
  g.a_cols = H;
  g.b = wdT;
  g.sb = swdT;
  g.b_rows = pl.E * I;
  g.b_cols = H;
  g.poff = poff;
  g.E = E;
  g.M = static_cast<int32_t>(pl.Rc);
  g.N = I;
  g.K = H;
  g.b_rows_per_expert = I;
  g.I = I;
  g.probs_perm = at<float>(sv, pl.probs_perm);
  g.gu_save = const_cast<uint16_t*>(at<uint16_t>(sv, pl.gu));
  g.q_out = at<uint8_t>(ws, pl.dguq);
  g.s_out = at<uint8_t>(ws, pl.sdguq);
  g.q_out_ld = 2 * I;
  g.s_out_rows = pl.Rc;
  g.qc_out = at<uint8_t>(ws, pl.dguc);
  g.sc_out = at<uint8_t>(ws, pl.sdguc);
  g.qc_ld = pl.Rc;
  g.sc_rows = 2 * I;
  g.dp_part = at<float>(ws, pl.dp);
  g.dp_ld = static_cast<int32_t>(pl.dp_ld);
  g.status = st;
  g.tiles_upper = (pl.Rc / (g.pair ? 256 : 128)) * (I / 128);
  MXG_TRY(launch_gemm(g, s));
  }

  // B3: dW_down[e] = dYc^T Hc over the tokens of e (or added into main_grad_down)
  if (run(MXG_BWD_WGRAD_DOWN)) {
  NvtxRange nvtx("mxg.bwd.wgrad_down");
  GemmArgs w{};
  w.epi = main_grad ? EPI_ACC_F32 : EPI_BF16;
  w.kgroup = true;
  w.pair = kUsePairTiles && H % 256 == 0 && I % 256 == 0;   // 256 x 256 output tiles
  w.a = at<uint8_t>(ws, pl.dyc);
  w.sa = at<uint8_t>(ws, pl.sdyc);
  w.a_rows = H;
  w.a_cols = pl.Rc;
  w.b = at<uint8_t>(sv, pl.hc);
  w.sb = at<uint8_t>(sv, pl.shc);
  w.b_rows = I;
  w.b_cols = pl.Rc;
  w.poff = poff;
  w.E = E;
  w.M = H;
  w.N = I;
  w.d = A->dw_down;
  w.dacc = A->main_grad_down;
  w.ldd = I;
  w.status = st;
  w.tiles_upper = w.pair ? pl.E * (H / 256) * (I / 256) : pl.E * (H / 128) * (I / gemm_pick_bn(EPI_BF16, I));
  MXG_TRY(launch_gemm(w, s));
  }

  // B4: dX_perm = dGU W_gate_up (MX along 2I)
  if (run(MXG_BWD_DGRAD_GATE_UP)) {
  NvtxRange nvtx("mxg.bwd.dgrad_gate_up");
  GemmArgs x{};
  x.epi = EPI_BF16;
  x.pair = kUsePairTiles && H % 256 == 0;
  x.a = at<uint8_t>(ws, pl.dguq);
  x.sa = at<uint8_t>(ws, pl.sdguq);
  x.a_rows = pl.Rc;
  x.a_cols = 2 * I;
  x.b = wguT;
  x.sb = swguT;
  x.b_rows = pl.E * H;
  x.b_cols = 2 * I;
  x.poff = poff;
  x.E = E;
  x.M = static_cast<int32_t>(pl.Rc);
  x.N = H;
  x.K = 2 * I;
  x.b_rows_per_expert = H;
  x.d = at<uint16_t>(ws, pl.dxperm);
  x.ldd = H;
  if (fuse_combine(k, 2 * I, pl.R)) {
    // B6 fused: dx[t] summed by the thread that stores the last of the token's rows
    MXG_TRY(cudaMemsetAsync(at<int32_t>(ws, pl.cmb_cnt_b), 0, 4 * pl.T * (H / 128) * 2, s));
    x.cmb_out = A->dx;
    x.cmb_prow_src = at<int32_t>(sv, pl.prow_src);
    x.cmb_prow_of_src = at<int32_t>(sv, pl.prow_of_src);
    x.cmb_count = at<int32_t>(ws, pl.cmb_cnt_b);
    x.cmb_k = k;
  }
  x.status = st;
  x.tiles_upper = x.pair ? (pl.Rc / 256) * (H / 256) : (pl.Rc / 128) * (H / gemm_pick_bn(EPI_BF16, H));
  MXG_TRY(launch_gemm(x, s));
  }

  // B5: dW_gate_up[e] = dGUc^T Xc over the tokens of e (or added into main_grad_gate_up)
  if (run(MXG_BWD_WGRAD_GATE_UP)) {
  NvtxRange nvtx("mxg.bwd.wgrad_gate_up");
  GemmArgs v{};
  v.epi = main_grad ? EPI_ACC_F32 : EPI_BF16;
  v.kgroup = true;
  v.pair = kUsePairTiles && H % 256 == 0;   // 2I is a multiple of 256
  v.a = at<uint8_t>(ws, pl.dguc);
  v.sa = at<uint8_t>(ws, pl.sdguc);
  v.a_rows = 2 * I;
  v.a_cols = pl.Rc;
  v.b = at<uint8_t>(sv, pl.xc);
  v.sb = at<uint8_t>(sv, pl.sxc);
  v.b_rows = H;
  v.b_cols = pl.Rc;
  v.poff = poff;
  v.E = E;
  v.M = 2 * I;
  v.N = H;
  v.d = A->dw_gate_up;
  v.dacc = A->main_grad_gate_up;
  v.ldd = H;
  v.status = st;
  v.tiles_upper = v.pair ? pl.E * (2 * I / 256) * (H / 256) : pl.E * (2 * I / 128) * (H / gemm_pick_bn(EPI_BF16, H));
  MXG_TRY(launch_gemm(v, s));
  }

  // B6, B7: combine dx, reduce d(prob)
  const int32_t* prow_of_src = at<int32_t>(sv, pl.prow_of_src);
  // B6: dx[t] = sum_j dX[row(t, j)] (fused into the dgrad-gate-up GEMM above for long contractions)
  if (run(MXG_BWD_COMBINE_DX) && !fuse_combine(k, 2 * I, pl.R)) {
    NvtxRange nvtx("mxg.bwd.combine_dx");
    MXG_TRY(launch_combine(at<uint16_t>(ws, pl.dxperm), prow_of_src, static_cast<int>(pl.T), static_cast<int>(k),
                           static_cast<int>(H), A->dx, s));
  }
  if (run(MXG_BWD_DPROBS)) {
    NvtxRange nvtx("mxg.bwd.dprobs");
    MXG_TRY(launch_dprob(at<float>(ws, pl.dp), static_cast<int>(pl.dp_ld), prow_of_src, static_cast<int>(pl.R),
                         A->dprobs, s));
  }
  return MXG_OK;
}

int mxg_grouped_mlp_bwd(const mxg_mlp_bwd_args* A, void* stream) { return bwd_impl(A, -1, stream); }

// Pre-grouped tokens: the layer with T = R rows, k = 1 and each row's expert
// given by split_sizes.  The rows are already in expert order, so the
// permute's stable counting sort leaves them in place; the k = 1 combine is
// the scatter of each row back to its own position.
static int64_t grouped_tail(int64_t R, int64_t E) { return align_up(4 * R, kAlign) + align_up(4 * E, kAlign); }

size_t mxg_mlp_grouped_saved_bytes(int R, int H, int I, int E) { return mxg_mlp_saved_bytes(R, H, I, E, 1); }

size_t mxg_mlp_grouped_workspace_bytes(int R, int H, int I, int E) {
  if (!mlp_shape_ok(R, H, I, E, 1)) return 0;
  return static_cast<size_t>(Plan(R, H, I, E, 1).ws_bytes() + grouped_tail(R, E));
}

int mxg_grouped_mlp_fwd_grouped_mx(const mxg_mlp_grouped_fwd_mx_args* G, void* stream) {
  if (!G) return MXG_ERR_ARG;
  const int R = G->R, H = G->H, I = G->I, E = G->E;
  if (R <= 0 || H <= 0 || I <= 0 || E <= 0) return MXG_ERR_ARG;
  if (!mlp_shape_ok(R, H, I, E, 1)) return MXG_ERR_SHAPE;
  if (!G->xq || !G->xs || !G->split_sizes || !G->workspace || !G->dev_status) return MXG_ERR_ARG;
  if (!aligned32(G->xq) || !aligned32(G->split_sizes) || !aligned32(G->workspace)) return MXG_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(G->xs) & 3u) return MXG_ERR_ALIGN;
  const Plan pl(R, H, I, E, 1);
  if (G->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes() + grouped_tail(R, E))) return MXG_ERR_WORKSPACE;
  NvtxRange nvtx("mxg.grouped_mlp_fwd_grouped_mx");
  int32_t* ids = at<int32_t>(G->workspace, pl.ws_bytes());
  int32_t* split_out = at<int32_t>(G->workspace, pl.ws_bytes() + align_up(4 * static_cast<int64_t>(R), kAlign));
  mxg_mlp_fwd_args A{};
  A.T = R;
  A.H = H;
  A.I = I;
  A.E = E;
  A.k = 1;
  A.x = nullptr;
  A.ids = ids;
  A.probs = G->probs;
  A.w_gate_up = G->w_gate_up;
  A.w_down = G->w_down;
  A.y = G->y;
  A.split_sizes = split_out;
  A.saved = G->saved;
  A.saved_bytes = G->saved_bytes;
  A.workspace = G->workspace;
  A.workspace_bytes = static_cast<uint64_t>(pl.ws_bytes());
  A.save_for_backward = 0;
  A.dev_status = G->dev_status;
  A.weight_cache = G->weight_cache;
  A.weight_cache_bytes = G->weight_cache_bytes;
  const int pre = fwd_impl(&A, MXG_FWD_NUM_STAGES, stream, G->xq, G->xs);
  if (pre != MXG_OK) return pre;
  MXG_TRY(launch_expand_splits(G->split_sizes, E, R, ids, G->dev_status, static_cast<cudaStream_t>(stream)));
  return fwd_impl(&A, -1, stream, G->xq, G->xs);
}

int mxg_grouped_mlp_fwd_grouped(const mxg_mlp_grouped_fwd_args* G, void* stream) {
  if (!G) return MXG_ERR_ARG;
  const int R = G->R, H = G->H, I = G->I, E = G->E;
  if (R <= 0 || H <= 0 || I <= 0 || E <= 0) return MXG_ERR_ARG;
  if (!mlp_shape_ok(R, H, I, E, 1)) return MXG_ERR_SHAPE;
  if (!G->split_sizes || !G->workspace || !G->dev_status) return MXG_ERR_ARG;
  if (!aligned32(G->split_sizes) || !aligned32(G->workspace)) return MXG_ERR_ALIGN;
  const Plan pl(R, H, I, E, 1);
  if (G->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes() + grouped_tail(R, E))) return MXG_ERR_WORKSPACE;
  int32_t* ids = at<int32_t>(G->workspace, pl.ws_bytes());
  int32_t* split_out = at<int32_t>(G->workspace, pl.ws_bytes() + align_up(4 * static_cast<int64_t>(R), kAlign));
  mxg_mlp_fwd_args A{};
  A.T = R;
  A.H = H;
  A.I = I;
  A.E = E;
  A.k = 1;
  A.x = G->x;
  A.ids = ids;
  A.probs = G->probs;
  A.w_gate_up = G->w_gate_up;
  A.w_down = G->w_down;
  A.y = G->y;
  A.split_sizes = split_out;
  A.saved = G->saved;
  A.saved_bytes = G->saved_bytes;
  A.workspace = G->workspace;
  A.workspace_bytes = static_cast<uint64_t>(pl.ws_bytes());
  A.save_for_backward = G->save_for_backward;
  A.dev_status = G->dev_status;
  A.weight_cache = G->weight_cache;
  A.weight_cache_bytes = G->weight_cache_bytes;
  // every other argument is checked by the forward before anything is launched
  const int pre = fwd_impl(&A, MXG_FWD_NUM_STAGES, stream);
  if (pre != MXG_OK) return pre;
  MXG_TRY(launch_expand_splits(G->split_sizes, E, R, ids, G->dev_status, static_cast<cudaStream_t>(stream)));
  return fwd_impl(&A, -1, stream);
}

int mxg_grouped_mlp_bwd_stage(const mxg_mlp_bwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_BWD_NUM_STAGES) return MXG_ERR_ARG;
  return bwd_impl(A, stage, stream);
}

}  // extern "C"
