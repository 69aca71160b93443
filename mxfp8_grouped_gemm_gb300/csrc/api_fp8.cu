// C-ABI entry points of the per-tensor FP8 grouped expert MLP: the same route
// -> permute -> gate-up + ScaledSwiGLU -> down -> combine path and its
// backward, with E4M3 operands that carry one power-of-two scale per expert
// tensor ("current scaling": MXFP8's scale rule with the whole tensor as its
// block) instead of MXFP8's scale per 32 values.  It is the FP8 variant the recipe also runs
// ("BioNeMo Uses Grouped Kernels and MXFP8", "Reducing memory pressure with
// MXFP8": FP8 and MXFP8 differ in scaling granularity).
//
// A tensor is one expert's GEMM operand: its weight matrix, or its rows of x,
// h, dy and dGU.  A transposed operand is the same tensor with the same codes,
// so one quantiser pass writes both orientations.  Because a scale depends on
// the whole tensor, h and dGU cannot be quantised inside the GEMM epilogue
// that produces them (MXFP8 can: its blocks lie inside one thread's row): the
// epilogues write them in bf16 and fold their largest magnitude into the
// expert's amax, and a quantiser pass follows.  The tensor-core kind is
// kind::f8f6f4 (no scale factors); the epilogue multiplies the fp32
// accumulators by the two tensors' dequantisation factors.  All GEMMs run as
// 256 x 256 CTA-pair tiles (H, I multiples of 256).
#include <climits>
#include <cstring>

#include "common.cuh"
#include "api_common.h"
#include "kernels.h"

namespace mxg {
namespace {

using namespace api;

constexpr int kGroupAlign = 256;   // CTA-pair tile height





bool shape_ok(int T, int H, int I, int E, int k) {
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return false;
  if (H % 256 || I % 256) return false;
  if (k > E || E > 256 || k > 32) return false;
  // padded row indices are int32: T*k rows plus up to 256 padding rows per group
  if (static_cast<int64_t>(T) * k + 256 * (static_cast<int64_t>(E) + 1) > INT32_MAX) return false;
  return true;
}

// Byte offsets of every buffer inside `saved` and `workspace`.  amax_* are
// fp32 [E]: the largest magnitude of each expert's tensor.
struct PlanF8 {
  int64_t T, H, I, E, k, R, Rc;
  int64_t poff, prow_src, prow_of_src, probs_perm, gu, xqT, hqT, wguT, wdT, amax_x, amax_wgu, amax_wd, amax_h,
      saved_bytes;
  int64_t counts, bases, offsets, xq, wgu, wd, h, hq, yperm, fwd_bytes;
  int64_t dyq, dyqT, dgu, dguq, dguqT, dxperm, dp, amax_dy, amax_dgu, bwd_bytes;
  int64_t dp_ld;

  PlanF8(int64_t T_, int64_t H_, int64_t I_, int64_t E_, int64_t k_) : T(T_), H(H_), I(I_), E(E_), k(k_) {
    R = T * k;
    Rc = align_up(R, kGroupAlign) + kGroupAlign * E;
    Carver s;
    poff = s.take(4 * (E + 1));
    prow_src = s.take(4 * Rc);
    prow_of_src = s.take(4 * R);
    probs_perm = s.take(4 * Rc);
    gu = s.take(2 * Rc * 2 * I);
    xqT = s.take(H * Rc);
    hqT = s.take(I * Rc);
    wguT = s.take(E * H * 2 * I);
    wdT = s.take(E * I * H);
    amax_x = s.take(4 * E);
    amax_wgu = s.take(4 * E);
    amax_wd = s.take(4 * E);
    amax_h = s.take(4 * E);
    saved_bytes = s.off;

    Carver f;
    const int64_t nblk = permute_num_blocks(static_cast<int>(R));
    counts = f.take(4 * nblk * E);
    bases = f.take(4 * nblk * E);
    offsets = f.take(4 * (E + 1));
    xq = f.take(Rc * H);
    wgu = f.take(E * 2 * I * H);
    wd = f.take(E * H * I);
    h = f.take(2 * Rc * I);
    hq = f.take(Rc * I);
    yperm = f.take(2 * Rc * H);
    fwd_bytes = f.off;

    Carver b;
    dp_ld = dswiglu_partials(static_cast<int>(I));
    dyq = b.take(Rc * H);
    dyqT = b.take(H * Rc);
    dgu = b.take(2 * Rc * 2 * I);
    dguq = b.take(Rc * 2 * I);
    dguqT = b.take(2 * I * Rc);
    dxperm = b.take(2 * Rc * H);
    dp = b.take(4 * Rc * dp_ld);
    amax_dy = b.take(4 * E);
    amax_dgu = b.take(4 * E);
    bwd_bytes = b.off;
  }
  int64_t ws_bytes() const { return fwd_bytes > bwd_bytes ? fwd_bytes : bwd_bytes; }
};

GemmArgs f8_gemm(int epi, bool kgroup, const uint8_t* a, int64_t a_rows, int64_t a_cols, const float* amax_a,
                 const uint8_t* b, int64_t b_rows, int64_t b_cols, const float* amax_b, const int32_t* poff, int E,
                 int32_t* st) {
  GemmArgs g{};
  g.epi = epi;
  g.kgroup = kgroup;
  g.pair = true;
  g.fp8 = true;
  g.a = a;
  g.a_rows = a_rows;
  g.a_cols = a_cols;
  g.amax_a = amax_a;
  g.b = b;
  g.b_rows = b_rows;
  g.b_cols = b_cols;
  g.amax_b = amax_b;
  g.poff = poff;
  g.E = E;
  g.status = st;
  return g;
}

// amax then per-tensor quantisation of a bf16 matrix batch, both orientations
// (either may be null).  Rows are gathered through src_rows when given; the
// tensors are the row groups of group_off (or the batches).
cudaError_t amax_quant(const uint16_t* x, int64_t ld_x, int64_t batch_stride, const int32_t* src_rows, int src_div,
                       int rows, int cols, int batch, const int32_t* rows_valid, const int32_t* group_off, int groups,
                       float* amax, int n_amax, uint8_t* q_row, uint8_t* q_col, int64_t ld_col, const float* probs,
                       float* probs_perm, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(amax, 0, 4 * static_cast<size_t>(n_amax), s);
  if (err != cudaSuccess) return err;
  AmaxParams ap{};
  ap.x = x;
  ap.ld_x = ld_x;
  ap.x_batch_stride = batch_stride;
  ap.src_rows = src_rows;
  ap.src_div = src_div;
  ap.rows = rows;
  ap.cols = cols;
  ap.batch = batch;
  ap.rows_valid = rows_valid;
  ap.group_off = group_off;
  ap.groups = groups;
  ap.amax = amax;
  err = launch_amax(ap, s);
  if (err != cudaSuccess) return err;
  QuantParams q{};
  q.x = x;
  q.ld_x = ld_x;
  q.x_batch_stride = batch_stride;
  q.src_rows = src_rows;
  q.src_div = src_div;
  q.probs = probs;
  q.probs_perm = probs_perm;
  q.rows = rows;
  q.cols = cols;
  q.batch = batch;
  q.rows_valid = rows_valid;
  q.q_row = q_row;
  q.q_col = q_col;
  q.ld_col = ld_col;
  q.pt_amax = amax;
  q.pt_group_off = group_off;
  q.pt_groups = groups;
  return launch_quant(q, s);
}

int fwd_impl(const mxg_mlp_fwd_args* A, int stage, void* stream) {
  if (!A) return MXG_ERR_ARG;
  const int T = A->T, H = A->H, I = A->I, E = A->E, k = A->k;
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!shape_ok(T, H, I, E, k)) return MXG_ERR_SHAPE;
  if (A->weight_cache) return MXG_ERR_ARG;   // the weight cache holds MXFP8 weights
  if (!A->x || !A->ids || !A->probs || !A->w_gate_up || !A->w_down || !A->y || !A->split_sizes || !A->saved ||
      !A->workspace || !A->dev_status)
    return MXG_ERR_ARG;
  if (!aligned32(A->x) || !aligned32(A->ids) || !aligned32(A->probs) || !aligned32(A->w_gate_up) ||
      !aligned32(A->w_down) || !aligned32(A->y) || !aligned32(A->split_sizes) || !aligned32(A->saved) ||
      !aligned32(A->workspace))
    return MXG_ERR_ALIGN;
  const PlanF8 pl(T, H, I, E, k);
  if (A->saved_bytes < static_cast<uint64_t>(pl.saved_bytes) ||
      A->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes()))
    return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* sv = A->saved;
  void* ws = A->workspace;
  const bool save = A->save_for_backward != 0;
  int32_t* st = A->dev_status;
  const int32_t* poff = at<int32_t>(sv, pl.poff);
  auto run = [stage](int id) { return stage < 0 || stage == id; };

  // permute into the 256-aligned padded layout
  if (run(MXG_FWD_PERMUTE)) {
    MXG_TRY(cudaMemsetAsync(at<int32_t>(sv, pl.prow_src), 0xFF, 4 * pl.Rc, s));
    PermuteParams pp{};
    pp.ids = A->ids;
    pp.R = static_cast<int32_t>(pl.R);
    pp.E = E;
    pp.counts = at<int32_t>(ws, pl.counts);
    pp.bases = at<int32_t>(ws, pl.bases);
    pp.offsets = at<int32_t>(ws, pl.offsets);
    pp.padded_offsets = at<int32_t>(sv, pl.poff);
    pp.pad = kGroupAlign;
    pp.split_sizes = A->split_sizes;
    pp.prow_src = at<int32_t>(sv, pl.prow_src);
    pp.prow_of_src = at<int32_t>(sv, pl.prow_of_src);
    pp.status = st;
    MXG_TRY(launch_permute(pp, s));
  }

  // weights: one tensor per expert; row-major codes for the forward GEMMs and
  // the transposed codes (same scale) for the backward's data-gradient GEMMs
  if (run(MXG_FWD_QUANT_WEIGHTS)) {
    MXG_TRY(amax_quant(A->w_gate_up, H, 2 * pl.I * H, nullptr, 1, 2 * I, H, E, nullptr, nullptr, 0,
                       at<float>(sv, pl.amax_wgu), E, at<uint8_t>(ws, pl.wgu), save ? at<uint8_t>(sv, pl.wguT) : nullptr,
                       2 * I, nullptr, nullptr, s));
    MXG_TRY(amax_quant(A->w_down, I, pl.H * I, nullptr, 1, H, I, E, nullptr, nullptr, 0, at<float>(sv, pl.amax_wd), E,
                       at<uint8_t>(ws, pl.wd), save ? at<uint8_t>(sv, pl.wdT) : nullptr, H, nullptr, nullptr, s));
  }

  // x gathered into the padded layout, one tensor per expert group (and its
  // transposed codes for the gate-up weight gradient); probabilities follow
  if (run(MXG_FWD_QUANT_X))
    MXG_TRY(amax_quant(A->x, H, 0, at<int32_t>(sv, pl.prow_src), k, static_cast<int>(pl.Rc), H, 1, poff + E, poff, E,
                       at<float>(sv, pl.amax_x), E, at<uint8_t>(ws, pl.xq), save ? at<uint8_t>(sv, pl.xqT) : nullptr,
                       pl.Rc, A->probs, at<float>(sv, pl.probs_perm), s));

  // gate-up GEMM + ScaledSwiGLU -> h (bf16) and amax(h) per expert, then h's codes
  if (run(MXG_FWD_GATE_UP)) {
    MXG_TRY(cudaMemsetAsync(at<float>(sv, pl.amax_h), 0, 4 * E, s));
    GemmArgs g = f8_gemm(EPI_SWIGLU, false, at<uint8_t>(ws, pl.xq), pl.Rc, H, at<float>(sv, pl.amax_x),
                         at<uint8_t>(ws, pl.wgu), pl.E * 2 * I, H, at<float>(sv, pl.amax_wgu), poff, E, st);
    g.M = static_cast<int32_t>(pl.Rc);
    g.N = 2 * I;
    g.K = H;
    g.b_rows_per_expert = 2 * I;
    g.I = I;
    g.probs_perm = at<float>(sv, pl.probs_perm);
    g.gu_save = save ? at<uint16_t>(sv, pl.gu) : nullptr;
    g.y_row = at<uint16_t>(ws, pl.h);
    g.y_row_ld = I;
    g.amax_out = at<float>(sv, pl.amax_h);
    g.tiles_upper = (pl.Rc / 256) * (I / 128);
    MXG_TRY(launch_gemm(g, s));
    QuantParams q{};
    q.x = at<uint16_t>(ws, pl.h);
    q.ld_x = I;
    q.rows = static_cast<int32_t>(pl.Rc);
    q.cols = I;
    q.batch = 1;
    q.rows_valid = poff + E;
    q.q_row = at<uint8_t>(ws, pl.hq);
    q.q_col = save ? at<uint8_t>(sv, pl.hqT) : nullptr;
    q.ld_col = pl.Rc;
    q.pt_amax = at<float>(sv, pl.amax_h);
    q.pt_group_off = poff;
    q.pt_groups = E;
    MXG_TRY(launch_quant(q, s));
  }

  // down GEMM
  if (run(MXG_FWD_DOWN)) {
    GemmArgs d = f8_gemm(EPI_BF16, false, at<uint8_t>(ws, pl.hq), pl.Rc, I, at<float>(sv, pl.amax_h),
                         at<uint8_t>(ws, pl.wd), pl.E * H, I, at<float>(sv, pl.amax_wd), poff, E, st);
    d.M = static_cast<int32_t>(pl.Rc);
    d.N = H;
    d.K = I;
    d.b_rows_per_expert = H;
    d.d = at<uint16_t>(ws, pl.yperm);
    d.ldd = H;
    d.tiles_upper = (pl.Rc / 256) * (H / 256);
    MXG_TRY(launch_gemm(d, s));
  }

  if (run(MXG_FWD_COMBINE))
    MXG_TRY(launch_combine(at<uint16_t>(ws, pl.yperm), at<int32_t>(sv, pl.prow_of_src), T, k, H, A->y, s));
  return MXG_OK;
}

int bwd_impl(const mxg_mlp_bwd_args* A, int stage, void* stream) {
  if (!A) return MXG_ERR_ARG;
  const int T = A->T, H = A->H, I = A->I, E = A->E, k = A->k;
  if (T <= 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!shape_ok(T, H, I, E, k)) return MXG_ERR_SHAPE;
  if (A->weight_cache || A->main_grad_gate_up || A->main_grad_down) return MXG_ERR_ARG;
  if (!A->dy || !A->saved || !A->dx || !A->dw_gate_up || !A->dw_down || !A->dprobs || !A->workspace ||
      !A->dev_status)
    return MXG_ERR_ARG;
  if (!aligned32(A->dy) || !aligned32(A->saved) || !aligned32(A->dx) || !aligned32(A->dw_gate_up) ||
      !aligned32(A->dw_down) || !aligned32(A->dprobs) || !aligned32(A->workspace))
    return MXG_ERR_ALIGN;
  const PlanF8 pl(T, H, I, E, k);
  if (A->saved_bytes < static_cast<uint64_t>(pl.saved_bytes) ||
      A->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes()))
    return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* sv = A->saved;
  void* ws = A->workspace;
  int32_t* st = A->dev_status;
  const int32_t* poff = at<int32_t>(sv, pl.poff);
  auto run = [stage](int id) { return stage < 0 || stage == id; };
  const float* amax_x = at<float>(sv, pl.amax_x);
  const float* amax_wgu = at<float>(sv, pl.amax_wgu);
  const float* amax_wd = at<float>(sv, pl.amax_wd);
  const float* amax_h = at<float>(sv, pl.amax_h);

  // dy gathered, one tensor per expert group: row codes for the data gradient,
  // transposed codes for the down weight gradient
  if (run(MXG_BWD_QUANT_DY))
    MXG_TRY(amax_quant(A->dy, H, 0, at<int32_t>(sv, pl.prow_src), k, static_cast<int>(pl.Rc), H, 1, poff + E, poff, E,
                       at<float>(ws, pl.amax_dy), E, at<uint8_t>(ws, pl.dyq), at<uint8_t>(ws, pl.dyqT), pl.Rc, nullptr,
                       nullptr, s));

  // dH = dY W_down with fused dSwiGLU -> dGU (bf16) and amax(dGU) per expert,
  // d(prob) partials; then dGU's codes in both orientations
  if (run(MXG_BWD_DGRAD_DOWN)) {
    MXG_TRY(cudaMemsetAsync(at<float>(ws, pl.amax_dgu), 0, 4 * E, s));
    GemmArgs g = f8_gemm(EPI_DSWIGLU, false, at<uint8_t>(ws, pl.dyq), pl.Rc, H, at<float>(ws, pl.amax_dy),
                         at<uint8_t>(sv, pl.wdT), pl.E * I, H, amax_wd, poff, E, st);
    g.M = static_cast<int32_t>(pl.Rc);
    g.N = I;
    g.K = H;
    g.b_rows_per_expert = I;
    g.I = I;
    g.probs_perm = at<float>(sv, pl.probs_perm);
    g.gu_save = const_cast<uint16_t*>(at<uint16_t>(sv, pl.gu));
    g.y_row = at<uint16_t>(ws, pl.dgu);
    g.y_row_ld = 2 * I;
    g.amax_out = at<float>(ws, pl.amax_dgu);
    g.dp_part = at<float>(ws, pl.dp);
    g.dp_ld = static_cast<int32_t>(pl.dp_ld);
    g.tiles_upper = (pl.Rc / 256) * (I / 128);
    MXG_TRY(launch_gemm(g, s));
    QuantParams q{};
    q.x = at<uint16_t>(ws, pl.dgu);
    q.ld_x = 2 * I;
    q.rows = static_cast<int32_t>(pl.Rc);
    q.cols = 2 * I;
    q.batch = 1;
    q.rows_valid = poff + E;
    q.q_row = at<uint8_t>(ws, pl.dguq);
    q.q_col = at<uint8_t>(ws, pl.dguqT);
    q.ld_col = pl.Rc;
    q.pt_amax = at<float>(ws, pl.amax_dgu);
    q.pt_group_off = poff;
    q.pt_groups = E;
    MXG_TRY(launch_quant(q, s));
  }

  // dW_down[e] = dY^T H over the tokens of e
  if (run(MXG_BWD_WGRAD_DOWN)) {
    GemmArgs w = f8_gemm(EPI_BF16, true, at<uint8_t>(ws, pl.dyqT), H, pl.Rc, at<float>(ws, pl.amax_dy),
                         at<uint8_t>(sv, pl.hqT), I, pl.Rc, amax_h, poff, E, st);
    w.M = H;
    w.N = I;
    w.d = A->dw_down;
    w.ldd = I;
    w.tiles_upper = pl.E * (H / 256) * (I / 256);
    MXG_TRY(launch_gemm(w, s));
  }

  // dX_perm = dGU W_gate_up
  if (run(MXG_BWD_DGRAD_GATE_UP)) {
    GemmArgs x = f8_gemm(EPI_BF16, false, at<uint8_t>(ws, pl.dguq), pl.Rc, 2 * I, at<float>(ws, pl.amax_dgu),
                         at<uint8_t>(sv, pl.wguT), pl.E * H, 2 * I, amax_wgu, poff, E, st);
    x.M = static_cast<int32_t>(pl.Rc);
    x.N = H;
    x.K = 2 * I;
    x.b_rows_per_expert = H;
    x.d = at<uint16_t>(ws, pl.dxperm);
    x.ldd = H;
    x.tiles_upper = (pl.Rc / 256) * (H / 256);
    MXG_TRY(launch_gemm(x, s));
  }

  // dW_gate_up[e] = dGU^T X over the tokens of e
  if (run(MXG_BWD_WGRAD_GATE_UP)) {
    GemmArgs v = f8_gemm(EPI_BF16, true, at<uint8_t>(ws, pl.dguqT), 2 * I, pl.Rc, at<float>(ws, pl.amax_dgu),
                         at<uint8_t>(sv, pl.xqT), H, pl.Rc, amax_x, poff, E, st);
    v.M = 2 * I;
    v.N = H;
    v.d = A->dw_gate_up;
    v.ldd = H;
    v.tiles_upper = pl.E * (2 * I / 256) * (H / 256);
    MXG_TRY(launch_gemm(v, s));
  }

  const int32_t* prow_of_src = at<int32_t>(sv, pl.prow_of_src);
  if (run(MXG_BWD_COMBINE_DX))
    MXG_TRY(launch_combine(at<uint16_t>(ws, pl.dxperm), prow_of_src, T, k, H, A->dx, s));
  if (run(MXG_BWD_DPROBS))
    MXG_TRY(launch_dprob(at<float>(ws, pl.dp), static_cast<int>(pl.dp_ld), prow_of_src, static_cast<int>(pl.R),
                         A->dprobs, s));
  return MXG_OK;
}

}  // namespace
}  // namespace mxg

using namespace mxg;

extern "C" {

size_t mxg_mlp_fp8_saved_bytes(int T, int H, int I, int E, int k) {
  if (!shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(PlanF8(T, H, I, E, k).saved_bytes);
}

size_t mxg_mlp_fp8_workspace_bytes(int T, int H, int I, int E, int k) {
  if (!shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(PlanF8(T, H, I, E, k).ws_bytes());
}

const void* mxg_mlp_fp8_saved_view(const void* saved, int T, int H, int I, int E, int k, int which) {
  if (!saved || !shape_ok(T, H, I, E, k)) return nullptr;
  const PlanF8 pl(T, H, I, E, k);
  switch (which) {
    case 0: return at<uint8_t>(saved, pl.xqT);
    case 1: return at<uint8_t>(saved, pl.amax_x);
    case 2: return at<uint8_t>(saved, pl.amax_wgu);
    case 3: return at<uint8_t>(saved, pl.amax_wd);
    case 4: return at<uint8_t>(saved, pl.amax_h);
    case 5: return at<uint8_t>(saved, pl.poff);
    default: return nullptr;
  }
}

int mxg_grouped_mlp_fp8_fwd(const mxg_mlp_fwd_args* A, void* stream) { return fwd_impl(A, -1, stream); }

int mxg_grouped_mlp_fp8_fwd_stage(const mxg_mlp_fwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_FWD_NUM_STAGES) return MXG_ERR_ARG;
  return fwd_impl(A, stage, stream);
}

int mxg_grouped_mlp_fp8_bwd(const mxg_mlp_bwd_args* A, void* stream) { return bwd_impl(A, -1, stream); }

int mxg_grouped_mlp_fp8_bwd_stage(const mxg_mlp_bwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_BWD_NUM_STAGES) return MXG_ERR_ARG;
  return bwd_impl(A, stage, stream);
}

}  // extern "C"
