// C-ABI entry points of the BF16 grouped expert MLP: the same route ->
// permute -> gate-up + ScaledSwiGLU -> down -> combine path and its backward,
// with bf16 operands on the tensor cores (tcgen05 kind::f16, fp32
// accumulators) and no quantisation.  It is the like-for-like reference the
// MXFP8 path is measured against ("BioNeMo Uses Grouped Kernels and MXFP8",
// "Training benchmark", Fig. 5: the recipe's BF16 and MXFP8 runs).
//
// Data flow differences from the MXFP8 path: the activations are gathered into
// the padded per-expert layout as bf16 (plus a transposed copy for the weight
// gradients), the weights are used as given for the forward GEMMs and
// transposed once for the data-gradient GEMMs, and the fused epilogues write
// h and dGU in bf16 (row-major and transposed) instead of MXFP8.  All GEMMs run
// as 256 x 256 CTA-pair tiles, so H and I must be multiples of 256 and expert
// groups start on multiples of 256 rows.
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

// Byte offsets of every buffer inside `saved` and `workspace`.
struct PlanBf {
  int64_t T, H, I, E, k, R, Rc;
  int64_t poff, prow_src, prow_of_src, probs_perm, gu, xT, hT, wguT, wdT, saved_bytes;
  int64_t counts, bases, offsets, xp, h, yperm, fwd_bytes;
  int64_t dyp, dyT, dgu, dguT, dxperm, dp, bwd_bytes;
  int64_t dp_ld;

  PlanBf(int64_t T_, int64_t H_, int64_t I_, int64_t E_, int64_t k_) : T(T_), H(H_), I(I_), E(E_), k(k_) {
    R = T * k;
    Rc = align_up(R, kGroupAlign) + kGroupAlign * E;
    Carver s;
    poff = s.take(4 * (E + 1));
    prow_src = s.take(4 * Rc);
    prow_of_src = s.take(4 * R);
    probs_perm = s.take(4 * Rc);
    gu = s.take(2 * Rc * 2 * I);
    xT = s.take(2 * H * Rc);
    hT = s.take(2 * I * Rc);
    wguT = s.take(2 * E * H * 2 * I);
    wdT = s.take(2 * E * I * H);
    saved_bytes = s.off;

    Carver f;
    const int64_t nblk = permute_num_blocks(static_cast<int>(R));
    counts = f.take(4 * nblk * E);
    bases = f.take(4 * nblk * E);
    offsets = f.take(4 * (E + 1));
    xp = f.take(2 * Rc * H);
    h = f.take(2 * Rc * I);
    yperm = f.take(2 * Rc * H);
    fwd_bytes = f.off;

    Carver b;
    dp_ld = dswiglu_partials(static_cast<int>(I));
    dyp = b.take(2 * Rc * H);
    dyT = b.take(2 * H * Rc);
    dgu = b.take(2 * Rc * 2 * I);
    dguT = b.take(2 * 2 * I * Rc);
    dxperm = b.take(2 * Rc * H);
    dp = b.take(4 * Rc * dp_ld);
    bwd_bytes = b.off;
  }
  int64_t ws_bytes() const { return fwd_bytes > bwd_bytes ? fwd_bytes : bwd_bytes; }
};

GemmArgs bf16_gemm(int epi, bool kgroup, const void* a, int64_t a_rows, int64_t a_cols, const void* b,
                   int64_t b_rows, int64_t b_cols, const int32_t* poff, int E, int32_t* st) {
  GemmArgs g{};
  g.epi = epi;
  g.kgroup = kgroup;
  g.pair = true;
  g.bf16 = true;
  g.a = static_cast<const uint8_t*>(a);
  g.a_rows = a_rows;
  g.a_cols = a_cols;
  g.b = static_cast<const uint8_t*>(b);
  g.b_rows = b_rows;
  g.b_cols = b_cols;
  g.poff = poff;
  g.E = E;
  g.status = st;
  return g;
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
  const PlanBf pl(T, H, I, E, k);
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

  // weights: transposed copies for the backward's data-gradient GEMMs
  if (run(MXG_FWD_QUANT_WEIGHTS) && save) {
    QuantParams wq{};
    wq.x = A->w_gate_up;
    wq.ld_x = H;
    wq.x_batch_stride = 2 * pl.I * H;
    wq.src_div = 1;
    wq.rows = 2 * I;
    wq.cols = H;
    wq.batch = E;
    wq.b_col = at<uint16_t>(sv, pl.wguT);
    wq.ld_col = 2 * I;
    MXG_TRY(launch_quant(wq, s));
    QuantParams dq = wq;
    dq.x = A->w_down;
    dq.ld_x = I;
    dq.x_batch_stride = pl.H * I;
    dq.rows = H;
    dq.cols = I;
    dq.b_col = at<uint16_t>(sv, pl.wdT);
    dq.ld_col = H;
    MXG_TRY(launch_quant(dq, s));
  }

  // gather x into the padded layout (and its transposed copy for the gate-up
  // weight gradient); probabilities follow the rows
  if (run(MXG_FWD_QUANT_X)) {
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
    xq.b_row = at<uint16_t>(ws, pl.xp);
    if (save) {
      xq.b_col = at<uint16_t>(sv, pl.xT);
      xq.ld_col = pl.Rc;
    }
    MXG_TRY(launch_quant(xq, s));
  }

  // gate-up GEMM + ScaledSwiGLU: h (bf16) and its transposed copy
  if (run(MXG_FWD_GATE_UP)) {
    GemmArgs g = bf16_gemm(EPI_SWIGLU, false, at<uint16_t>(ws, pl.xp), pl.Rc, H, A->w_gate_up, pl.E * 2 * I, H,
                           poff, E, st);
    g.M = static_cast<int32_t>(pl.Rc);
    g.N = 2 * I;
    g.K = H;
    g.b_rows_per_expert = 2 * I;
    g.I = I;
    g.probs_perm = at<float>(sv, pl.probs_perm);
    g.gu_save = save ? at<uint16_t>(sv, pl.gu) : nullptr;
    g.y_row = at<uint16_t>(ws, pl.h);
    g.y_row_ld = I;
    if (save) {
      g.y_col = at<uint16_t>(sv, pl.hT);
      g.y_col_ld = pl.Rc;
    }
    g.tiles_upper = (pl.Rc / 256) * (I / 128);
    MXG_TRY(launch_gemm(g, s));
  }

  // down GEMM
  if (run(MXG_FWD_DOWN)) {
    GemmArgs d = bf16_gemm(EPI_BF16, false, at<uint16_t>(ws, pl.h), pl.Rc, I, A->w_down, pl.E * H, I, poff, E, st);
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
  const PlanBf pl(T, H, I, E, k);
  if (A->saved_bytes < static_cast<uint64_t>(pl.saved_bytes) ||
      A->workspace_bytes < static_cast<uint64_t>(pl.ws_bytes()))
    return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void* sv = A->saved;
  void* ws = A->workspace;
  int32_t* st = A->dev_status;
  const int32_t* poff = at<int32_t>(sv, pl.poff);
  auto run = [stage](int id) { return stage < 0 || stage == id; };

  // gather dy (row copy for the data gradient, transposed copy for the weight gradient)
  if (run(MXG_BWD_QUANT_DY)) {
    QuantParams yq{};
    yq.x = A->dy;
    yq.ld_x = H;
    yq.src_rows = at<int32_t>(sv, pl.prow_src);
    yq.src_div = k;
    yq.rows = static_cast<int32_t>(pl.Rc);
    yq.cols = H;
    yq.batch = 1;
    yq.rows_valid = poff + E;
    yq.b_row = at<uint16_t>(ws, pl.dyp);
    yq.b_col = at<uint16_t>(ws, pl.dyT);
    yq.ld_col = pl.Rc;
    MXG_TRY(launch_quant(yq, s));
  }

  // dH = dY W_down with fused dSwiGLU: dGU (bf16, both layouts), d(prob) partials
  if (run(MXG_BWD_DGRAD_DOWN)) {
    GemmArgs g = bf16_gemm(EPI_DSWIGLU, false, at<uint16_t>(ws, pl.dyp), pl.Rc, H, at<uint16_t>(sv, pl.wdT),
                           pl.E * I, H, poff, E, st);
    g.M = static_cast<int32_t>(pl.Rc);
    g.N = I;
    g.K = H;
    g.b_rows_per_expert = I;
    g.I = I;
    g.probs_perm = at<float>(sv, pl.probs_perm);
    g.gu_save = const_cast<uint16_t*>(at<uint16_t>(sv, pl.gu));
    g.y_row = at<uint16_t>(ws, pl.dgu);
    g.y_row_ld = 2 * I;
    g.y_col = at<uint16_t>(ws, pl.dguT);
    g.y_col_ld = pl.Rc;
    g.dp_part = at<float>(ws, pl.dp);
    g.dp_ld = static_cast<int32_t>(pl.dp_ld);
    g.tiles_upper = (pl.Rc / 256) * (I / 128);
    MXG_TRY(launch_gemm(g, s));
  }

  // dW_down[e] = dY^T H over the tokens of e
  if (run(MXG_BWD_WGRAD_DOWN)) {
    GemmArgs w = bf16_gemm(EPI_BF16, true, at<uint16_t>(ws, pl.dyT), H, pl.Rc, at<uint16_t>(sv, pl.hT), I, pl.Rc,
                           poff, E, st);
    w.M = H;
    w.N = I;
    w.d = A->dw_down;
    w.ldd = I;
    w.tiles_upper = pl.E * (H / 256) * (I / 256);
    MXG_TRY(launch_gemm(w, s));
  }

  // dX_perm = dGU W_gate_up
  if (run(MXG_BWD_DGRAD_GATE_UP)) {
    GemmArgs x = bf16_gemm(EPI_BF16, false, at<uint16_t>(ws, pl.dgu), pl.Rc, 2 * I, at<uint16_t>(sv, pl.wguT),
                           pl.E * H, 2 * I, poff, E, st);
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
    GemmArgs v = bf16_gemm(EPI_BF16, true, at<uint16_t>(ws, pl.dguT), 2 * I, pl.Rc, at<uint16_t>(sv, pl.xT), H,
                           pl.Rc, poff, E, st);
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

size_t mxg_mlp_bf16_saved_bytes(int T, int H, int I, int E, int k) {
  if (!shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(PlanBf(T, H, I, E, k).saved_bytes);
}

size_t mxg_mlp_bf16_workspace_bytes(int T, int H, int I, int E, int k) {
  if (!shape_ok(T, H, I, E, k)) return 0;
  return static_cast<size_t>(PlanBf(T, H, I, E, k).ws_bytes());
}

int mxg_grouped_mlp_bf16_fwd(const mxg_mlp_fwd_args* A, void* stream) { return fwd_impl(A, -1, stream); }

int mxg_grouped_mlp_bf16_fwd_stage(const mxg_mlp_fwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_FWD_NUM_STAGES) return MXG_ERR_ARG;
  return fwd_impl(A, stage, stream);
}

int mxg_grouped_mlp_bf16_bwd(const mxg_mlp_bwd_args* A, void* stream) { return bwd_impl(A, -1, stream); }

int mxg_grouped_mlp_bf16_bwd_stage(const mxg_mlp_bwd_args* A, int stage, void* stream) {
  if (stage < 0 || stage >= MXG_BWD_NUM_STAGES) return MXG_ERR_ARG;
  return bwd_impl(A, stage, stream);
}

}  // extern "C"
