"""Pins for the oracle's routing, permute, forward and backward against facts
fixed outside it: brute-force sorting, numpy's stable argsort, exact rational
GEMMs, the per-expert loop (the equivalence grouping rests on), the dense
SwiGLU MLP special case, empty experts, and finite differences of the
unquantised forward."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synthetic
from conftest import read_golden
from oracle import moe, mx


def _case(T, H, I, E, k, seed, **kw):
    d = synthetic.make_case(T, H, I, E, k, seed, **kw)
    return {n: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for n, v in d.items()}


def test_golden_structure():
    g = read_golden("moe_structure.txt")
    c = _case(64, 32, 32, g["router_experts"], g["router_top_k"], 1)
    ids, probs = moe.route_topk(c["logits"], g["router_top_k"])
    assert ids.shape == (64, 2) and np.allclose(probs.sum(1), 1.0)
    out = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    assert out["gu"].shape[1] == g["gate_up_out_over_hidden_in"] * 32


def test_route_topk_brute_force():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((300, 8)).astype(np.float32)
    logits[:40, 3] = logits[:40, 5]                 # exact ties -> lower id first
    logits[40:60] = 0.0                             # all tied
    for k in (1, 2, 3, 8):
        ids, probs = moe.route_topk(logits, k)
        for t in range(logits.shape[0]):
            order = sorted(range(8), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert list(ids[t]) == order
        # renormalised over the chosen = full softmax restricted and renormalised
        full = np.exp(logits.astype(np.float64) - logits.max(1, keepdims=True))
        full /= full.sum(1, keepdims=True)
        sel = np.take_along_axis(full, ids.astype(np.int64), 1)
        np.testing.assert_allclose(probs, sel / sel.sum(1, keepdims=True), rtol=1e-13)


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (64, 8), (5, 1)])
def test_permute_matches_stable_argsort(E, k):
    rng = np.random.default_rng(E * 10 + k)
    T = 333
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = moe.permute(ids, E)
    flat = ids.reshape(-1)
    np.testing.assert_array_equal(p["src_of_row"], np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(p["split_sizes"], np.bincount(flat, minlength=E))
    assert p["split_sizes"].sum() == T * k
    np.testing.assert_array_equal(p["row_of_src"][p["src_of_row"]], np.arange(T * k))
    assert np.all(p["padded_offsets"] % 128 == 0)
    pads = np.diff(p["padded_offsets"])
    assert np.all((pads >= p["split_sizes"]) & (pads < p["split_sizes"] + 128))
    p256 = moe.permute(ids, E, pad=256)
    pads = np.diff(p256["padded_offsets"])
    assert np.all(p256["padded_offsets"] % 256 == 0)
    assert np.all((pads >= p["split_sizes"]) & (pads < p["split_sizes"] + 256))
    np.testing.assert_array_equal(p256["src_of_row"], p["src_of_row"])


def _exact_dot(qa, sa, qb, sb):
    """Exact rational A_deq @ B_deq^T from codes and scale bytes."""
    def deq(q, s):
        out = []
        for r in range(q.shape[0]):
            row = []
            for c in range(q.shape[1]):
                code = int(q[r, c])
                sign = -1 if code & 0x80 else 1
                ef, mf = (code >> 3) & 0xF, code & 7
                v = Fraction(mf, 8) / 64 if ef == 0 else (1 + Fraction(mf, 8)) * Fraction(2) ** (ef - 7)
                row.append(sign * v * Fraction(2) ** (int(s[r, c // 32]) - 127))
            out.append(row)
        return out
    A, B = deq(qa, sa), deq(qb, sb)
    return [[sum(a * b for a, b in zip(A[i], B[j])) for j in range(len(B))] for i in range(len(A))]


def test_gemm_exact_rational():
    """GU = deq(Xq) deq(Wq)^T in fp64 equals the exact rational product up to the
    fp64 summation error bound."""
    c = _case(8, 64, 32, 1, 1, 21)
    x, w = c["x"], c["w_gate_up"][0]
    qa, sa = mx.quantize_blocks(x)
    qb, sb = mx.quantize_blocks(w)
    exact = _exact_dot(qa, sa, qb, sb)
    ids = np.zeros((8, 1), dtype=np.int32)
    out = moe.mlp_fwd(x, ids, np.ones((8, 1)), c["w_gate_up"], c["w_down"])
    gu = out["gu"]
    absdot = np.abs(mx.dequantize_blocks(qa, sa)) @ np.abs(mx.dequantize_blocks(qb, sb)).T
    for i in range(8):
        for j in range(64):
            err = abs(Fraction(float(gu[i, j])) - exact[i][j])
            assert err <= Fraction(64 * 2.0 ** -53 * absdot[i, j])


@pytest.mark.parametrize("quant", [True, False])
def test_grouped_equals_per_expert_loop(quant):
    """The grouped result equals a per-token, per-expert loop (the Python-loop
    baseline's structure): grouping changes how work reaches the device, not
    what each expert computes."""
    T, H, I, E, k = 50, 64, 64, 5, 2
    c = _case(T, H, I, E, k, 31)
    ids, probs = moe.route_topk(c["logits"], k)
    out = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"], quant=quant)
    fq = mx.fake_quant if quant else (lambda a: a)
    y = np.zeros((T, H))
    for e in range(E):                       # loop over experts, select their tokens
        wg = fq(c["w_gate_up"][e])
        wd = fq(c["w_down"][e])
        for t in range(T):
            for j in range(k):
                if ids[t, j] != e:
                    continue
                gu = fq(c["x"][t:t + 1]) @ wg.T
                g, u = gu[:, :I], gu[:, I:]
                h = probs[t, j] * (g / (1 + np.exp(-g))) * u
                y[t] += (fq(h) @ wd.T)[0]
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu_mlp():
    """k=1, every token to expert 0, p=1: the dense SwiGLU MLP (torch fp64
    silu/matmul on the same dequantised operands)."""
    T, H, I = 40, 64, 96
    c = _case(T, H, I, 1, 1, 41)
    ids = np.zeros((T, 1), dtype=np.int32)
    for quant in (False, True):
        out = moe.mlp_fwd(c["x"], ids, np.ones((T, 1)), c["w_gate_up"], c["w_down"], quant=quant)
        fq = mx.fake_quant if quant else (lambda a: a)
        xt = torch.from_numpy(fq(c["x"]))
        wg = torch.from_numpy(fq(c["w_gate_up"][0]))
        wd = torch.from_numpy(fq(c["w_down"][0]))
        gu = xt @ wg.T
        h = torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]
        y = torch.from_numpy(fq(h.numpy())) @ wd.T
        np.testing.assert_allclose(out["y"], y.numpy(), rtol=1e-12, atol=1e-13)


def test_empty_experts_contribute_nothing():
    T, H, I, E, k = 64, 64, 32, 6, 2
    c = _case(T, H, I, E, k, 51, empty_experts=(1, 4))
    ids, probs = moe.route_topk(c["logits"], k)
    assert not np.isin(ids, [1, 4]).any()
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    g = moe.mlp_bwd(ctx, c["dy"])
    for e in (1, 4):
        assert not g["dw_gate_up"][e].any() and not g["dw_down"][e].any()
    # scrambling an empty expert's weights changes nothing
    w2 = c["w_gate_up"].copy()
    w2[1] = 123.0
    ctx2 = moe.mlp_fwd(c["x"], ids, probs, w2, c["w_down"])
    np.testing.assert_array_equal(ctx2["y"], ctx["y"])


def test_k1_combine_is_inverse_permutation():
    T, H, I, E = 70, 32, 32, 3
    c = _case(T, H, I, E, 1, 61)
    ids, probs = moe.route_topk(c["logits"], 1)
    out = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    row = out["perm"]["row_of_src"]
    np.testing.assert_array_equal(out["y"], out["y_perm"][row])


def test_backward_finite_differences():
    """With quantisation as identity the backward is the exact gradient of
    L = sum(y * dy): compare with central differences in fp64."""
    T, H, I, E, k = 12, 32, 32, 3, 2
    c = _case(T, H, I, E, k, 71)
    ids, probs = moe.route_topk(c["logits"], k)
    x, wgu, wd, dy = c["x"], c["w_gate_up"], c["w_down"], c["dy"]
    ctx = moe.mlp_fwd(x, ids, probs, wgu, wd, quant=False)
    g = moe.mlp_bwd(ctx, dy)

    def loss(x_, p_, wgu_, wd_):
        return float(np.sum(moe.mlp_fwd(x_, ids, p_, wgu_, wd_, quant=False)["y"] * dy))

    rng = np.random.default_rng(0)
    eps = 1e-6

    def check(arr, grad, setter, n=12):
        for _ in range(n):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            fd = (setter(a1) - setter(a2)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (idx, fd, grad[idx])

    check(x, g["dx"], lambda a: loss(a, probs, wgu, wd))
    check(probs, g["dprobs"], lambda a: loss(x, a, wgu, wd))
    check(wgu, g["dw_gate_up"], lambda a: loss(x, probs, a, wd), n=20)
    check(wd, g["dw_down"], lambda a: loss(x, probs, wgu, a), n=20)
    # make sure both halves of W_gate_up (gate rows and up rows) were probed
    for half in (slice(0, I), slice(I, 2 * I)):
        for _ in range(6):
            e, n_, h_ = rng.integers(E), rng.integers(half.start, half.stop), rng.integers(H)
            a1, a2 = wgu.copy(), wgu.copy()
            a1[e, n_, h_] += eps
            a2[e, n_, h_] -= eps
            fd = (loss(x, probs, a1, wd) - loss(x, probs, a2, wd)) / (2 * eps)
            assert abs(fd - g["dw_gate_up"][e, n_, h_]) <= 1e-6 * max(1.0, abs(fd))


def test_backward_quantised_uses_mx_operands():
    """With quantisation on, each backward GEMM equals the fp64 product of the
    explicitly quantised operands (row-wise along the contraction axis for
    dgrad, token-column-wise from each group's first row for wgrad)."""
    T, H, I, E, k = 80, 64, 64, 3, 2
    c = _case(T, H, I, E, k, 81)
    ids, probs = moe.route_topk(c["logits"], k)
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    g = moe.mlp_bwd(ctx, c["dy"])
    perm = ctx["perm"]
    tok = perm["src_of_row"] // k
    for e in range(E):
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        dyp = c["dy"][tok[a:b]]
        dh = mx.fake_quant(dyp) @ mx.fake_quant(c["w_down"][e].T).T
        np.testing.assert_allclose(g["dh"][a:b], dh, rtol=1e-12, atol=1e-12)
        dwd = mx.fake_quant_group_columns(dyp).T @ mx.fake_quant_group_columns(ctx["h"][a:b])
        np.testing.assert_allclose(g["dw_down"][e], dwd, rtol=1e-12, atol=1e-14)


def test_sampled_evaluation_equals_full_oracle():
    """The sampled evaluation used at full sizes reproduces the full oracle on
    the sampled tokens and weight-gradient slices."""
    from oracle import sampled
    T, H, I, E, k = 96, 64, 96, 4, 2
    c = _case(T, H, I, E, k, 91, empty_experts=(2,))
    ids, probs = moe.route_topk(c["logits"], k)
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    g = moe.mlp_bwd(ctx, c["dy"])
    perm = ctx["perm"]
    expert_of_row = np.repeat(np.arange(E), perm["split_sizes"])
    W = {e: moe.expert_weights(c["w_gate_up"][e], c["w_down"][e]) for e in range(E)}
    tokens = [0, 5, 17, 95]
    s = sampled.rows_forward_backward(tokens, c["x"], c["dy"], probs, perm["row_of_src"], expert_of_row, k, W)
    np.testing.assert_allclose(s["y"], ctx["y"][tokens], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s["dx"], g["dx"][tokens], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s["dprobs"], g["dprobs"][tokens], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(s["gu"], ctx["gu"][s["rows"]], rtol=1e-11, atol=1e-13)
    # one expert at a time, summed: the same outputs (the full-size tests hold
    # one expert's weights in memory at a time)
    acc = {n: 0.0 for n in ("y", "dx", "dprobs")}
    done = np.zeros_like(s["done"])
    for e in W:
        part = sampled.rows_forward_backward(tokens, c["x"], c["dy"], probs, perm["row_of_src"], expert_of_row, k,
                                             {e: W[e]})
        for n in acc:
            acc[n] = acc[n] + part[n]
        assert not (done & part["done"]).any()
        done |= part["done"]
    assert done.all()
    for n in acc:
        np.testing.assert_allclose(acc[n], s[n], rtol=1e-12, atol=1e-14)
    tok = perm["src_of_row"] // k
    for e in (0, 3):
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        xe, dye, pe = c["x"][tok[a:b]], c["dy"][tok[a:b]], ctx["p_perm"][a:b]
        cols = np.array([0, 7, 50, 95])
        got = sampled.dw_down_columns(xe, dye, pe, c["w_gate_up"][e], cols)
        np.testing.assert_allclose(got, g["dw_down"][e][:, cols], rtol=1e-11, atol=1e-13)
        rows = np.array([1, 60, 96, 150, 191])
        got = sampled.dw_gate_up_rows(xe, dye, pe, c["w_gate_up"][e], c["w_down"][e], rows)
        np.testing.assert_allclose(got, g["dw_gate_up"][e][rows], rtol=1e-11, atol=1e-13)


def test_weight_quant_pool_equals_oracle():
    """The multi-process weight quantisation used by the full-size tests gives
    exactly oracle.moe.expert_weights."""
    from oracle_pool import WeightQuantPool
    wgu = synthetic.random_bf16((2 * 96, 128), 5, std=0.02)
    wd = synthetic.random_bf16((128, 96), 6, std=0.02)
    ref = moe.expert_weights(wgu.double().numpy(), wd.double().numpy())
    pool = WeightQuantPool(workers=3)
    try:
        got = pool.expert_weights(wgu, wd)
    finally:
        pool.close()
    for n in ("wg", "wd", "wdT", "wguT"):
        assert np.array_equal(got[n], ref[n]), n


def test_backward_quantised_dgrad_and_wgrad_gate_up_operands():
    """With quantisation on, dX of an expert's rows equals deq(MX(dGU) along 2I)
    times deq(MX(W_gate_up^T) along 2I), and dW_gate_up equals
    deq(colMX(dGU))^T deq(colMX(X)) with token blocks from the group's first
    row.  Every operand is built here from codes and scale bytes along the
    stated axis; the plausible mistakes (the weight quantised along H, dGU
    quantised over tokens for the dgrad, or row-wise for the wgrad) are shown
    to give different results, so the pin tells them apart."""
    T, H, I, E, k = 80, 64, 96, 3, 2                 # H != 2I: a transposed operand cannot go unnoticed
    c = _case(T, H, I, E, k, 83)
    ids, probs = moe.route_topk(c["logits"], k)
    ctx = moe.mlp_fwd(c["x"], ids, probs, c["w_gate_up"], c["w_down"])
    g = moe.mlp_bwd(ctx, c["dy"])
    perm = ctx["perm"]
    tok = perm["src_of_row"] // k
    for e in range(E):
        a, b = perm["offsets"][e], perm["offsets"][e + 1]
        m = b - a
        assert m > 32                                  # spans more than one token block
        dgu = g["dgu"][a:b]                            # [m, 2I]
        dgu_q = mx.dequantize_blocks(*mx.quantize_blocks(dgu))              # blocks along 2I
        wT = np.ascontiguousarray(c["w_gate_up"][e].T)                      # [H, 2I]
        wT_q = mx.dequantize_blocks(*mx.quantize_blocks(wT))                # blocks along 2I
        dx_rows = dgu_q @ wT_q.T
        np.testing.assert_allclose(g["dx_perm"][a:b], dx_rows, rtol=1e-12, atol=1e-13)
        w_along_h = mx.fake_quant(c["w_gate_up"][e])                       # [2I, H], blocks along H
        assert not np.allclose(g["dx_perm"][a:b], dgu_q @ w_along_h, rtol=1e-6, atol=0)
        dgu_tok = mx.fake_quant_group_columns(dgu)                          # blocks over tokens
        assert not np.allclose(g["dx_perm"][a:b], dgu_tok @ wT_q.T, rtol=1e-6, atol=0)

        x_perm = c["x"][tok[a:b]]                      # [m, H]
        cd, sd = mx.quantize_group_columns(dgu)        # [2I, mpad]: 32-token blocks from the group start
        cx, sx = mx.quantize_group_columns(x_perm)     # [H, mpad]
        mpad = cd.shape[1]
        assert mpad == -(-m // 32) * 32 and cx.shape == (H, mpad)
        dw = mx.dequantize_blocks(cd, sd) @ mx.dequantize_blocks(cx, sx).T  # padding tokens are zero codes
        np.testing.assert_allclose(g["dw_gate_up"][e], dw, rtol=1e-12, atol=1e-13)
        row_wise = dgu_q.T @ mx.fake_quant_group_columns(x_perm)
        assert not np.allclose(g["dw_gate_up"][e], row_wise, rtol=1e-6, atol=0)


def _f32_patterns() -> np.ndarray:
    """fp32 bit patterns covering every exponent and sign with the low 16 bits
    at 0, 1, just below / at / just above the halfway point and all ones, the
    kept bit (bit 16) both 0 and 1, plus the overflow boundary, the largest
    finite values, infinities, zeros and a random sweep (no NaNs: out of scope)."""
    pats = []
    for sign in (0, 1):
        for e in range(0, 255):
            for keep in (0, 1):
                for upper in (0x00, 0x15, 0x3F):          # mantissa bits 17..22
                    for low in (0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
                        pats.append((sign << 31) | (e << 23) | (upper << 17) | (keep << 16) | low)
    pats += [0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0x7F800000, 0xFF800000, 0x00000000, 0x80000000,
             0x00008000, 0x00018000, 0x80008000]
    rng = np.random.default_rng(7)
    rnd = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    rnd = rnd[((rnd >> 23) & 0xFF) != 0xFF]            # drop NaN / inf exponents from the random part
    return np.concatenate([np.array(pats, dtype=np.uint32), rnd])


def test_bf16_round_matches_torch_cast_on_fp32_patterns():
    """moe.bf16_round on fp32-representable values (its first step, fp64 ->
    fp32, is then exact) equals torch's round-to-nearest-even fp32 -> bf16
    cast bit for bit, ties to even included, overflow to infinity included."""
    bits = _f32_patterns()
    f = bits.view(np.float32)
    ours = moe.bf16_round(f.astype(np.float64)).astype(np.float32).view(np.uint32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float32).numpy().view(np.uint32)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [hex(int(bits[i])) for i in bad[:8]]
    # spot values: a tie rounds to the even neighbour, one unit above it rounds up
    one = np.float64(1.0)
    assert moe.bf16_round(np.array([one + 2.0 ** -8]))[0] == one               # tie, even below
    assert moe.bf16_round(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6  # tie, even above
    assert moe.bf16_round(np.array([one + 2.0 ** -8 + 2.0 ** -20]))[0] == one + 2.0 ** -7


def test_bf16_round_of_fp64_values_is_rounding_via_fp32():
    """For general fp64 values the result is the fp32 rounding followed by the
    bf16 rounding (what the docstring states), checked against torch doing the
    same two casts, and it is always one of the two bf16 neighbours of v."""
    rng = np.random.default_rng(8)
    v = rng.standard_normal(100_000) * np.exp2(rng.integers(-30, 30, size=100_000))
    ours = moe.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ours, ref)
    lo = torch.from_numpy(v).to(torch.bfloat16).double().numpy()   # some bf16 neighbour of v
    assert np.all(np.abs(ours - v) <= np.abs(v) * 2.0 ** -8 * (1 + 2.0 ** -15))
    assert np.all((ours == lo) | (np.abs(ours - lo) <= np.abs(v) * 2.0 ** -7))
