"""Seeded synthetic workloads for the grouped MoE expert MLP.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic (no quantisation, routing, GEMM or activation).  Both the
CUDA path (through the tests and bench.py) and the CPU oracle take their inputs
from here, so the two sides always see the same bytes.

Workload shapes.  The pages measure Mixtral-8x7B training (BioNeMo Uses Grouped
Kernels and MXFP8, "Training benchmark", Fig. 5) and motivate MXFP8 with long
genomic sequences ("Reducing memory pressure with MXFP8").  No dataset is
involved: seeded normal draws with the shapes below stand in for activations,
master weights, router logits and upstream gradients.

Generation recipe (per named workload with index c):
  SeedSequence(1000 + c) spawned into six children used in this fixed order:
  logits, x, W_gate_up, W_down, dy, zipf; each drives a numpy
  Generator(PCG64).  The two weight children are spawned once more into one
  stream per expert (drawn in parallel threads, each expert from its own
  stream, so the result does not depend on the thread count).
  fp32 normal draws are rounded to bf16 (round-to-nearest-even, via torch).
  logits ~ N(0,1) fp32; x ~ N(0,1); W ~ N(0, 0.02); dy ~ N(0,1).

Skewed routing ("skew"): two seeded experts receive no tokens; the other six
are ranked by a seeded permutation and given finite Zipf weights r^-1.2
(r = 1..6).  Each token draws its first expert from those weights and its
second from the remaining five (renormalised).  The logits of the two drawn
experts are N(0,1); every other logit is N(0,1) - 64, so that top-2 selection
on the logits returns exactly the drawn pair and the routing probability is
the softmax over the drawn pair's logits.  If any non-empty split is a
multiple of 128 the seed is advanced by one (recorded in ``seed_used``).
"""
from __future__ import annotations

import concurrent.futures as cf
import dataclasses
import os

import numpy as np
import torch

WEIGHT_STD = 0.02


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed index c (SeedSequence(1000 + c))
    T: int              # tokens
    H: int              # hidden
    I: int              # intermediate (gate-up out_features = 2*I)
    E: int              # experts
    k: int              # top-k
    backward: bool = True
    skew: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k

    def gemm_flops(self, backward: bool | None = None) -> float:
        """Algorithmic GEMM flops: 6*R*H*I forward, 18*R*H*I forward+backward."""
        bwd = self.backward if backward is None else backward
        return (18.0 if bwd else 6.0) * self.R * self.H * self.I


WORKLOADS = {
    "tiny": Workload("tiny", 1, T=256, H=128, I=256, E=4, k=2, backward=False),
    "mid": Workload("mid", 2, T=4096, H=1024, I=2816, E=8, k=2),
    "mixtral": Workload("mixtral", 3, T=16384, H=4096, I=14336, E=8, k=2),
    "skew": Workload("skew", 4, T=16384, H=4096, I=14336, E=8, k=2, skew=True),
    "fine": Workload("fine", 5, T=8192, H=2048, I=1024, E=64, k=8),
    # one expert of the Mixtral layer at its uniform load (4096 rows): the same
    # per-tile work as "mixtral" with ~1.5 GB on the device, for profiler captures
    "mixtral_e1": Workload("mixtral_e1", 6, T=4096, H=4096, I=14336, E=1, k=1),
    # the Mixtral layer's tokens (x and dy at full size, top-2 of 8 experts)
    # with a narrow intermediate dimension: the activation quantisers' full
    # work with ~3 GB on the device, for profiler captures
    "mixtral_tokens": Workload("mixtral_tokens", 7, T=16384, H=4096, I=1024, E=8, k=2),
}


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 numpy -> bf16 torch CPU tensor (round-to-nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal_bf16(rng: np.random.Generator, shape, std: float, chunk_rows: int | None = None) -> torch.Tensor:
    """Normal draws rounded to bf16; large tensors are drawn in leading-dim chunks
    (same stream, same order) to bound host memory."""
    if chunk_rows is None or shape[0] <= chunk_rows:
        a = rng.standard_normal(shape, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        return to_bf16(a)
    out = torch.empty(shape, dtype=torch.bfloat16)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        a = rng.standard_normal((e - s,) + tuple(shape[1:]), dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        out[s:e] = to_bf16(a)
    return out


def _expert_weights(ss: np.random.SeedSequence, E: int, shape, std: float) -> torch.Tensor:
    """[E, *shape] bf16, expert e drawn from the e-th child of ``ss``."""
    out = torch.empty((E,) + tuple(shape), dtype=torch.bfloat16)
    children = ss.spawn(E)

    def one(e):
        g = np.random.Generator(np.random.PCG64(children[e]))
        a = g.standard_normal(tuple(shape), dtype=np.float32)
        a *= np.float32(std)
        out[e] = to_bf16(a)

    workers = max(1, min(E, os.cpu_count() or 1, 16))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(one, range(E)))
    return out


def _skew_logits(rng_logits, rng_zipf, T, E, k):
    assert k == 2 and E >= 3
    empty = rng_zipf.choice(E, size=2, replace=False)
    live = np.array([e for e in range(E) if e not in set(empty.tolist())])
    live = live[rng_zipf.permutation(live.size)]
    w = np.arange(1, live.size + 1, dtype=np.float64) ** -1.2
    w /= w.sum()
    first = rng_zipf.choice(live.size, size=T, p=w)
    second = np.empty(T, dtype=np.int64)
    u = rng_zipf.random(T)
    for j in range(live.size):          # second draw from the remaining five
        sel = first == j
        if not sel.any():
            continue
        w2 = w.copy()
        w2[j] = 0.0
        c = np.cumsum(w2 / w2.sum())
        second[sel] = np.minimum(np.searchsorted(c, u[sel], side="right"), live.size - 1)
    e1, e2 = live[first], live[second]
    base = rng_logits.standard_normal((T, E), dtype=np.float32)
    logits = base - np.float32(64.0)
    rows = np.arange(T)
    logits[rows, e1] = base[rows, e1]
    logits[rows, e2] = base[rows, e2]
    counts = np.bincount(np.concatenate([e1, e2]), minlength=E)
    return logits, counts, empty


def make_inputs(wl: Workload | str, seed_offset: int = 0, with_weights: bool = True) -> dict:
    """Draw one workload's inputs.

    Returns a dict with torch CPU tensors: logits fp32 [T,E], x bf16 [T,H],
    w_gate_up bf16 [E,2I,H], w_down bf16 [E,H,I], dy bf16 [T,H] (if the workload
    has a backward pass), plus ``seed_used`` and, for the skewed workload,
    ``drawn_counts``/``empty_experts``.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    off = seed_offset
    while True:
        ss = np.random.SeedSequence(1000 + wl.index + off)
        kids = ss.spawn(6)
        r_logits, r_x, _, _, r_dy, r_zipf = [np.random.Generator(np.random.PCG64(s)) for s in kids]
        ss_wgu, ss_wd = kids[2], kids[3]
        out: dict = {"seed_used": 1000 + wl.index + off}
        if wl.skew:
            logits, counts, empty = _skew_logits(r_logits, r_zipf, wl.T, wl.E, wl.k)
            if any(c > 0 and c % 128 == 0 for c in counts):
                off += 1
                continue
            out["drawn_counts"] = counts
            out["empty_experts"] = np.sort(empty)
        else:
            logits = r_logits.standard_normal((wl.T, wl.E), dtype=np.float32)
        break
    out["logits"] = torch.from_numpy(logits)
    out["x"] = _normal_bf16(r_x, (wl.T, wl.H), 1.0, chunk_rows=4096)
    if with_weights:
        out["w_gate_up"] = _expert_weights(ss_wgu, wl.E, (2 * wl.I, wl.H), WEIGHT_STD)
        out["w_down"] = _expert_weights(ss_wd, wl.E, (wl.H, wl.I), WEIGHT_STD)
    if wl.backward:
        out["dy"] = _normal_bf16(r_dy, (wl.T, wl.H), 1.0, chunk_rows=4096)
    return out


def make_case(T: int, H: int, I: int, E: int, k: int, seed: int, empty_experts=(),
              logit_scale: float = 1.0) -> dict:
    """A small seeded case of arbitrary shape for parity tests.

    ``empty_experts`` are pushed out of every token's top-k by lowering their
    logits by 64, so they receive no rows (exercises empty groups).
    """
    ss = np.random.SeedSequence(seed)
    r_logits, r_x, r_wgu, r_wd, r_dy = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]
    logits = r_logits.standard_normal((T, E), dtype=np.float32) * np.float32(logit_scale)
    for e in empty_experts:
        logits[:, e] -= np.float32(64.0)
    return {
        "seed_used": seed,
        "logits": torch.from_numpy(logits),
        "x": _normal_bf16(r_x, (T, H), 1.0),
        "w_gate_up": _normal_bf16(r_wgu, (E, 2 * I, H), WEIGHT_STD),
        "w_down": _normal_bf16(r_wd, (E, H, I), WEIGHT_STD),
        "dy": _normal_bf16(r_dy, (T, H), 1.0),
    }


def random_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    """Seeded bf16 normal matrix (quantiser and GEMM unit cases)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed)))
    return _normal_bf16(rng, tuple(shape), std)
