"""Runs the oracle's expert-weight fake-quantisation on all host cores.

Workers are spawned (never forked: the test process has a CUDA context) and
exchange the weights through shared memory.  Each worker calls
oracle.mx.fake_quant on a slice of rows; the result equals
oracle.moe.expert_weights(...) element for element."""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np
import torch


def _work(task):
    in_name, in_shape, out_name, out_shape, transpose, r0, r1 = task
    from oracle import mx
    shm_in = shared_memory.SharedMemory(name=in_name)
    shm_out = shared_memory.SharedMemory(name=out_name)
    try:
        src = np.ndarray(in_shape, dtype=np.uint16, buffer=shm_in.buf)
        out = np.ndarray(out_shape, dtype=np.float64, buffer=shm_out.buf)
        block = src[:, r0:r1].T if transpose else src[r0:r1]
        vals = (block.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        out[r0:r1] = mx.fake_quant(vals)
    finally:
        shm_in.close()
        shm_out.close()
    return r0


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class WeightQuantPool:
    def __init__(self, workers: int | None = None):
        n = workers or min(16, os.cpu_count() or 1)
        self.ex = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
        self.n = n

    def close(self):
        self.ex.shutdown()

    def _fq(self, w_bits: np.ndarray, transpose: bool) -> np.ndarray:
        rows_out = w_bits.shape[1] if transpose else w_bits.shape[0]
        cols_out = w_bits.shape[0] if transpose else w_bits.shape[1]
        shm_in = shared_memory.SharedMemory(create=True, size=w_bits.nbytes)
        shm_out = shared_memory.SharedMemory(create=True, size=rows_out * cols_out * 8)
        try:
            np.ndarray(w_bits.shape, dtype=np.uint16, buffer=shm_in.buf)[:] = w_bits
            step = max(1, -(-rows_out // (4 * self.n)))
            tasks = [(shm_in.name, w_bits.shape, shm_out.name, (rows_out, cols_out), transpose, r, min(rows_out, r + step))
                     for r in range(0, rows_out, step)]
            list(self.ex.map(_work, tasks))
            return np.ndarray((rows_out, cols_out), dtype=np.float64, buffer=shm_out.buf).copy()
        finally:
            shm_in.close()
            shm_in.unlink()
            shm_out.close()
            shm_out.unlink()

    def expert_weights(self, w_gate_up_e: torch.Tensor, w_down_e: torch.Tensor) -> dict:
        """Same as oracle.moe.expert_weights(w_gate_up_e, w_down_e)."""
        g = _bits(w_gate_up_e)
        d = _bits(w_down_e)
        return {"wg": self._fq(g, False), "wd": self._fq(d, False), "wdT": self._fq(d, True),
                "wguT": self._fq(g, True)}
