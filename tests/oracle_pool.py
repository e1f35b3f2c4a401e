"""Runs the oracle's NVFP4 quantizer over row chunks of a full-size matrix in
a pool of spawned processes (the oracle itself is unchanged: NVFP4 blocks lie
within a row, so quantizing row chunks with the whole tensor's scale s_t is
the same computation as quantizing the whole matrix)."""
import multiprocessing as mp
import os

import numpy as np

from oracle import quant as Q


def _rows(args):
    W, s_t = args
    c, s, _ = Q.nvfp4_quantize(W, s_t=s_t)
    return c, s


def nvfp4_quantize_parallel(W, procs=None):
    W = np.ascontiguousarray(W, dtype=np.float32)
    s_t = Q.nvfp4_tensor_scale(W)
    n = procs or max(1, min(16, os.cpu_count() or 1))
    chunks = np.array_split(W, n, axis=0)
    with mp.get_context("spawn").Pool(n) as pool:
        parts = pool.map(_rows, [(ch, s_t) for ch in chunks])
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]), s_t
