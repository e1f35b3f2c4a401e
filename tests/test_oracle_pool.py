"""The row-chunked, multi-process run of the oracle's NVFP4 quantizer used by
the full-size GPU tests gives the same codes as one call on the whole matrix."""
import numpy as np

from oracle import quant as Q
from tests.oracle_pool import nvfp4_quantize_parallel
import synth


def test_parallel_quantize_equals_whole_matrix():
    W = synth.weight_fp32((67, 512), seed=9, index=3).numpy()
    W[5, 17] = 0.9          # an outlier sets the tensor scale
    c, s, t = Q.nvfp4_quantize(W)
    cp, sp, tp = nvfp4_quantize_parallel(W, procs=3)
    assert tp == t and np.array_equal(cp, c) and np.array_equal(sp, s)
