"""CPU oracle for the decode-step weight stream.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
library under ``bit_weight_streaming_gb300`` never imports it and has no CPU
fallback; the two share no code (only the seeded generators in ``synth``).

What it computes, written plainly from the pages (numpy; FP32 where the method
makes a rounding decision, FP64 for every product and sum):

* ``formats``   E2M1 / E4M3 / E8M0 codecs and round-to-nearest-even encoders,
                BF16 rounding.
* ``quant``     NVFP4, MXFP4 and row-wise FP8 quantizers; MXFP8 activations.
* ``products``  dequantization and exact (FP64) matrix-vector products.
* ``model``     SwiGLU MLP, top-k MoE with a shared expert, weightless RMSNorm,
                and the layer recipe of the dense and MoE stacks.
* ``accounting`` algorithmic bytes of each workload.
* ``tolerance`` the comparison bound the GPU results must meet.

Page references in docstrings use these short names:
  [Spark27B]  mdjawad.com, DGX Spark post on Qwen3.8-27B NVFP4 decoding
  [SparkSpec] carouter.ai, "Tuning speculative decoding on CARouter's DGX Spark"
  [LingMoE]   magicnetworld.com, reading of "3 Ways to Boost MoE Inference on
              NVIDIA DGX Spark" (Ling-3.0-flash, sections numbered 一 to 十八)

Every function here is pinned by the ``-m "not gpu"`` tests to values that
do not come from this code (closed forms, brute force, page figures,
library routines); none is unpinned.
"""
from . import formats, quant, products, model, accounting, tolerance  # noqa: F401
