"""Pins the end-to-end stack tolerance: perturb the oracle's activations
before each BF16 rounding by up to 2^-14 relative (well above what FP32
accumulation of a few thousand exact products can differ from FP64), which
flips a fraction of the BF16 roundings, and check that the logits move far
less than the slack the GPU stack test allows."""
import numpy as np

from oracle import model as M, formats as F, products as P, quant as Q
from tests.stack_util import STACK_SLACK
import synth


def _mk(shape, i, fmt="nv"):
    W = synth.weight_fp32(shape, seed=77, index=i).numpy()
    if fmt == "nv":
        return P.nvfp4_dequantize(*Q.nvfp4_quantize(W))
    return P.fp8_dequantize(*Q.fp8_rowwise_quantize(W))


def test_stack_flip_sensitivity_is_inside_slack(monkeypatch):
    d, inter, V = 256, 512, 777
    layers = []
    idx = 0
    for i in range(4):
        if i % 4 == 3:
            ins = [(384, d), (64, d), (64, d)]
        else:
            ins = [(640, d)]
        L = {"in": [_mk(s, idx + j) for j, s in enumerate(ins)], "out": _mk((d, 192), idx + 10),
             "gate": _mk((inter, d), idx + 11), "up": _mk((inter, d), idx + 12), "down": _mk((d, inter), idx + 13)}
        idx += 20
        layers.append(L)
    head = _mk((V, d), 999, "f8")
    x0 = F.round_bf16(synth.activation_bf16(4, d, seed=77).float().numpy())
    base, _, _ = M.decode_stack(x0, layers, head)
    rng = np.random.default_rng(0)
    orig = F.round_bf16

    def perturbed(v):
        v = np.asarray(v, np.float64)
        return orig(v * (1.0 + rng.uniform(-2.0 ** -14, 2.0 ** -14, size=v.shape)))

    worst = 0.0
    for _ in range(3):
        monkeypatch.setattr(M, "round_bf16", perturbed)
        got, _, _ = M.decode_stack(x0, layers, head)
        monkeypatch.setattr(M, "round_bf16", orig)
        rms = np.sqrt(np.mean(base ** 2, axis=1, keepdims=True))
        worst = max(worst, float(np.max(np.abs(got - base) / rms)))
    print(f'worst |dlogit| / rms(logits) = {worst:.3g}')
    assert 0.0 < worst < STACK_SLACK / 2, worst
