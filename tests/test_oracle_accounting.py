"""Byte-account pins against the figures the pages print (CPU only)."""
import pytest

from oracle import accounting as B
from tests.conftest import load_golden

G = load_golden("page_figures.json")


def test_bits_per_weight():
    assert B.bits_per_weight_nvfp4() == G["nvfp4_bits_per_weight"]["value"]


def test_config0_bytes():
    d_out, d_in = G["mlp_gate_shape"]["value"]
    assert B.config_bytes(0) == d_out * d_in * 4.5 / 8 == 50_135_040


def test_stack_27b_matches_pages():
    s = B.stack_27b_bytes()
    assert s["layers"] == 17_824_481_280
    assert abs(s["layers"] / 1e9 - G["stack_gb"]["value"]) / G["stack_gb"]["value"] < 1e-3
    V, d = G["head_shape"]["value"]
    assert s["head"] == V * d + 4 * V
    assert round(s["head"] / 1e9, 2) == G["head_gb"]["value"]
    assert round(s["total"] / 1e9, 2) == G["step_gb"]["value"]
    kinds = [B.layer_kind_27b(i) for i in range(64)]
    assert kinds.count("attn") == G["layers"]["full_attention"]
    assert kinds.count("gdn") == G["layers"]["linear_attention"]


def test_pages_ceiling_arithmetic():
    c = G["ceiling_ms_at_273"]
    step = G["step_gb"]["value"]
    assert round(step / c["bw_gbs"] * 1e3, 1) == c["value"]
    assert round(c["bw_gbs"] / step, 1) == c["tok_s"]
    m = G["measured_step_ms"]
    assert round(step / (m["value"] / 1e3)) == m["achieved_gbs"]


def test_pages_mixed_checkpoint_mlp_share():
    """The pages' real checkpoint: NVFP4 MLPs in layers 0-55, FP8 in the last
    eight; the MLPs are 59% of the 17.83 GB of layer bytes."""
    mlp_w = 3 * 17408 * 5120
    mc = G["mixed_checkpoint"]
    b = mc["nvfp4_mlp_layers"] * mlp_w * B.NVFP4_BYTES_PER_WEIGHT + mc["fp8_mlp_layers"] * mlp_w * 1.0
    assert round(b / (G["stack_gb"]["value"] * 1e9), 2) == G["mlp_share_of_layer_bytes"]["value"]


def test_intensity_16_over_b():
    for fmt, b in (("nvfp4", 4), ("fp8", 8)):
        assert 16 / b == G["intensity_per_bits"][fmt]


def test_ling_head_and_step():
    V, d = G["ling_vocab"]["value"], G["ling_hidden"]["value"]
    h = G["ling_head_params_m"]
    assert round(V * d / 1e6, 2) == h["value"]
    assert round(V * d * 2 / 1e9, 3) == h["bf16_gb"]
    assert round(V * d / 1e9, 3) == h["fp8_gb"]
    be = G["ling_beff"]
    assert round(be["step_gb"] / be["tpot_ms"] * 1e3) == be["beff_gbs"]
    assert round(be["beff_gbs"] / 273, 2) == be["u"]


def test_config4_bytes():
    e = B.expert_bytes()
    assert e == 3_133_440
    assert B.config_bytes(4) == 1_587_460_096
    assert B.config_bytes(4, distinct_per_layer=[30] * 40) == \
        40 * 31 * e + B.moe_step_bytes([0] * 40)["dense"] + B.moe_step_bytes([0] * 40)["head"]


def test_config2_bytes():
    assert B.config_bytes(1) == 150_405_120
    assert B.config_bytes(2) == 203_489_280


def test_mixed_checkpoint_composition_matches_pages():
    """The mixed-checkpoint workload (FP8 mixers everywhere, NVFP4 MLPs in
    layers 0-55, FP8 MLPs in 56-63, linear-attention projections
    14336x5120 / 5120x8192): its layers come within 0.5 % of the pages'
    17.83 GB, its MLPs are 59 % of them, and the step is 19.05 GB."""
    from bit_weight_streaming_gb300 import workloads as W
    fmt = W.mixed_fmt()
    size = {1: B.nvfp4_bytes, 3: B.fp8_rowwise_bytes}
    layers = mlp = 0
    for i in range(64):
        mixer_in, mixer_out, mlps = W.dense_layer_shapes(i, gdn=W.MIXED_GDN)
        mix = sum(size[fmt(i, "mixer")](*s) for s in mixer_in + [mixer_out])
        m = sum(size[fmt(i, "mlp")](*s) for s in mlps.values())
        layers += mix + m
        mlp += m
    assert abs(layers / 1e9 - G["stack_gb"]["value"]) / G["stack_gb"]["value"] < 5e-3
    assert round(mlp / layers, 2) == G["mlp_share_of_layer_bytes"]["value"]
    V, d = G["head_shape"]["value"]
    assert round((layers + B.fp8_rowwise_bytes(V, d)) / 1e9, 2) == 19.05
