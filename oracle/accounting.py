"""Algorithmic bytes of the weight stream.

[Spark27B] § "Decode speed is bytes divided by bandwidth": a matrix of
d_out x d_in weights at b bits per weight is d_out*d_in*b/8 bytes and must be
read once per decode step; the step time is bytes read divided by achieved
bandwidth. Bytes counted here are the codes plus the block (or row) scales
that a step must read; the 4-byte per-tensor scales are left out.
[LingMoE] §四: for a MoE only the activated experts are read.
"""
from dataclasses import dataclass, field

NVFP4_BYTES_PER_WEIGHT = 0.5 + 1.0 / 16      # E2M1 code + E4M3 per 16
MXFP4_BYTES_PER_WEIGHT = 0.5 + 1.0 / 32      # E2M1 code + E8M0 per 32


def nvfp4_bytes(d_out, d_in):
    return d_out * d_in // 2 + d_out * d_in // 16


def mxfp4_bytes(d_out, d_in):
    return d_out * d_in // 2 + d_out * d_in // 32


def fp8_rowwise_bytes(rows, cols):
    return rows * cols + 4 * rows


def bits_per_weight_nvfp4():
    """4 + 8/16 = 4.5 bits ([Spark27B] § "Fewer bytes per weight: NVFP4")."""
    return 8.0 * NVFP4_BYTES_PER_WEIGHT


# ---- the dense 27B-shape stack -------------------------------------------

HIDDEN_27B = 5120
MLP_INTER_27B = 17408
N_LAYERS_27B = 64
VOCAB_27B = 248320


def layer_kind_27b(i):
    """Every fourth layer is full attention, the other 48 Gated DeltaNet
    ([Spark27B] § "Decode speed is bytes divided by bandwidth")."""
    return "attn" if i % 4 == 3 else "gdn"


def mixer_shapes_27b(kind, hidden=HIDDEN_27B):
    """Token-mixer projections (d_out, d_in). The pages give only the
    largest (12288 x 5120) and the stack total (17.83 GB); these shapes are
    this project's reading, chosen so the all-NVFP4 stack totals 17.824 GB."""
    if kind == "attn":
        return {"in": [(12288, hidden), (1024, hidden), (1024, hidden)],
                "out": (hidden, 6144)}
    return {"in": [(46336, hidden)], "out": (hidden, 6144)}


def mlp_shapes(hidden, inter):
    return {"gate": (inter, hidden), "up": (inter, hidden), "down": (hidden, inter)}


def stack_27b_layer_bytes(i, hidden=HIDDEN_27B, inter=MLP_INTER_27B):
    m = mixer_shapes_27b(layer_kind_27b(i), hidden)
    b = sum(nvfp4_bytes(*s) for s in m["in"]) + nvfp4_bytes(*m["out"])
    b += sum(nvfp4_bytes(*s) for s in mlp_shapes(hidden, inter).values())
    return b


def stack_27b_bytes(n_layers=N_LAYERS_27B):
    layers = sum(stack_27b_layer_bytes(i) for i in range(n_layers))
    head = fp8_rowwise_bytes(VOCAB_27B, HIDDEN_27B)
    return {"layers": layers, "head": head, "total": layers + head}


# ---- the Ling-3.0-flash-shape MoE stack ----------------------------------

HIDDEN_MOE = 2560
EXPERT_INTER = 768
N_EXPERTS = 512
TOPK = 8
N_MOE_LAYERS = 40
N_DENSE_LAYERS = 2
DENSE_INTER_MOE = 9 * EXPERT_INTER          # reading: 6912
VOCAB_MOE = 157184


def expert_bytes(hidden=HIDDEN_MOE, inter=EXPERT_INTER):
    """gate + up + down of one expert in MXFP4."""
    return 2 * mxfp4_bytes(inter, hidden) + mxfp4_bytes(hidden, inter)


def moe_step_bytes(distinct_per_layer, n_dense=N_DENSE_LAYERS):
    """distinct_per_layer: list of #distinct routed experts per MoE layer
    (the shared expert is added here)."""
    e = expert_bytes()
    moe = sum((k + 1) * e for k in distinct_per_layer)
    dense = n_dense * (2 * mxfp4_bytes(DENSE_INTER_MOE, HIDDEN_MOE)
                       + mxfp4_bytes(HIDDEN_MOE, DENSE_INTER_MOE))
    head = fp8_rowwise_bytes(VOCAB_MOE, HIDDEN_MOE)
    return {"moe": moe, "dense": dense, "head": head, "total": moe + dense + head}


# ---- the five workloads ----------------------------------------------------

@dataclass
class Workload:
    name: str
    n_tokens: int
    bytes: int
    detail: dict = field(default_factory=dict)


def config_bytes(cfg, n_tokens=None, distinct_per_layer=None):
    """Algorithmic weight bytes of workload cfg (0..4)."""
    if cfg == 0:
        return nvfp4_bytes(MLP_INTER_27B, HIDDEN_27B)
    if cfg == 1:
        return sum(nvfp4_bytes(*s) for s in mlp_shapes(HIDDEN_27B, MLP_INTER_27B).values())
    if cfg == 2:
        return config_bytes(1) + nvfp4_bytes(12288, HIDDEN_27B) + nvfp4_bytes(HIDDEN_27B, 6144)
    if cfg == 3:
        return stack_27b_bytes()["total"]
    if cfg == 4:
        if distinct_per_layer is None:
            distinct_per_layer = [TOPK] * N_MOE_LAYERS
        return moe_step_bytes(distinct_per_layer)["total"]
    raise ValueError(cfg)
