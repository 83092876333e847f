"""Seeded synthetic inputs for KDA forward + backward.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes, dtypes and distributions of the workloads measured in
"KDA Memory with Recompute: FLA vs cuDNN Frontend FROST" (section "Sources and
measurement configuration": D128, bf16 Q/K/V/raw gate/raw beta/dO, fp32
A_log = dt_bias = 0, equal-length packed sequences) and the small fp32 preset
of "KDA at the production shape ..." (section 2, b=10 t=512 h=12 K=V=64).
Both the CUDA path and the oracle consume exactly these tensors.

Recipe: a torch.Generator on the requested device, seeded with the workload's
seed, draws in this fixed order: Q, K, V, raw gate, raw beta, dO (each in
fp32, then cast to the workload dtype), then -- only when ``param_std`` > 0 --
A_log and dt_bias (fp32). Otherwise A_log and dt_bias are zeros. The raw gate
is N(gate_mean, gate_std); everything else is N(0, 1).

GDN-2 workloads (``gates == "channel"``, the channel-wise erase / write gate
form of "KDA at the production shape ...", section 1.6) draw the raw erase
gate and the raw write gate, both [S,H,D] N(0, 1), in place of raw beta:
Q, K, V, raw gate, raw erase, raw write, dO, then A_log / dt_bias as above.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    lengths: tuple          # tokens per packed sequence
    H: int
    D: int
    dtype: str = "bf16"    # "bf16" or "f32"
    seed: int = 0
    gate_mean: float = 0.0
    gate_std: float = 1.0
    param_std: float = 0.0  # std of A_log / dt_bias draws (0 -> zeros)
    scale: float = 1.0
    gates: str = "scalar"   # "scalar" (KDA beta) or "channel" (GDN-2 erase / write gates)
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _equal(n, t):
    return tuple([t] * n)


# The five workloads (seed = 20260 + index; the H sweep of workload 4 uses
# sub-seeds 202641 and 202642).
WORKLOADS = {
    "tiny_t256_h2_d64_bf16": Workload("tiny_t256_h2_d64_bf16", _equal(1, 256), 2, 64, "bf16", 20261),
    "b10_t512_h12_d64_f32": Workload("b10_t512_h12_d64_f32", _equal(10, 512), 12, 64, "f32", 20262),
    "mbs8_8k_h16_d128_bf16": Workload("mbs8_8k_h16_d128_bf16", _equal(8, 8192), 16, 128, "bf16", 20263),
    "mbs2_8k_h96_d128_bf16_gate2": Workload("mbs2_8k_h96_d128_bf16_gate2", _equal(2, 8192), 96, 128,
                                            "bf16", 20264, gate_std=2.0),
    "mbs1_8k_h64_d128_bf16_gate2": Workload("mbs1_8k_h64_d128_bf16_gate2", _equal(1, 8192), 64, 128,
                                            "bf16", 202641, gate_std=2.0),
    "mbs1_8k_h128_d128_bf16_gate2": Workload("mbs1_8k_h128_d128_bf16_gate2", _equal(1, 8192), 128, 128,
                                             "bf16", 202642, gate_std=2.0),
    "mbs1_128k_h96_d128_bf16": Workload("mbs1_128k_h96_d128_bf16", _equal(1, 131072), 96, 128,
                                        "bf16", 20265),
    # The long-context shape cut to 8192 tokens: the same launch configuration
    # (96 sequence-heads) for profiler captures that must stay small.
    "mbs1_8k_h96_d128_bf16": Workload("mbs1_8k_h96_d128_bf16", _equal(1, 8192), 96, 128, "bf16", 20266),
    # Unequal-length packing: 8 sequences of mean length 1024 (8192 tokens),
    # the shape of the pages' varlen forward comparisons, at H = 96.
    "varlen8_8k_h96_d128_bf16": Workload("varlen8_8k_h96_d128_bf16",
                                         (512, 1536, 768, 1280, 256, 1792, 1024, 1024), 96, 128,
                                         "bf16", 20267),
    # GDN-2 (channel-wise erase / write gates): the pages' own fp32 preset
    # shape (b=10 t=512 h=12 K=V=64) and a bf16 D = 128 shape of the
    # MBS8 x 8K x H16 workload.
    "gdn2_b10_t512_h12_d64_f32": Workload("gdn2_b10_t512_h12_d64_f32", _equal(10, 512), 12, 64, "f32",
                                          20268, gates="channel"),
    "gdn2_mbs8_8k_h16_d128_bf16": Workload("gdn2_mbs8_8k_h16_d128_bf16", _equal(8, 8192), 16, 128,
                                           "bf16", 20269, gates="channel"),
}
HEADLINE = "mbs1_128k_h96_d128_bf16"


def cu_seqlens_of(lengths, device="cpu") -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def make_inputs(w: Workload, device="cpu", with_dO: bool = True) -> dict:
    """Draw the workload's tensors on ``device`` (see the module recipe)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(w.seed))
    dt = _DTYPES[w.dtype]
    S, H, D = w.total_tokens, w.H, w.D

    def normal(shape, mean=0.0, std=1.0):
        x = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if mean != 0.0:
            x.add_(mean)
        return x.to(dt)

    out = {}
    out["q"] = normal((S, H, D))
    out["k"] = normal((S, H, D))
    out["v"] = normal((S, H, D))
    out["g"] = normal((S, H, D), w.gate_mean, w.gate_std)
    if w.gates == "channel":
        out["erase"] = normal((S, H, D))
        out["write"] = normal((S, H, D))
    else:
        out["beta"] = normal((S, H))
    out["dO"] = normal((S, H, D)) if with_dO else None
    if w.param_std > 0:
        out["A_log"] = torch.randn((H,), generator=gen, device=dev) * w.param_std
        out["dt_bias"] = torch.randn((H, D), generator=gen, device=dev) * w.param_std
    else:
        out["A_log"] = torch.zeros((H,), device=dev)
        out["dt_bias"] = torch.zeros((H, D), device=dev)
    out["cu_seqlens"] = cu_seqlens_of(w.lengths, dev)
    return out


def make_states(w: Workload, device="cpu", seed_offset: int = 1000, dht_std: float = 0.05) -> dict:
    """Seeded initial states h0 ~ N(0, 0.5^2) and final-state gradients
    dht ~ N(0, dht_std^2), both [N, H, D, D] float32 (rows: key channel),
    drawn from their own generator (seed = workload seed + seed_offset).
    0.05 is the size of the state gradient inside a sequence at these
    workloads (entries of order 0.01 - 0.1), i.e. what a following segment's
    initial-state gradient hands back."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(w.seed) + seed_offset)
    shape = (w.num_seqs, w.H, w.D, w.D)
    h0 = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * 0.5
    dht = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * dht_std
    return {"h0": h0, "dht": dht}
