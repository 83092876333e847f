"""The seeded input recipe (CPU only): draw order, distributions, dtypes and
determinism of recompute_kda_chunkwise_gb300.inputs, as stated in its module
docstring."""
import torch

from recompute_kda_chunkwise_gb300 import WORKLOADS, Workload, make_inputs, make_states


def _draws(seed, shapes):
    gen = torch.Generator().manual_seed(seed)
    return [torch.randn(s, generator=gen) for s in shapes]


def test_kda_draw_order_and_cast():
    w = WORKLOADS["tiny_t256_h2_d64_bf16"]
    inp = make_inputs(w)
    S, H, D = w.total_tokens, w.H, w.D
    q, k, v, g, b, dO = _draws(w.seed, [(S, H, D)] * 4 + [(S, H), (S, H, D)])
    for name, ref in zip(["q", "k", "v", "g", "beta", "dO"], [q, k, v, g, b, dO]):
        assert inp[name].dtype == torch.bfloat16
        assert torch.equal(inp[name], ref.to(torch.bfloat16)), name
    assert torch.equal(inp["A_log"], torch.zeros(H)) and torch.equal(inp["dt_bias"], torch.zeros(H, D))
    assert inp["cu_seqlens"].tolist() == [0, 256]


def test_gdn2_draws_erase_and_write_in_place_of_beta():
    w = WORKLOADS["gdn2_b10_t512_h12_d64_f32"]
    inp = make_inputs(w)
    S, H, D = w.total_tokens, w.H, w.D
    draws = _draws(w.seed, [(S, H, D)] * 7)
    for name, ref in zip(["q", "k", "v", "g", "erase", "write", "dO"], draws):
        assert inp[name].dtype == torch.float32 and torch.equal(inp[name], ref), name
    assert "beta" not in inp


def test_gate_distribution_parameters_and_param_draws():
    w = Workload("gate", (4096,), 2, 64, "f32", seed=5, gate_mean=-6.0, gate_std=2.0, param_std=0.5)
    inp = make_inputs(w)
    g = inp["g"].double()
    assert abs(g.mean().item() + 6.0) < 0.05 and abs(g.std().item() - 2.0) < 0.05
    assert inp["A_log"].abs().sum() > 0 and inp["dt_bias"].abs().sum() > 0


def test_deterministic_and_states_seeded_apart():
    w = WORKLOADS["b10_t512_h12_d64_f32"]
    a, b = make_inputs(w), make_inputs(w)
    assert all(torch.equal(a[n], b[n]) for n in a)
    s1, s2 = make_states(w), make_states(w)
    assert torch.equal(s1["h0"], s2["h0"]) and torch.equal(s1["dht"], s2["dht"])
    assert s1["h0"].shape == (w.num_seqs, w.H, w.D, w.D)
    assert abs(s1["h0"].std().item() - 0.5) < 0.01 and abs(s1["dht"].std().item() - 0.05) < 0.001
