"""GPU parity of the GDN-2 operator (channel-wise erase and write gates,
kda_gdn2_fwd / kda_gdn2_bwd through the C ABI) against the fp64 oracle's
GDN-2 mode, element by element, with the same tolerances as KDA:
max|x - ref| (beyond the output's own rounding) <= 2e-2 * RMS(ref) for bf16
inputs and <= 1e-4 * RMS(ref) for fp32 inputs, for o, every gradient
(dq, dk, dv, dg, derase, dwrite, dA_log, ddt_bias) and the states. bf16
problems with D = 128 run the tensor-core forward (with and without helper
CTAs) and the fp32 CUDA-core backward; the rest, and the forced cases, the
CUDA-core kernels in both directions."""
import pytest
import torch

import oracle
from recompute_kda_chunkwise_gb300 import WORKLOADS, Workload, make_inputs, make_states
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import TOL, compare, to_dev

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
NAMES = ["o", "dq", "dk", "dv", "dg", "derase", "dwrite", "dA_log", "ddt_bias"]
ARGS = ["q", "k", "v", "g", "erase", "write", "A_log", "dt_bias", "cu_seqlens"]


def run_gpu(inp, scale, states=None, flags=0):
    h0 = dht = None
    if states is not None:
        h0, dht = states["h0"], states["dht"]
    args = [inp[n] for n in ARGS]
    r = K.gdn2_fwd(*args, scale=scale, h0=h0, final_state=states is not None, flags=flags)
    out = K.gdn2_bwd(*args, inp["dO"], r[1], scale=scale, dht=dht, want_dh0=states is not None, flags=flags)
    torch.cuda.synchronize()
    out["o"] = r[0]
    if states is not None:
        out["hT"] = r[2]
    return out


def run_oracle(inp, scale, heads=None, states=None):
    cpu = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    if heads is not None:
        idx = torch.tensor(heads)
        for n in ["q", "k", "v", "g", "erase", "write", "dO"]:
            cpu[n] = cpu[n].index_select(1, idx)
        cpu["A_log"] = cpu["A_log"].index_select(0, idx)
        cpu["dt_bias"] = cpu["dt_bias"].index_select(0, idx)
    kw = {}
    if states is not None:
        kw = dict(h0=states["h0"].cpu(), dht=states["dht"].cpu())
    return oracle.gdn2_reference(*[cpu[n] for n in ARGS], cpu["dO"], scale=scale, **kw)


def check(w: Workload, heads=None, states=False, flags=0):
    inp = to_dev(make_inputs(w, device="cpu"))
    st = to_dev(make_states(w)) if states else None
    gpu = run_gpu(inp, w.scale, st, flags)
    ref = run_oracle(inp, w.scale, heads, st)
    names = NAMES + (["hT", "dh0"] if states else [])
    return compare(gpu, ref, TOL[_DT[w.dtype]], heads=heads, names=names)


def test_pages_preset_all_heads():
    # the pages' own GDN-2 shape: 10 sequences x 512 tokens, 12 heads, K = V = 64, fp32
    check(WORKLOADS["gdn2_b10_t512_h12_d64_f32"])


def test_kernel_family_dispatch():
    # 2: tensor-core forward, CUDA-core backward
    g = K.KDA_FLAG_CHANNEL_GATES
    assert K.kernel_family(K.make_problem(64, 1, 2, 128, torch.bfloat16, flags=g)) == 2
    assert K.kernel_family(K.make_problem(64, 1, 2, 128, torch.bfloat16, flags=g | K.KDA_FLAG_FORCE_SIMT)) == 0
    assert K.kernel_family(K.make_problem(64, 1, 2, 64, torch.bfloat16, flags=g)) == 0
    assert K.kernel_family(K.make_problem(64, 1, 2, 128, torch.float32, flags=g)) == 0


def test_mbs8_8k_h16_d128_bf16_all_heads():
    # 8 x 8192 tokens, 16 heads, bf16 D = 128: 128 sequence-heads, too many
    # for the forward's helper CTAs; every head against the oracle
    check(WORKLOADS["gdn2_mbs8_8k_h16_d128_bf16"])


@pytest.mark.parametrize("dtype,D,flags", [("bf16", 64, 0), ("f32", 64, 0), ("f32", 128, 0), ("bf16", 128, 0),
                                           ("bf16", 128, K.KDA_FLAG_FORCE_SIMT)])
def test_ragged_lengths_states_and_parameters(dtype, D, flags):
    # partial chunks, an empty sequence, single tokens, checkpoint-segment
    # crossings, nonzero A_log / dt_bias, scale 1/sqrt(D), initial states and
    # final-state gradients (bf16 D = 128: 24 sequence-heads, so the
    # tensor-core forward runs with helper CTAs; forced: the CUDA-core forward)
    lengths = (1, 15, 0, 17, 100, 1029, 2049, 3)
    w = Workload(f"gdn2_ragged_d{D}_{dtype}", lengths, 3, D, dtype, seed=7400 + D, param_std=0.5,
                 scale=D ** -0.5, gates="channel")
    check(w, states=True, flags=flags)


def test_tensor_core_forward_long_memory_and_saturated_gates():
    # bf16 D = 128 (tensor-core forward): a long-memory decay gate
    # (N(-6, 1)) over sequences that cross checkpoint segments, and a second
    # problem whose raw gates sit far in both tails (erase / write near 0 and 1)
    w = Workload("gdn2_tc_long", (2100, 700, 5), 4, 128, "bf16", seed=7450, gate_mean=-6.0,
                 param_std=0.3, gates="channel")
    check(w)
    inp = to_dev(make_inputs(w, device="cpu"))
    inp["erase"] = inp["erase"] * 6.0
    inp["write"] = inp["write"] * 6.0
    gpu = run_gpu(inp, w.scale)
    compare(gpu, run_oracle(inp, w.scale), TOL[torch.bfloat16], names=NAMES)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_long_memory_gate(dtype):
    # raw gate N(-6, 1): decays near 1, so state memory spans hundreds of
    # tokens and crosses every chunk boundary
    w = Workload(f"gdn2_long_{dtype}", (700, 1300), 4, 64, dtype, seed=7500, gate_mean=-6.0,
                 gates="channel")
    check(w)


def test_equal_gates_match_the_kda_kernels():
    # erase = write = beta on every channel is KDA: the GDN-2 kernels agree
    # with the KDA CUDA-core kernels on the same problem (fp32 bar)
    w = Workload("gdn2_vs_kda", (300, 511), 3, 64, "f32", seed=7600, param_std=0.3)
    inp = to_dev(make_inputs(w, device="cpu"))
    b3 = inp["beta"][:, :, None].expand(-1, -1, 64).contiguous()
    args = [inp[n] for n in ["q", "k", "v", "g"]]
    o, ctx = K.gdn2_fwd(*args, b3, b3, inp["A_log"], inp["dt_bias"], inp["cu_seqlens"])
    r = K.gdn2_bwd(*args, b3, b3, inp["A_log"], inp["dt_bias"], inp["cu_seqlens"], inp["dO"], ctx)
    ok, kctx = K.kda_fwd(*args, inp["beta"], inp["A_log"], inp["dt_bias"], inp["cu_seqlens"],
                         flags=K.KDA_FLAG_FORCE_SIMT)
    rk = K.kda_bwd(*args, inp["beta"], inp["A_log"], inp["dt_bias"], inp["cu_seqlens"], inp["dO"],
                   kctx, flags=K.KDA_FLAG_FORCE_SIMT)
    torch.cuda.synchronize()
    r["o"], rk["o"] = o, ok
    r["dbeta"] = r["derase"].sum(-1) + r["dwrite"].sum(-1)
    ref = {n: rk[n].double().cpu().numpy() for n in ["o", "dq", "dk", "dv", "dg", "dbeta", "dA_log",
                                                       "ddt_bias"]}
    compare(r, ref, 1e-4, names=list(ref))


def test_autograd_function_matches_direct_calls():
    w = Workload("gdn2_autograd", (200, 77), 2, 64, "bf16", seed=7700, param_std=0.3,
                 gates="channel")
    inp = to_dev(make_inputs(w, device="cpu"))
    leaves = {n: inp[n].clone().requires_grad_(True)
              for n in ["q", "k", "v", "g", "erase", "write", "A_log", "dt_bias"]}
    o = K.gdn2(*[leaves[n] for n in ["q", "k", "v", "g", "erase", "write", "A_log", "dt_bias"]],
               inp["cu_seqlens"])
    o.backward(inp["dO"])
    args = [inp[n] for n in ARGS]
    o2, ctx = K.gdn2_fwd(*args)
    r = K.gdn2_bwd(*args, inp["dO"], ctx)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    pairs = dict(q="dq", k="dk", v="dv", g="dg", erase="derase", write="dwrite", A_log="dA_log",
                 dt_bias="ddt_bias")
    for leaf, gname in pairs.items():
        assert torch.equal(leaves[leaf].grad, r[gname]), gname


def test_inference_forward_matches_the_training_forward():
    # without checkpoints (KDA_FLAG_NO_CHECKPOINTS, no ctx kept) the forward
    # writes the same o, bit for bit, and the same final states
    w = Workload("gdn2_infer", (1500, 33, 1), 3, 128, "bf16", seed=7800, param_std=0.3,
                 gates="channel")
    inp = to_dev(make_inputs(w, device="cpu"))
    args = [inp[n] for n in ARGS]
    o, ctx, hT = K.gdn2_fwd(*args, final_state=True)
    o2, ctx2, hT2 = K.gdn2_fwd(*args, save_ctx=False, final_state=True)
    torch.cuda.synchronize()
    assert ctx2 is None
    assert torch.equal(o, o2) and torch.equal(hT, hT2)
