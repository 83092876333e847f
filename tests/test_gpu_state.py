"""GPU parity with an initial state h0, a final state hT and their gradients
(dhT in, dh0 out), through the C ABI, against the fp64 oracle.

Bar, per tensor (o, every input gradient, hT and dh0): max|x - ref| beyond
the output's own half-ulp rounding <= 2e-2 * RMS(ref) for bf16 inputs and
<= 1e-4 * RMS(ref) for fp32 inputs, exactly as in the stateless tests.
Elements dominated by a direct product of a state and a state gradient (the
gate gradient of a sequence's first or last token: in a one-token sequence
h0 and dhT meet in one product) stand far above their tensor's RMS, so these
cases check that the kernels carry states at better than fp16 precision
wherever a state meets a state gradient.
"""
import numpy as np
import pytest
import torch

import oracle
from recompute_kda_chunkwise_gb300 import Workload, make_inputs, make_states
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import OUT_NAMES, TOL, compare, to_dev

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
STATE_NAMES = OUT_NAMES + ["hT", "dh0"]


def _args(inp):
    return [inp[n] for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "cu_seqlens")]


def run_gpu_state(inp, st, scale=1.0, flags=0, noalloc=False):
    o, ctx, hT = K.kda_fwd(*_args(inp), scale=scale, flags=flags, h0=st["h0"], final_state=True)
    if noalloc:
        r = K.kda_bwd_noalloc(*_args(inp), inp["dO"], ctx, scale=scale, dht=st["dht"], want_dh0=True)
    else:
        r = K.kda_bwd(*_args(inp), inp["dO"], ctx, scale=scale, flags=flags, dht=st["dht"],
                      want_dh0=True)
    torch.cuda.synchronize()
    r["o"], r["hT"] = o, hT
    return r


def oracle_state(inp, st, heads=None, scale=1.0):
    cpu = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    h0, dht = st["h0"].cpu(), st["dht"].cpu()
    if heads is not None:  # heads are independent: run the sampled heads only
        idx = torch.tensor(heads)
        for n in ("q", "k", "v", "g", "dO", "beta"):
            cpu[n] = cpu[n].index_select(1, idx)
        cpu["A_log"], cpu["dt_bias"] = cpu["A_log"][idx], cpu["dt_bias"][idx]
        h0, dht = h0.index_select(1, idx), dht.index_select(1, idx)
    return oracle.kda_reference(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"], cpu["A_log"],
                                cpu["dt_bias"], cpu["cu_seqlens"], cpu["dO"], scale=scale, h0=h0,
                                dht=dht)


def _compare_state(gpu, ref, tol, heads=None):
    if heads is not None:
        idx = torch.tensor(heads, device=gpu["hT"].device)
        gpu = dict(gpu)
        gpu["hT"] = gpu["hT"].index_select(1, idx)
        gpu["dh0"] = gpu["dh0"].index_select(1, idx)
        rep = compare(gpu, ref, tol, heads=heads, names=OUT_NAMES)
        rep.update(compare(gpu, ref, tol, names=["hT", "dh0"]))
        return rep
    return compare(gpu, ref, tol, names=STATE_NAMES)


@pytest.mark.parametrize("dtype,D,flags", [("bf16", 128, 0), ("f32", 64, 0),
                                           ("bf16", 128, K.KDA_FLAG_FORCE_SIMT)])
def test_ragged_lengths_with_states(dtype, D, flags):
    # partial chunks, an empty sequence, single tokens and checkpoint-segment
    # crossings, with an initial state and a final-state gradient everywhere
    w = Workload(f"state_ragged_d{D}_{dtype}", (1, 15, 0, 17, 100, 1029, 2049, 3), 3, D, dtype,
                 seed=7700 + D, param_std=0.5, scale=D ** -0.5)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w))
    gpu = run_gpu_state(inp, st, scale=w.scale, flags=flags)
    ref = oracle_state(inp, st, scale=w.scale)
    _compare_state(gpu, ref, TOL[_DT[dtype]])
    # the empty sequence (index 2) passes its state through, and its gradient back
    torch.testing.assert_close(gpu["hT"][2], st["h0"][2], rtol=0, atol=0)
    torch.testing.assert_close(gpu["dh0"][2], st["dht"][2], rtol=0, atol=0)


def test_large_final_state_gradient():
    # dhT twenty times the in-sequence state gradient: the gradients of each
    # sequence's last tokens then stand far above the rest of their tensors
    w = Workload("state_big_dht", (1, 15, 17, 1024), 3, 128, "bf16", seed=7750, param_std=0.5,
                 scale=128 ** -0.5)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w, dht_std=1.0))
    gpu = run_gpu_state(inp, st, scale=w.scale)
    ref = oracle_state(inp, st, scale=w.scale)
    _compare_state(gpu, ref, TOL[torch.bfloat16])


def test_split_mode_launch_with_states():
    # 96 (sequence, head) items: the forward and the backward run with helper
    # CTAs (split mode); the oracle checks a sample of heads
    w = Workload("state_split_h96", (2048,), 96, 128, "bf16", seed=7800, param_std=0.3)
    inp = make_inputs(w, device="cuda")
    st = make_states(w, device="cuda")
    gpu = run_gpu_state(inp, st)
    heads = [0, 50, 95]
    ref = oracle_state(inp, st, heads=heads)
    _compare_state(gpu, ref, TOL[torch.bfloat16], heads=heads)


def test_noalloc_backward_with_states_matches_kda_bwd():
    w = Workload("state_noalloc", (700, 0, 300), 3, 128, "bf16", seed=7900, param_std=0.3)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w))
    a = run_gpu_state(inp, st)
    b = run_gpu_state(inp, st, noalloc=True)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dh0"):
        torch.testing.assert_close(a[n], b[n], rtol=0, atol=0, msg=n)


def test_sequence_split_through_its_state_matches_the_whole():
    # running tokens [0, T) equals running [0, T1) and then [T1, T) from the
    # first part's final state (and, backwards, feeding the second part's dh0
    # to the first part as its dhT): checked against the oracle on the whole
    w = Workload("state_chain", (1500,), 4, 128, "bf16", seed=8000, param_std=0.3)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w))
    T1 = 600

    def part(a, b):
        p = {k: (v[a:b] if k in ("q", "k", "v", "g", "beta", "dO") else v) for k, v in inp.items()}
        p["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32, device="cuda")
        return p

    p1, p2 = part(0, T1), part(T1, 1500)
    o1, ctx1, h_mid = K.kda_fwd(*_args(p1), h0=st["h0"], final_state=True)
    o2, ctx2, hT = K.kda_fwd(*_args(p2), h0=h_mid, final_state=True)
    r2 = K.kda_bwd(*_args(p2), p2["dO"], ctx2, dht=st["dht"], want_dh0=True)
    r1 = K.kda_bwd(*_args(p1), p1["dO"], ctx1, dht=r2["dh0"], want_dh0=True)
    torch.cuda.synchronize()
    gpu = {"o": torch.cat([o1, o2]), "hT": hT, "dh0": r1["dh0"],
           "dA_log": r1["dA_log"] + r2["dA_log"], "ddt_bias": r1["ddt_bias"] + r2["ddt_bias"]}
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        gpu[n] = torch.cat([r1[n], r2[n]])
    ref = oracle_state(inp, st)
    compare(gpu, ref, TOL[torch.bfloat16], names=STATE_NAMES)


def test_autograd_with_initial_and_final_state():
    w = Workload("state_autograd", (300, 45), 2, 128, "bf16", seed=8100, param_std=0.3)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w))
    leaves = {n: inp[n].clone().requires_grad_(True)
              for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias")}
    h0 = st["h0"].clone().requires_grad_(True)
    o, hT = K.kda(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], leaves["A_log"],
                  leaves["dt_bias"], inp["cu_seqlens"], initial_state=h0, output_final_state=True)
    ((o.float() * inp["dO"].float()).sum() + (hT * st["dht"]).sum()).backward()
    direct = run_gpu_state(inp, st)
    torch.testing.assert_close(o, direct["o"], rtol=0, atol=0)
    torch.testing.assert_close(hT, direct["hT"], rtol=0, atol=0)
    torch.testing.assert_close(h0.grad, direct["dh0"], rtol=0, atol=0)
    for n, g in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                 ("A_log", "dA_log"), ("dt_bias", "ddt_bias")):
        torch.testing.assert_close(leaves[n].grad, direct[g], rtol=0, atol=0, msg=n)


def test_zero_states_match_the_stateless_call():
    w = Workload("state_zero", (257, 64), 2, 128, "bf16", seed=8200)
    inp = to_dev(make_inputs(w))
    z = {"h0": torch.zeros(2, 2, 128, 128, device="cuda"), "dht": torch.zeros(2, 2, 128, 128, device="cuda")}
    a = run_gpu_state(inp, z)
    o, ctx = K.kda_fwd(*_args(inp))
    b = K.kda_bwd(*_args(inp), inp["dO"], ctx)
    torch.cuda.synchronize()
    torch.testing.assert_close(a["o"], o, rtol=0, atol=0)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"):
        torch.testing.assert_close(a[n], b[n], rtol=0, atol=0, msg=n)
    assert np.isfinite(a["hT"].cpu().numpy()).all()
