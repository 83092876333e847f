"""GPU parity of the forward with 16-token chunks (KDA_FLAG_CHUNK16) against
the fp64 oracle, through the C ABI: its outputs and final states, and (fed to
the default backward through the checkpoints it stores) the gradients, at the
same bars as every other bf16 test (2e-2 of the reference's RMS beyond the
output's own rounding)."""
import pytest
import torch

from recompute_kda_chunkwise_gb300 import Workload, make_inputs, make_states
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import OUT_NAMES, TOL, compare, oracle_for, to_dev
from tests.test_gpu_state import _args, _compare_state, oracle_state

pytestmark = pytest.mark.gpu


def test_chunk16_training_forward_ragged_with_states():
    # partial chunks, an empty sequence, single tokens and checkpoint-segment
    # crossings, h0 and dhT everywhere; the backward reads the 16-token
    # forward's checkpoints
    w = Workload("chunk16_ragged", (1, 15, 0, 17, 100, 1029, 2049, 3), 3, 128, "bf16", seed=8100,
                 param_std=0.5, scale=128 ** -0.5)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w))
    o, ctx, hT = K.kda_fwd(*_args(inp), scale=w.scale, flags=K.KDA_FLAG_CHUNK16, h0=st["h0"],
                           final_state=True)
    r = K.kda_bwd(*_args(inp), inp["dO"], ctx, scale=w.scale, dht=st["dht"], want_dh0=True)
    torch.cuda.synchronize()
    r["o"], r["hT"] = o, hT
    _compare_state(r, oracle_state(inp, st, scale=w.scale), TOL[torch.bfloat16])
    torch.testing.assert_close(hT[2], st["h0"][2], rtol=0, atol=0)  # the empty sequence


def test_chunk16_inference_more_items_than_ctas_and_gate_floor():
    # 180 (sequence, head) items on at most 152 CTAs: CTAs walk several items;
    # gate std 2 drives some per-token gates to the -5 floor
    w = Workload("chunk16_items", (300, 77, 512, 129, 1, 64, 200, 33, 400, 17), 18, 128, "bf16",
                 seed=8200, gate_std=2.0)
    inp = to_dev(make_inputs(w))
    o, _ = K.kda_fwd(*_args(inp), scale=w.scale, flags=K.KDA_FLAG_CHUNK16, save_ctx=False)
    o64, _ = K.kda_fwd(*_args(inp), scale=w.scale, save_ctx=False)
    torch.cuda.synchronize()
    ref = oracle_for(inp, scale=w.scale)
    compare({"o": o}, ref, TOL[torch.bfloat16], names=["o"])
    compare({"o": o64}, ref, TOL[torch.bfloat16], names=["o"])


def test_chunk16_rejects_other_problems():
    w = Workload("chunk16_f32", (40,), 2, 64, "f32", seed=8300)
    inp = to_dev(make_inputs(w))
    with pytest.raises(K.KdaError) as e:
        K.kda_fwd(*_args(inp), flags=K.KDA_FLAG_CHUNK16)
    assert e.value.status == 2  # KDA_ERR_UNSUPPORTED
    w = Workload("chunk16_simt", (40,), 2, 128, "bf16", seed=8301)
    inp = to_dev(make_inputs(w))
    with pytest.raises(K.KdaError) as e:
        K.kda_fwd(*_args(inp), flags=K.KDA_FLAG_CHUNK16 | K.KDA_FLAG_FORCE_SIMT)
    assert e.value.status == 2


def test_chunk16_through_the_autograd_wrapper():
    # kda(..., chunk_size=16) runs the 16-token forward and the default backward:
    # the same bits as the direct calls
    w = Workload("chunk16_autograd", (300, 77), 2, 128, "bf16", seed=8400, param_std=0.3)
    inp = to_dev(make_inputs(w))
    o_d, ctx = K.kda_fwd(*_args(inp), flags=K.KDA_FLAG_CHUNK16)
    direct = K.kda_bwd(*_args(inp), inp["dO"], ctx)
    leaves = {n: inp[n].clone().requires_grad_(True)
              for n in ["q", "k", "v", "g", "beta", "A_log", "dt_bias"]}
    o = K.kda(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], leaves["A_log"],
              leaves["dt_bias"], inp["cu_seqlens"], chunk_size=16)
    o.backward(inp["dO"])
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o_d)
    for n, gname in [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                     ("A_log", "dA_log"), ("dt_bias", "ddt_bias")]:
        assert torch.equal(leaves[n].grad, direct[gname]), n
