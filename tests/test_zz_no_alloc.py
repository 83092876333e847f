"""kda_bwd_noalloc, the backward for callers that cannot allocate device
memory where they run it, checked through the C ABI against kda_bwd (the
entry point with a caller workspace) on two calls in a row.

This file is named so that pytest collects it last. It must pass both on its
own in a fresh process (the first call then sets up the library's fixed
scratch array on this device) and after the other tests."""
import pytest
import torch

from recompute_kda_chunkwise_gb300 import Workload, make_inputs
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import TOL, compare, to_dev

pytestmark = pytest.mark.gpu

NAMES = ["dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"]


def _two_calls_match(w: Workload, flags: int = 0):
    inp = to_dev(make_inputs(w))
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
            inp["cu_seqlens"])
    o, ctx = K.kda_fwd(*args, flags=flags)
    ref = K.kda_bwd(*args, inp["dO"], ctx, flags=flags)
    torch.cuda.synchronize()
    ref_np = {n: ref[n].double().cpu().numpy() for n in NAMES}
    tol = TOL[inp["q"].dtype]
    for _ in range(2):
        got = K.kda_bwd_noalloc(*args, inp["dO"], ctx)
        torch.cuda.synchronize()
        assert K.noalloc_device_status() == 0
        compare(got, ref_np, tol, names=NAMES)
        # the same kernels run in both entry points: the results agree bit for bit
        for n in NAMES:
            assert torch.equal(got[n], ref[n]), n


@pytest.mark.parametrize("D,dtype", [(64, "bf16"), (128, "bf16"), (64, "f32")])
def test_noalloc_backward_matches_workspace_backward_twice(D, dtype):
    # 15 sequence-heads: on the tensor-core family kda_bwd runs with helper
    # CTAs (split mode) here, while the no-allocation backward runs inline
    w = Workload(f"noalloc_d{D}_{dtype}", (1, 700, 0, 2100, 33), 3, D, dtype, seed=7800 + D,
                 param_std=0.3)
    _two_calls_match(w)


def test_noalloc_backward_loops_over_more_items_than_its_ctas():
    # 4 x 1100 tokens x 16 heads = 64 sequence-heads at D = 128: the fixed
    # buffer holds about 31 CTAs' segment states, so each CTA walks several
    # items through the same scratch slot (kda_bwd itself runs in split mode)
    w = Workload("noalloc_many_items", (1100, 1100, 1100, 1100), 16, 128, "bf16", seed=7850,
                 param_std=0.3)
    _two_calls_match(w)


def test_noalloc_rejects_problems_beyond_its_buffer():
    # 20 million sequence-heads of gate-parameter partials cannot fit in the
    # fixed buffer: the call must fail on the host with a clear message
    dev = torch.device("cuda")
    cu = torch.zeros(2, dtype=torch.int32, device=dev)
    p = K.make_problem(0, 1, 1, 128, torch.bfloat16, cu)
    p.num_seqs = 200000
    p.num_heads = 100
    import ctypes
    lib = K.load_library()
    al = ctypes.c_void_p(1 << 20)
    # (p, q, k, v, g, beta, A_log, dt_bias, dO, dhT, ctx, dq, dk, dv, dg, dbeta, dA_log,
    #  ddt_bias, dh0, stream)
    st = lib.kda_bwd_noalloc(ctypes.byref(p), *([al] * 8), None, al, *([al] * 7), None, None)
    assert st == 3  # KDA_ERR_WORKSPACE
    assert b"fixed buffer" in lib.kda_last_error_message()
