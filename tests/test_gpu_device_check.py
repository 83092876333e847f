"""Device-side check of cu_seqlens: a malformed boundary array is caught on
the GPU before any kernel loads through it, reported as
KDA_ERR_DEVICE_CHECK in the call's status word, and leaves the context
usable. The malformed arrays keep every entry inside [0, S], so even a
missed check could not reach memory outside the allocated tensors."""
import pytest
import torch

from recompute_kda_chunkwise_gb300 import Workload, make_inputs
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import TOL, compare, oracle_for, run_gpu, to_dev

pytestmark = pytest.mark.gpu

DEVICE_CHECK = 6  # KDA_ERR_DEVICE_CHECK

# lengths (300, 200, 500) -> cu = [0, 300, 500, 1000]; S = 1000
BAD = {
    "non_monotone": [0, 300, 200, 1000],
    "last_below_S": [0, 300, 500, 900],
    "first_not_zero": [10, 300, 500, 1000],
}


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f32"), (128, "f32")])
@pytest.mark.parametrize("case", sorted(BAD))
def test_malformed_cu_seqlens_is_reported_and_context_stays_usable(case, D, dtype):
    w = Workload(f"devcheck_{case}_d{D}_{dtype}", (300, 200, 500), 2, D, dtype, seed=7900 + D)
    inp = to_dev(make_inputs(w))
    args = lambda cu: (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                       inp["dt_bias"], cu)
    good_cu = inp["cu_seqlens"]
    bad_cu = torch.tensor(BAD[case], dtype=torch.int32, device=good_cu.device)
    # forward with the malformed boundaries: reported in ctx
    o, ctx = K.kda_fwd(*args(bad_cu))
    torch.cuda.synchronize()
    assert K.query_device_status(ctx) == DEVICE_CHECK
    # backward with the malformed boundaries (ctx of a good forward): reported in the workspace
    _, good_ctx = K.kda_fwd(*args(good_cu))
    p = K.make_problem(w.total_tokens, w.num_seqs, w.H, w.D, inp["q"].dtype, bad_cu)
    ws = torch.empty(K.workspace_bytes(p), dtype=torch.uint8, device=good_cu.device)
    K.kda_bwd(*args(bad_cu), inp["dO"], good_ctx, workspace=ws)
    torch.cuda.synchronize()
    assert K.query_device_status(ws) == DEVICE_CHECK
    # the no-allocation backward reports through its own status query
    K.kda_bwd_noalloc(*args(bad_cu), inp["dO"], good_ctx)
    assert K.noalloc_device_status() == DEVICE_CHECK
    # a clean call afterwards, in the same process, matches the oracle
    gpu, ctx2 = run_gpu(inp)
    assert K.query_device_status(ctx2) == 0
    compare(gpu, oracle_for(inp), TOL[inp["q"].dtype])
    K.kda_bwd_noalloc(*args(good_cu), inp["dO"], ctx2)
    assert K.noalloc_device_status() == 0
