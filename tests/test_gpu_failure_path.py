"""Device-side failure path, exercised without faulting the GPU: with
KDA_FLAG_TEST_TIMEOUT the tensor-core forward skips its first tile load, its
bounded wait runs out, the kernel records KDA_ERR_TIMEOUT in ctx and returns.
The host reads the status, and the same process then runs a normal forward
and backward that still match the oracle."""
import pytest
import torch

from recompute_kda_chunkwise_gb300 import Workload, make_inputs
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import TOL, compare, oracle_for, run_gpu, to_dev

pytestmark = pytest.mark.gpu

KDA_ERR_TIMEOUT = 5


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    w = Workload("failure_path", (200, 77), 2, 128, "bf16", seed=8100)
    inp = to_dev(make_inputs(w))
    args = (inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
            inp["cu_seqlens"])
    _, ctx = K.kda_fwd(*args, flags=K.KDA_FLAG_TEST_TIMEOUT)
    torch.cuda.synchronize()
    assert K.query_device_status(ctx) == KDA_ERR_TIMEOUT
    # a clean call afterwards resets the status and computes correct results
    gpu, ctx2 = run_gpu(inp)
    assert K.query_device_status(ctx2) == 0
    compare(gpu, oracle_for(inp), TOL[torch.bfloat16])
