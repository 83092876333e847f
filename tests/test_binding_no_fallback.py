"""The Python binding has no CPU path: CPU tensors, mixed dtypes and a
missing library are refused with an error instead of being computed some
other way (CPU only; no kernel runs)."""
import pytest
import torch

from recompute_kda_chunkwise_gb300 import WORKLOADS, make_inputs
from recompute_kda_chunkwise_gb300 import kda as K


def _cpu_inputs(gates="scalar"):
    name = "gdn2_b10_t512_h12_d64_f32" if gates == "channel" else "tiny_t256_h2_d64_bf16"
    return make_inputs(WORKLOADS[name], device="cpu")


def test_kda_refuses_cpu_tensors():
    inp = _cpu_inputs()
    args = [inp[n] for n in ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "cu_seqlens"]]
    with pytest.raises(ValueError, match="CUDA"):
        K.kda_fwd(*args)
    with pytest.raises(ValueError, match="CUDA"):
        K.kda_bwd(*args, inp["dO"], None)
    with pytest.raises(ValueError, match="CUDA"):
        K.kda_bwd_noalloc(*args, inp["dO"], None)


def test_kda_autograd_checks_its_chunk_size_and_refuses_cpu_tensors():
    inp = _cpu_inputs()
    args = [inp[n] for n in ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "cu_seqlens"]]
    with pytest.raises(ValueError, match="chunk_size"):
        K.kda(*args, chunk_size=32)
    for c in (16, 64):
        with pytest.raises(ValueError, match="CUDA"):
            K.kda(*args, chunk_size=c)


def test_gdn2_refuses_cpu_tensors():
    inp = _cpu_inputs("channel")
    args = [inp[n] for n in ["q", "k", "v", "g", "erase", "write", "A_log", "dt_bias", "cu_seqlens"]]
    with pytest.raises(ValueError, match="CUDA"):
        K.gdn2_fwd(*args)
    with pytest.raises(ValueError, match="CUDA"):
        K.gdn2_bwd(*args, inp["dO"], None)


def test_missing_library_raises(tmp_path):
    # load_library caches the first library it loads: ask for a path that
    # does not exist with the cache cleared, then restore the cache
    saved = K._lib
    K._lib = None
    try:
        with pytest.raises(RuntimeError, match="not built"):
            K.load_library(str(tmp_path / "absent.so"))
    finally:
        K._lib = saved


def test_binding_checks_shapes_and_buffers_before_any_call():
    # the C ABI takes bare pointers, so the binding checks every shape the
    # kernels index by (CPU tensors here: the checks themselves run no kernel)
    S, H, D = 40, 3, 16
    q = torch.zeros(S, H, D)
    ok = torch.zeros(S, H, D)
    K._check_shapes(q, (("k", ok),), torch.zeros(S, H), (torch.zeros(H), torch.zeros(H, D)))
    with pytest.raises(ValueError, match="k must have"):
        K._check_shapes(q, (("k", torch.zeros(S - 1, H, D)),))
    with pytest.raises(ValueError, match="beta"):
        K._check_shapes(q, (), torch.zeros(S, H, D))
    with pytest.raises(ValueError, match="A_log"):
        K._check_shapes(q, (), None, (torch.zeros(H), torch.zeros(H)))
    with pytest.raises(ValueError, match="out"):
        K._check_like(torch.zeros(S, H, D, dtype=torch.bfloat16), q, "out")
    with pytest.raises(ValueError, match="dq"):
        K._check_like(torch.zeros(S, H, D + 1), q, "dq")
    with pytest.raises(ValueError, match="required"):
        K._check_buffer(None, 16, q, "ctx")
    with pytest.raises(ValueError, match="CUDA buffer"):
        K._check_buffer(torch.zeros(64, dtype=torch.uint8), 16, q, "workspace")


def test_backward_ctx_size_excludes_the_forward_hand_off():
    # the backward reads the header, the cu_seqlens copy and the checkpoints;
    # a tensor-core problem with spare SMs also sizes ctx for the forward's
    # helper hand-off, which the backward does not need
    tc = K.make_problem(131072, 1, 96, 128, torch.bfloat16)
    simt = K.make_problem(131072, 1, 96, 128, torch.bfloat16, flags=K.KDA_FLAG_FORCE_SIMT)
    assert K._bwd_ctx_bytes(tc) == K.ctx_bytes(simt) < K.ctx_bytes(tc)
    assert tc.flags == 0  # the query does not change the caller's problem
    inference = K.make_problem(131072, 1, 96, 128, torch.bfloat16, flags=K.KDA_FLAG_NO_CHECKPOINTS)
    assert K.ctx_bytes(inference) < K._bwd_ctx_bytes(tc)
