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
