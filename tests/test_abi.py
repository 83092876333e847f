"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function declared in include/kda.h, validates arguments and sizes
buffers without touching the device."""
import ctypes
import os
import re

import pytest
import torch

from recompute_kda_chunkwise_gb300 import build as kbuild
from recompute_kda_chunkwise_gb300 import kda as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(kda_\w+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "kda_fwd" in names and "kda_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_problem_struct_layout_matches_header():
    assert ctypes.sizeof(K.KdaProblem) == 48
    assert K.KdaProblem.cu_seqlens.offset == 40


def test_size_queries(lib):
    p = K.make_problem(131072, 1, 96, 128, torch.bfloat16)
    ckpts = 131072 // 1024 + 1
    # 256-byte header (status word), the checked copy of cu_seqlens (N + 1
    # int32 rounded up to 256 bytes), then the fp32 checkpoints
    states = 256 + 256 + ckpts * 96 * 128 * 128 * 4
    # tensor-core family with fewer items than the 152-CTA grid: the forward's
    # hand-off area (5 counters per item, 4 slots of 98816 bytes) follows
    handoff = (96 * 5 * 4 + 255) // 256 * 256 + 96 * 4 * 98816
    assert K.ctx_bytes(p) == states + handoff
    simt = K.make_problem(131072, 1, 96, 128, torch.bfloat16, flags=K.KDA_FLAG_FORCE_SIMT)
    assert K.ctx_bytes(simt) == states
    many = K.make_problem(131072, 2, 96, 128, torch.bfloat16)  # 192 items: no helpers
    assert K.ctx_bytes(many) == 256 + 256 + (131072 // 1024 + 2) * 96 * 128 * 128 * 4
    assert K.workspace_bytes(p) > 256 + 96 * 129 * 4
    assert K.kernel_family(p) in (0, 1)
    bad = K.make_problem(16, 1, 2, 96, torch.bfloat16)
    assert K.ctx_bytes(bad) == 0 and K.workspace_bytes(bad) == 0 and K.kernel_family(bad) == -1
    assert b"head_dim" in lib.kda_last_error_message()


def test_invalid_arguments_are_rejected_on_host(lib):
    cu = torch.tensor([0, 16], dtype=torch.int32)  # host tensor: never dereferenced
    p = K.make_problem(16, 1, 2, 64, torch.bfloat16, cu)
    nul = ctypes.c_void_p(0)
    # kda_fwd(p, q, k, v, g, beta, A_log, dt_bias, h0, o, hT, ctx, stream)
    st = lib.kda_fwd(ctypes.byref(p), *([nul] * 12))
    assert st == 1  # KDA_ERR_INVALID_ARG
    assert b"NULL" in lib.kda_last_error_message()
    mis = ctypes.c_void_p(0x1008)  # not 16-byte aligned
    al = ctypes.c_void_p(0x1000)
    st = lib.kda_fwd(ctypes.byref(p), mis, *([al] * 6), nul, al, nul, nul, nul)
    assert st == 1 and b"aligned" in lib.kda_last_error_message()
    st = lib.kda_fwd(ctypes.byref(p), *([al] * 7), mis, al, nul, nul, nul)  # misaligned h0
    assert st == 1 and b"h0" in lib.kda_last_error_message()
    st = lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, mis, nul, nul)  # misaligned hT
    assert st == 1 and b"hT" in lib.kda_last_error_message()
    p.gate_lower_bound = -8.0
    st = lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, nul, nul, nul)
    assert st == 2  # KDA_ERR_UNSUPPORTED
    p.gate_lower_bound = -5.0
    p.num_seqs = 0
    # kda_bwd(p, q, k, v, g, beta, A_log, dt_bias, dO, dhT, ctx, dq, dk, dv, dg, dbeta,
    #         dA_log, ddt_bias, dh0, workspace, stream)
    assert lib.kda_bwd(ctypes.byref(p), *([al] * 19), nul) == 1
    p.num_seqs = 1
    st = lib.kda_bwd(ctypes.byref(p), *([al] * 8), mis, *([al] * 10), nul)  # misaligned dhT
    assert st == 1 and b"dhT" in lib.kda_last_error_message()
    p.dtype = 7
    assert lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, nul, nul, nul) == 2
    p.dtype = 0
    p.flags = 32  # no such flag
    assert lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, nul, nul, nul) == 1
    assert b"unknown flags" in lib.kda_last_error_message()
    # 16-token chunks: tensor-core KDA problems only, refused before any launch
    # (this problem has head_dim 64; then bf16 D = 128 forced onto the CUDA cores)
    p.flags = K.KDA_FLAG_CHUNK16
    assert lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, nul, al, nul) == 2
    assert b"CHUNK16" in lib.kda_last_error_message()
    p128 = K.make_problem(16, 1, 2, 128, torch.bfloat16, cu, flags=K.KDA_FLAG_CHUNK16 | K.KDA_FLAG_FORCE_SIMT)
    assert lib.kda_fwd(ctypes.byref(p128), *([al] * 7), nul, al, nul, al, nul) == 2
    p.flags = K.KDA_FLAG_FORCE_SIMT | K.KDA_FLAG_TEST_TIMEOUT  # both known: sizes still answer
    assert lib.kda_ctx_bytes(ctypes.byref(p)) > 0
    # inference: no checkpoints, so ctx shrinks to the status header and the
    # checked copy of cu_seqlens; the backward refuses a problem flagged that way
    p.flags = K.KDA_FLAG_NO_CHECKPOINTS
    assert lib.kda_ctx_bytes(ctypes.byref(p)) == 256 + 256
    assert lib.kda_bwd(ctypes.byref(p), *([al] * 8), nul, *([al] * 8), nul, al, nul) == 1
    assert b"NO_CHECKPOINTS" in lib.kda_last_error_message()


def test_gdn2_entry_points_and_flag_on_host(lib):
    cu = torch.tensor([0, 16], dtype=torch.int32)  # host tensor: never dereferenced
    nul = ctypes.c_void_p(0)
    al = ctypes.c_void_p(0x1000)
    # bf16 D = 128 GDN-2 problems: tensor-core forward (ctx sized like KDA's,
    # with the helper hand-off area), CUDA-core backward (workspace sized
    # like the forced CUDA-core KDA backward's)
    g = K.make_problem(131072, 1, 96, 128, torch.bfloat16, flags=K.KDA_FLAG_CHANNEL_GATES)
    kda_tc = K.make_problem(131072, 1, 96, 128, torch.bfloat16)
    simt = K.make_problem(131072, 1, 96, 128, torch.bfloat16, flags=K.KDA_FLAG_FORCE_SIMT)
    assert K.kernel_family(g) == 2
    assert K.ctx_bytes(g) == K.ctx_bytes(kda_tc) and K.workspace_bytes(g) == K.workspace_bytes(simt)
    g64 = K.make_problem(131072, 1, 96, 64, torch.bfloat16, flags=K.KDA_FLAG_CHANNEL_GATES)
    assert K.kernel_family(g64) == 0
    p = K.make_problem(16, 1, 2, 64, torch.bfloat16, cu, flags=K.KDA_FLAG_CHANNEL_GATES)
    # the KDA entry points refuse a GDN-2 problem ...
    assert lib.kda_fwd(ctypes.byref(p), *([al] * 7), nul, al, nul, al, nul) == 1
    assert b"kda_gdn2_fwd" in lib.kda_last_error_message()
    assert lib.kda_bwd(ctypes.byref(p), *([al] * 8), nul, *([al] * 8), nul, al, nul) == 1
    assert b"kda_gdn2_bwd" in lib.kda_last_error_message()
    assert lib.kda_bwd_noalloc(ctypes.byref(p), *([al] * 8), nul, *([al] * 8), nul, nul) == 1
    # ... and the GDN-2 entry points refuse a problem without the flag
    # kda_gdn2_fwd(p, q, k, v, g, erase, write, A_log, dt_bias, h0, o, hT, ctx, stream)
    p.flags = 0
    assert lib.kda_gdn2_fwd(ctypes.byref(p), *([al] * 8), nul, al, nul, al, nul) == 1
    assert b"KDA_FLAG_CHANNEL_GATES" in lib.kda_last_error_message()
    # GDN-2 has no 16-token forward
    g128 = K.make_problem(16, 1, 2, 128, torch.bfloat16, cu,
                          flags=K.KDA_FLAG_CHANNEL_GATES | K.KDA_FLAG_CHUNK16)
    assert lib.kda_gdn2_fwd(ctypes.byref(g128), *([al] * 8), nul, al, nul, al, nul) == 2
    assert b"CHUNK16" in lib.kda_last_error_message()
    # kda_gdn2_bwd(p, q, k, v, g, erase, write, A_log, dt_bias, dO, dhT, ctx, dq, dk, dv, dg,
    #              derase, dwrite, dA_log, ddt_bias, dh0, workspace, stream)
    assert lib.kda_gdn2_bwd(ctypes.byref(p), *([al] * 9), nul, *([al] * 10), nul, al, nul) == 1
    p.flags = K.KDA_FLAG_CHANNEL_GATES
    # a missing write gate is an argument error found on the host
    assert lib.kda_gdn2_fwd(ctypes.byref(p), *([al] * 5), nul, *([al] * 2), nul, al, nul, al, nul) == 1
    assert b"write_raw" in lib.kda_last_error_message()
    assert lib.kda_gdn2_bwd(ctypes.byref(p), *([al] * 9), nul, *([al] * 6), nul, *([al] * 2), nul, al,
                            nul) == 1
    assert b"dwrite_raw" in lib.kda_last_error_message()
    assert lib.kda_gdn2_bwd(ctypes.byref(p), *([al] * 9), nul, *([al] * 5), nul, *([al] * 3), nul, al,
                            nul) == 1
    assert b"derase_raw" in lib.kda_last_error_message()


def test_status_strings(lib):
    for i, name in enumerate(K.STATUS_NAMES):
        assert lib.kda_status_string(i).decode() == name
    assert lib.kda_version() >= 200
