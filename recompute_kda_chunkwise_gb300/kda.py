"""Thin Python binding of the KDA C ABI (include/kda.h).

Argument marshalling only: every step of the forward and backward runs in
the CUDA library ``_build/libkda_gb300.so``. PyTorch supplies device memory
and the current stream. There is no CPU fallback: if the library is missing
or a call fails, a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda_gb300.so")

KDA_DTYPE_BF16 = 0
KDA_DTYPE_F32 = 1
_DTYPE_CODE = {torch.bfloat16: KDA_DTYPE_BF16, torch.float32: KDA_DTYPE_F32}
STATUS_NAMES = ["KDA_OK", "KDA_ERR_INVALID_ARG", "KDA_ERR_UNSUPPORTED", "KDA_ERR_WORKSPACE",
                "KDA_ERR_CUDA", "KDA_ERR_TIMEOUT", "KDA_ERR_DEVICE_CHECK"]


class KdaProblem(ctypes.Structure):
    """Mirror of ``kda_problem`` in include/kda.h."""
    _fields_ = [("total_tokens", ctypes.c_int64), ("num_seqs", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("gate_lower_bound", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("flags", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name}: {detail}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"KDA CUDA library not built: {path} is missing "
                                   "(run recompute_kda_chunkwise_gb300.build.build())")
            lib = ctypes.CDLL(path)
            vp, P = ctypes.c_void_p, ctypes.POINTER(KdaProblem)
            lib.kda_ctx_bytes.restype = ctypes.c_size_t
            lib.kda_ctx_bytes.argtypes = [P]
            lib.kda_bwd_workspace_bytes.restype = ctypes.c_size_t
            lib.kda_bwd_workspace_bytes.argtypes = [P]
            lib.kda_fwd.restype = ctypes.c_int
            lib.kda_fwd.argtypes = [P] + [vp] * 12
            lib.kda_bwd.restype = ctypes.c_int
            lib.kda_bwd.argtypes = [P] + [vp] * 20
            lib.kda_bwd_noalloc.restype = ctypes.c_int
            lib.kda_bwd_noalloc.argtypes = [P] + [vp] * 19
            lib.kda_gdn2_fwd.restype = ctypes.c_int
            lib.kda_gdn2_fwd.argtypes = [P] + [vp] * 13
            lib.kda_gdn2_bwd.restype = ctypes.c_int
            lib.kda_gdn2_bwd.argtypes = [P] + [vp] * 22
            lib.kda_query_device_status.restype = ctypes.c_int
            lib.kda_query_device_status.argtypes = [vp, vp]
            lib.kda_noalloc_device_status.restype = ctypes.c_int
            lib.kda_noalloc_device_status.argtypes = [vp]
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.kda_state_prefix.restype = ctypes.c_int
            lib.kda_state_prefix.argtypes = [i32, i32, i32, i32, i32, i64, i64, vp, vp, vp, vp, vp, vp]
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [ctypes.c_int]
            lib.kda_last_error_message.restype = ctypes.c_char_p
            lib.kda_last_error_message.argtypes = []
            lib.kda_kernel_family.restype = ctypes.c_int
            lib.kda_kernel_family.argtypes = [P]
            lib.kda_version.restype = ctypes.c_int
            lib.kda_version.argtypes = []
            _lib = lib
    return _lib


def _check(status: int, where: str):
    if status != 0:
        msg = load_library().kda_last_error_message().decode(errors="replace")
        raise KdaError(status, where, msg)


KDA_FLAG_FORCE_SIMT = 1
KDA_FLAG_TEST_TIMEOUT = 2  # test only: the forward's bounded wait runs out (see include/kda.h)
KDA_FLAG_NO_CHECKPOINTS = 4  # inference: ctx holds no checkpoints (scratch for the forward only)
KDA_FLAG_CHANNEL_GATES = 8  # GDN-2 problem (channel-wise erase / write gates)
KDA_FLAG_CHUNK16 = 16  # kda_fwd with 16-token chunks (tensor-core KDA problems; see include/kda.h)


def make_problem(total_tokens: int, num_seqs: int, num_heads: int, head_dim: int, dtype,
                 cu_seqlens=None, scale: float = 1.0, lower_bound: float = -5.0,
                 eps: float = 1e-6, flags: int = 0) -> KdaProblem:
    code = _DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    ptr = 0 if cu_seqlens is None else cu_seqlens.data_ptr()
    return KdaProblem(int(total_tokens), int(num_seqs), int(num_heads), int(head_dim), code,
                      float(scale), float(lower_bound), float(eps), int(flags), ptr)


def ctx_bytes(p: KdaProblem) -> int:
    return int(load_library().kda_ctx_bytes(ctypes.byref(p)))


def workspace_bytes(p: KdaProblem) -> int:
    return int(load_library().kda_bwd_workspace_bytes(ctypes.byref(p)))


def kernel_family(p: KdaProblem) -> int:
    return int(load_library().kda_kernel_family(ctypes.byref(p)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _problem_from(q, beta, cu_seqlens, scale, lower_bound, eps, flags=0):
    if q.dim() != 3:
        raise ValueError("q must be [S, H, D]")
    S, H, D = q.shape
    if q.dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != q.device:
        raise ValueError("cu_seqlens must be int32 on the same device as q")
    return make_problem(S, cu_seqlens.numel() - 1, H, D, q.dtype, cu_seqlens, scale, lower_bound, eps,
                        flags)


def _check_tensors(q, *others, params=()):
    for t in (q,) + tuple(others):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("all activations must be contiguous CUDA tensors of one dtype and device")
    for t in params:
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32 or t.device != q.device:
            raise ValueError("A_log and dt_bias must be contiguous float32 CUDA tensors")


def _check_shapes(q, same=(), beta=None, params=()):
    """The kernels index every tensor by q's [S, H, D]: the activations in
    ``same`` (name, tensor) must have that shape, beta [S, H], and the gate
    parameters (A_log, dt_bias) [H] and [H, D]."""
    if q.dim() != 3:
        raise ValueError("q must be [S, H, D]")
    S, H, D = q.shape
    for name, t in same:
        if tuple(t.shape) != (S, H, D):
            raise ValueError(f"{name} must have q's shape {(S, H, D)} (got {tuple(t.shape)})")
    if beta is not None and tuple(beta.shape) != (S, H):
        raise ValueError(f"beta must be [S, H] = {(S, H)} (got {tuple(beta.shape)})")
    if params:
        A_log, dt_bias = params
        if tuple(A_log.shape) != (H,) or tuple(dt_bias.shape) != (H, D):
            raise ValueError(f"A_log must be [H] = {(H,)} and dt_bias [H, D] = {(H, D)}")


def _check_like(t, ref, name):
    """A caller-supplied output: the shape, dtype and device of ``ref``, contiguous."""
    if (tuple(t.shape) != tuple(ref.shape) or t.dtype != ref.dtype or t.device != ref.device
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {ref.dtype} tensor of shape {tuple(ref.shape)} "
                         f"on {ref.device}")


def _check_buffer(t, nbytes, q, name):
    """A ctx or workspace buffer: contiguous, on q's device, at least nbytes."""
    if t is None:
        raise ValueError(f"{name} is required")
    if (not t.is_cuda or t.device != q.device or not t.is_contiguous()
            or t.numel() * t.element_size() < nbytes):
        raise ValueError(f"{name} must be a contiguous CUDA buffer on {q.device} of at least {nbytes} bytes")


def _bwd_ctx_bytes(p) -> int:
    """Bytes of ctx the backward reads: the status header, the checked
    cu_seqlens copy and the checkpoints (the CUDA-core family's ctx, which
    has no forward hand-off area after them)."""
    simt = KdaProblem.from_buffer_copy(p)
    simt.flags |= KDA_FLAG_FORCE_SIMT
    return ctx_bytes(simt)


def _check_state(t, q, cu_seqlens, name):
    """States are fp32 [N, H, D, D] (rows: key channel), contiguous, on q's device."""
    if t is None:
        return
    S, H, D = q.shape
    want = (cu_seqlens.numel() - 1, H, D, D)
    if (not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32 or t.device != q.device
            or tuple(t.shape) != want):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {want}")


def _state_like(q, cu_seqlens):
    S, H, D = q.shape
    return torch.empty((cu_seqlens.numel() - 1, H, D, D), dtype=torch.float32, device=q.device)


def kda_fwd(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, *, scale: float = 1.0,
            lower_bound: float = -5.0, eps: float = 1e-6, save_ctx: bool = True, out=None,
            ctx=None, flags: int = 0, h0=None, final_state=False):
    """Forward. Returns (o, ctx); ctx is None when save_ctx is False. ``out``
    and ``ctx`` may be preallocated (ctx of at least ctx_bytes(problem)).
    Without save_ctx the forward runs as inference (KDA_FLAG_NO_CHECKPOINTS):
    no checkpoints are written, and a small scratch ctx (``ctx`` when given)
    carries only the status word and the helper hand-off area.
    h0: initial states [N, H, D, D] fp32 (zero when None). With final_state
    True (or a preallocated [N, H, D, D] fp32 tensor) the final states are
    returned too: (o, ctx, hT)."""
    _check_tensors(q, k, v, g, beta, params=(A_log, dt_bias))
    _check_shapes(q, (("k", k), ("v", v), ("g", g)), beta, (A_log, dt_bias))
    _check_state(h0, q, cu_seqlens, "h0")
    if not save_ctx:
        flags |= KDA_FLAG_NO_CHECKPOINTS
    p = _problem_from(q, beta, cu_seqlens, scale, lower_bound, eps, flags)
    hT = None
    if final_state is not False and final_state is not None:
        hT = _state_like(q, cu_seqlens) if final_state is True else final_state
        _check_state(hT, q, cu_seqlens, "final_state")
    if out is not None:
        _check_like(out, q, "out")
    o = torch.empty_like(q) if out is None else out
    if ctx is None:
        ctx = torch.empty(ctx_bytes(p), dtype=torch.uint8, device=q.device)
    else:
        _check_buffer(ctx, ctx_bytes(p), q, "ctx")
    st = load_library().kda_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o), _ptr(hT), _ptr(ctx),
                                _stream_handle(q.device))
    _check(st, "kda_fwd")
    if not save_ctx:
        ctx = None
    return (o, ctx) if hT is None else (o, ctx, hT)


def _grad_outs(outs, q, k, v, g, beta, A_log, dt_bias, cu_seqlens, want_dh0):
    like = dict(dq=q, dk=k, dv=v, dg=g, dbeta=beta, dA_log=A_log, ddt_bias=dt_bias)
    if outs is None:
        outs = {n: torch.empty_like(t) for n, t in like.items()}
    for n, t in like.items():
        if n not in outs:
            raise ValueError(f"outs is missing {n}")
        _check_like(outs[n], t, n)
    if want_dh0 and outs.get("dh0") is None:
        outs["dh0"] = _state_like(q, cu_seqlens)
    _check_state(outs.get("dh0"), q, cu_seqlens, "dh0")
    return outs


def kda_bwd(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, dO, ctx, *, scale: float = 1.0,
            lower_bound: float = -5.0, eps: float = 1e-6, workspace=None, outs=None,
            flags: int = 0, dht=None, want_dh0: bool = False):
    """Backward. Returns dict dq, dk, dv, dg, dbeta, dA_log, ddt_bias, and dh0
    (the initial-state gradient) when want_dh0. dht: gradient of the final
    states [N, H, D, D] fp32 (zero when None). ctx must come from a forward
    with the same h0."""
    _check_tensors(q, k, v, g, beta, dO, params=(A_log, dt_bias))
    _check_shapes(q, (("k", k), ("v", v), ("g", g), ("dO", dO)), beta, (A_log, dt_bias))
    _check_state(dht, q, cu_seqlens, "dht")
    p = _problem_from(q, beta, cu_seqlens, scale, lower_bound, eps, flags)
    if q.shape[0] > 0:
        _check_buffer(ctx, _bwd_ctx_bytes(p), q, "ctx")
    outs = _grad_outs(outs, q, k, v, g, beta, A_log, dt_bias, cu_seqlens, want_dh0)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(p), dtype=torch.uint8, device=q.device)
    else:
        _check_buffer(workspace, workspace_bytes(p), q, "workspace")
    st = load_library().kda_bwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
        _ptr(dO), _ptr(dht), _ptr(ctx), _ptr(outs["dq"]), _ptr(outs["dk"]), _ptr(outs["dv"]),
        _ptr(outs["dg"]), _ptr(outs["dbeta"]), _ptr(outs["dA_log"]), _ptr(outs["ddt_bias"]),
        _ptr(outs.get("dh0")), _ptr(workspace), _stream_handle(q.device))
    _check(st, "kda_bwd")
    return outs


def kda_bwd_noalloc(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, dO, ctx, *, scale: float = 1.0,
                    lower_bound: float = -5.0, eps: float = 1e-6, outs=None, dht=None,
                    want_dh0: bool = False):
    """Backward through kda_bwd_noalloc: no workspace, the library's fixed
    scratch array is used instead (for callers that cannot allocate device
    memory at this point; calls must not overlap on the GPU). Returns the
    same dict as kda_bwd."""
    _check_tensors(q, k, v, g, beta, dO, params=(A_log, dt_bias))
    _check_shapes(q, (("k", k), ("v", v), ("g", g), ("dO", dO)), beta, (A_log, dt_bias))
    _check_state(dht, q, cu_seqlens, "dht")
    p = _problem_from(q, beta, cu_seqlens, scale, lower_bound, eps)
    if q.shape[0] > 0:
        _check_buffer(ctx, _bwd_ctx_bytes(p), q, "ctx")
    outs = _grad_outs(outs, q, k, v, g, beta, A_log, dt_bias, cu_seqlens, want_dh0)
    st = load_library().kda_bwd_noalloc(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
        _ptr(dO), _ptr(dht), _ptr(ctx), _ptr(outs["dq"]), _ptr(outs["dk"]), _ptr(outs["dv"]),
        _ptr(outs["dg"]), _ptr(outs["dbeta"]), _ptr(outs["dA_log"]), _ptr(outs["ddt_bias"]),
        _ptr(outs.get("dh0")), _stream_handle(q.device))
    _check(st, "kda_bwd_noalloc")
    return outs


def gdn2_fwd(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, *, scale: float = 1.0,
             lower_bound: float = -5.0, eps: float = 1e-6, save_ctx: bool = True, out=None,
             ctx=None, h0=None, final_state=False, flags: int = 0):
    """GDN-2 forward (kda_gdn2_fwd): KDA with the scalar beta replaced by the
    channel-wise erase gate sigmoid(erase) on key channels and write gate
    sigmoid(write) on value channels; erase and write are [S, H, D] in q's
    dtype. Returns (o, ctx) or (o, ctx, hT) as kda_fwd does."""
    _check_tensors(q, k, v, g, erase, write, params=(A_log, dt_bias))
    _check_shapes(q, (("k", k), ("v", v), ("g", g), ("erase", erase), ("write", write)), None,
                  (A_log, dt_bias))
    _check_state(h0, q, cu_seqlens, "h0")
    flags |= KDA_FLAG_CHANNEL_GATES | (0 if save_ctx else KDA_FLAG_NO_CHECKPOINTS)
    p = _problem_from(q, None, cu_seqlens, scale, lower_bound, eps, flags)
    hT = None
    if final_state is not False and final_state is not None:
        hT = _state_like(q, cu_seqlens) if final_state is True else final_state
        _check_state(hT, q, cu_seqlens, "final_state")
    if out is not None:
        _check_like(out, q, "out")
    o = torch.empty_like(q) if out is None else out
    if ctx is None:
        ctx = torch.empty(ctx_bytes(p), dtype=torch.uint8, device=q.device)
    else:
        _check_buffer(ctx, ctx_bytes(p), q, "ctx")
    st = load_library().kda_gdn2_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(erase),
                                     _ptr(write), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o), _ptr(hT),
                                     _ptr(ctx), _stream_handle(q.device))
    _check(st, "kda_gdn2_fwd")
    if not save_ctx:
        ctx = None
    return (o, ctx) if hT is None else (o, ctx, hT)


def gdn2_bwd(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, dO, ctx, *, scale: float = 1.0,
             lower_bound: float = -5.0, eps: float = 1e-6, workspace=None, outs=None, dht=None,
             want_dh0: bool = False, flags: int = 0):
    """GDN-2 backward (kda_gdn2_bwd). Returns dict dq, dk, dv, dg, derase,
    dwrite, dA_log, ddt_bias, and dh0 when want_dh0. ``flags`` must match
    the forward's (KDA_FLAG_FORCE_SIMT)."""
    _check_tensors(q, k, v, g, erase, write, dO, params=(A_log, dt_bias))
    _check_shapes(q, (("k", k), ("v", v), ("g", g), ("erase", erase), ("write", write), ("dO", dO)),
                  None, (A_log, dt_bias))
    _check_state(dht, q, cu_seqlens, "dht")
    p = _problem_from(q, None, cu_seqlens, scale, lower_bound, eps, flags | KDA_FLAG_CHANNEL_GATES)
    if q.shape[0] > 0:
        _check_buffer(ctx, _bwd_ctx_bytes(p), q, "ctx")
    like = dict(dq=q, dk=k, dv=v, dg=g, derase=erase, dwrite=write, dA_log=A_log, ddt_bias=dt_bias)
    if outs is None:
        outs = {n: torch.empty_like(t) for n, t in like.items()}
    for n, t in like.items():
        if n not in outs:
            raise ValueError(f"outs is missing {n}")
        _check_like(outs[n], t, n)
    if want_dh0 and outs.get("dh0") is None:
        outs["dh0"] = _state_like(q, cu_seqlens)
    _check_state(outs.get("dh0"), q, cu_seqlens, "dh0")
    if workspace is None:
        workspace = torch.empty(workspace_bytes(p), dtype=torch.uint8, device=q.device)
    else:
        _check_buffer(workspace, workspace_bytes(p), q, "workspace")
    st = load_library().kda_gdn2_bwd(
        ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(erase), _ptr(write), _ptr(A_log),
        _ptr(dt_bias), _ptr(dO), _ptr(dht), _ptr(ctx), _ptr(outs["dq"]), _ptr(outs["dk"]),
        _ptr(outs["dv"]), _ptr(outs["dg"]), _ptr(outs["derase"]), _ptr(outs["dwrite"]),
        _ptr(outs["dA_log"]), _ptr(outs["ddt_bias"]), _ptr(outs.get("dh0")), _ptr(workspace),
        _stream_handle(q.device))
    _check(st, "kda_gdn2_bwd")
    return outs


def query_device_status(buf) -> int:
    """Status word written by the kernels into a ctx or workspace buffer."""
    return int(load_library().kda_query_device_status(_ptr(buf), _stream_handle(buf.device)))


def noalloc_device_status(device=None) -> int:
    """Status word of the last kda_bwd_noalloc call on ``device`` (the
    current CUDA device by default), read without any allocation."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(load_library().kda_noalloc_device_status(_stream_handle(dev)))


KDA_PREFIX_FORWARD = 0
KDA_PREFIX_BACKWARD = 1


def state_prefix(A, B, x0=None, *, direction: int, layout: str, x_end=None):
    """kda_state_prefix: the affine prefix over the pieces of each sequence.

    A, B: fp32 CUDA tensors of D x D matrices, either ``layout="seq_major"``
    [N, P, H, D, D] (each sequence's pieces packed as consecutive sequences,
    as kda_fwd / kda_bwd return their states) or ``layout="piece_major"``
    [P, N, H, D, D] (maps gathered from P ranks). x0: [N, H, D, D] or None
    (zero). Returns (xs, x_end): xs in A's layout holds each piece's start
    state (KDA_PREFIX_FORWARD) or end-state gradient (KDA_PREFIX_BACKWARD);
    x_end [N, H, D, D] the final state / the gradient of the first piece's
    start state."""
    if A.dim() != 5 or A.shape != B.shape or A.dtype != torch.float32 or B.dtype != torch.float32:
        raise ValueError("A and B must be fp32 tensors of one 5-d shape")
    for t in (A, B):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("A and B must be contiguous CUDA tensors")
    if layout == "seq_major":
        N, P, H, D, _ = A.shape
        ps, ss = H, P * H
    elif layout == "piece_major":
        P, N, H, D, _ = A.shape
        ps, ss = N * H, H
    else:
        raise ValueError("layout must be 'seq_major' or 'piece_major'")
    want = (N, H, D, D)
    if x0 is not None and (tuple(x0.shape) != want or x0.dtype != torch.float32 or not x0.is_contiguous()):
        raise ValueError(f"x0 must be a contiguous fp32 tensor of shape {want}")
    xs = torch.empty_like(A)
    if x_end is None:
        x_end = torch.empty(want, dtype=torch.float32, device=A.device)
    st = load_library().kda_state_prefix(N, P, H, D, int(direction), ps, ss, _ptr(A), _ptr(B), _ptr(x0),
                                         _ptr(xs), _ptr(x_end), _stream_handle(A.device))
    _check(st, "kda_state_prefix")
    return xs, x_end


class GDN2Function(torch.autograd.Function):
    """Autograd wrapper of the GDN-2 operator (saves the inputs and ctx only)."""

    @staticmethod
    def forward(actx, q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, h0, output_final_state,
                scale, lower_bound, eps):
        r = gdn2_fwd(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, scale=scale,
                     lower_bound=lower_bound, eps=eps, save_ctx=True, h0=h0,
                     final_state=bool(output_final_state))
        actx.save_for_backward(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, r[1])
        actx.args = (scale, lower_bound, eps, h0 is not None)
        return (r[0], r[2]) if output_final_state else r[0]

    @staticmethod
    def backward(actx, dO, dht=None):
        q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, ctx = actx.saved_tensors
        scale, lower_bound, eps, has_h0 = actx.args
        r = gdn2_bwd(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, dO.contiguous(), ctx,
                     scale=scale, lower_bound=lower_bound, eps=eps,
                     dht=None if dht is None else dht.contiguous(), want_dh0=has_h0)
        return (r["dq"], r["dk"], r["dv"], r["dg"], r["derase"], r["dwrite"], r["dA_log"],
                r["ddt_bias"], None, r.get("dh0"), None, None, None, None)


def gdn2(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, scale: float = 1.0,
         lower_bound: float = -5.0, eps: float = 1e-6, initial_state=None,
         output_final_state: bool = False):
    """Differentiable GDN-2 (channel-wise erase / write gates) over packed
    sequences; arguments as for ``kda`` with erase / write [S, H, D] in place
    of beta."""
    return GDN2Function.apply(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, initial_state,
                              output_final_state, scale, lower_bound, eps)


class KDAFunction(torch.autograd.Function):
    """Autograd wrapper: forward saves the inputs and the checkpoint ctx only."""

    @staticmethod
    def forward(actx, q, k, v, g, beta, A_log, dt_bias, cu_seqlens, h0, output_final_state, scale,
                lower_bound, eps, fwd_flags=0):
        r = kda_fwd(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, scale=scale, lower_bound=lower_bound,
                    eps=eps, save_ctx=True, h0=h0, final_state=bool(output_final_state), flags=fwd_flags)
        o, ctx = r[0], r[1]
        actx.save_for_backward(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, ctx)
        actx.args = (scale, lower_bound, eps, h0 is not None, bool(output_final_state))
        return (o, r[2]) if output_final_state else o

    @staticmethod
    def backward(actx, dO, dht=None):
        q, k, v, g, beta, A_log, dt_bias, cu_seqlens, ctx = actx.saved_tensors
        scale, lower_bound, eps, has_h0, _ = actx.args
        r = kda_bwd(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, dO.contiguous(), ctx,
                    scale=scale, lower_bound=lower_bound, eps=eps,
                    dht=None if dht is None else dht.contiguous(), want_dh0=has_h0)
        return (r["dq"], r["dk"], r["dv"], r["dg"], r["dbeta"], r["dA_log"], r["ddt_bias"],
                None, r.get("dh0"), None, None, None, None, None)


def kda(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, scale: float = 1.0,
        lower_bound: float = -5.0, eps: float = 1e-6, initial_state=None,
        output_final_state: bool = False, chunk_size: int = 64):
    """Differentiable KDA over packed sequences (see include/kda.h). With
    initial_state ([N, H, D, D] fp32) the recurrences start from it; with
    output_final_state the call returns (o, final_state). chunk_size 16
    selects the forward with 16-token chunks (KDA_FLAG_CHUNK16: bf16, head_dim
    128); the backward is the same either way."""
    if chunk_size not in (16, 64):
        raise ValueError(f"chunk_size must be 16 or 64 (got {chunk_size})")
    return KDAFunction.apply(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, initial_state,
                             output_final_state, scale, lower_bound, eps,
                             KDA_FLAG_CHUNK16 if chunk_size == 16 else 0)
