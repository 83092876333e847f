"""fp64 CPU oracle for Kimi Delta Attention (KDA) forward and backward.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may use this package; the product library never does. The
oracle shares no code with the CUDA path. It is plain C (``kda_oracle.c``,
token-by-token recurrence plus its hand-derived reverse-time adjoint) built
with gcc into ``oracle/_build/libkda_oracle.so`` and called through ctypes.

Parity status of each part (what pins it is listed in the tests):
  * recurrence, output and final state -- pinned (explicit transition-matrix
    product form, closed-form special cases, invariants, chaining of a
    sequence split in two through its state);
  * backward, with the initial-state gradient -- pinned (central finite
    differences, fp64 autograd of an independent explicit-matrix forward);
  * gate formula g = L*sigmoid(exp(A_log)*(a + dt_bias)) and the shapes
    A_log[H], dt_bias[H,D] -- parity unpinned: the pages name only a
    "safe gate with lower bound -5" built from these three inputs;
  * GDN-2 channel-wise erase / write gates (``gdn2_reference``) -- recurrence
    and backward pinned (explicit-matrix autograd, finite differences, the
    KDA special case b = w = beta, the closed form with no erasing); the
    sigmoid activation of the two raw gates is a reading (unpinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, portable, no -march flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            f = lib.kda_oracle_run
            dp = ctypes.POINTER(ctypes.c_double)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                          ctypes.c_int, dp, dp, dp, dp, dp, dp, dp,
                          ctypes.c_double, ctypes.c_double, ctypes.c_double, dp,
                          dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            f2 = lib.gdn2_oracle_run
            f2.restype = ctypes.c_int
            f2.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                           ctypes.c_int, dp, dp, dp, dp, dp, dp, dp, dp,
                           ctypes.c_double, ctypes.c_double, ctypes.c_double, dp,
                           dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x, shape=None):
    if hasattr(x, "detach"):  # a torch tensor: widen on its own side first
        x = x.detach().to("cpu").double().numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def kda_reference(q, k, v, g, beta, A_log, dt_bias, cu_seqlens, dO=None, *,
                  scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6,
                  threads: int | None = None, want_o: bool = True, h0=None, dht=None,
                  want_state: bool = False) -> dict:
    """Run the oracle.

    Arrays are numpy arrays or torch tensors; they are widened to float64
    (exact for bf16 and fp32 values). q,k,v,g,dO: [S,H,D]; beta: [S,H]; A_log: [H];
    dt_bias: [H,D]; cu_seqlens: [N+1] int; h0 (initial states) and dht
    (gradient of the final states): [N,H,D,D] (rows: key index), zero when
    None. Returns float64 arrays: 'o' (when want_o) and, when dO is given,
    'dq','dk','dv','dg','dbeta','dA_log','ddt_bias'. With want_state (or h0 /
    dht given) it also returns the final states 'hT' and, when dO is given,
    the initial-state gradient 'dh0', both [N,H,D,D].
    """
    q = _f64(q)
    if q.ndim != 3:
        raise ValueError("q must be [S,H,D]")
    S, H, D = q.shape
    k = _f64(k, (S, H, D)); v = _f64(v, (S, H, D)); g = _f64(g, (S, H, D))
    beta = _f64(beta, (S, H)); A_log = _f64(A_log, (H,)); dt_bias = _f64(dt_bias, (H, D))
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or cu[-1] != S:
        raise ValueError("cu_seqlens must start at 0 and end at S")
    N = cu.size - 1
    want_state = want_state or h0 is not None or dht is not None
    h0 = None if h0 is None else _f64(h0, (N, H, D, D))
    dht = None if dht is None else _f64(dht, (N, H, D, D))
    out = {}
    hT = dh0 = None
    if want_state:
        hT = out["hT"] = np.zeros((N, H, D, D))
        if dO is not None:
            dh0 = out["dh0"] = np.zeros((N, H, D, D))
    o = np.zeros((S, H, D), np.float64) if want_o else None
    if want_o:
        out["o"] = o
    grads = None
    if dO is not None:
        dO = _f64(dO, (S, H, D))
        grads = dict(dq=np.zeros((S, H, D)), dk=np.zeros((S, H, D)), dv=np.zeros((S, H, D)),
                     dg=np.zeros((S, H, D)), dbeta=np.zeros((S, H)),
                     dA_log=np.zeros((H,)), ddt_bias=np.zeros((H, D)))
        out.update(grads)
    if threads is None:
        threads = os.cpu_count() or 1
    lib = _load()
    fp = dpt = ctypes.c_double
    G = grads or {}
    rc = lib.kda_oracle_run(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, D,
        _ptr(q, fp), _ptr(k, fp), _ptr(v, fp), _ptr(g, fp), _ptr(beta, fp),
        _ptr(A_log, fp), _ptr(dt_bias, fp), float(scale), float(lower_bound), float(eps),
        _ptr(dO, fp), _ptr(o, dpt), _ptr(G.get("dq"), dpt), _ptr(G.get("dk"), dpt),
        _ptr(G.get("dv"), dpt), _ptr(G.get("dg"), dpt), _ptr(G.get("dbeta"), dpt),
        _ptr(G.get("dA_log"), dpt), _ptr(G.get("ddt_bias"), dpt), _ptr(h0, fp), _ptr(hT, dpt),
        _ptr(dht, fp), _ptr(dh0, dpt), int(threads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_run failed with code {rc}")
    return out


def kda_reference_heads(inputs: dict, heads, dO=True, *, scale=1.0, lower_bound=-5.0,
                        eps=1e-6, threads=None, group=16) -> dict:
    """Oracle over a subset of heads (heads are independent, so this equals the
    full run restricted to those heads). ``inputs`` holds torch tensors or
    arrays named q,k,v,g,beta,A_log,dt_bias,cu_seqlens and optionally dO.
    Results are stacked along the head axis in the order of ``heads``; heads
    are processed ``group`` at a time to bound host memory."""
    heads = list(heads)
    parts = []
    for s in range(0, len(heads), group):
        hs = heads[s:s + group]
        def sel(x, axis):
            if hasattr(x, "detach"):
                import torch
                return x.index_select(axis, torch.tensor(hs, device=x.device)).cpu()
            return np.take(np.asarray(x), hs, axis=axis)
        parts.append(kda_reference(
            sel(inputs["q"], 1), sel(inputs["k"], 1), sel(inputs["v"], 1), sel(inputs["g"], 1),
            sel(inputs["beta"], 1), sel(inputs["A_log"], 0), sel(inputs["dt_bias"], 0),
            inputs["cu_seqlens"], sel(inputs["dO"], 1) if dO else None,
            scale=scale, lower_bound=lower_bound, eps=eps, threads=threads))
    out = {}
    for key in parts[0]:
        axis = 0 if key in ("dA_log", "ddt_bias") else 1
        out[key] = np.concatenate([p[key] for p in parts], axis=axis)
    return out


def gdn2_reference(q, k, v, g, erase, write, A_log, dt_bias, cu_seqlens, dO=None, *,
                   scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6,
                   threads: int | None = None, want_o: bool = True, h0=None, dht=None,
                   want_state: bool = False) -> dict:
    """Run the GDN-2 oracle: KDA with the scalar beta replaced by channel-wise
    gates, erase b_t = sigmoid(erase_t) on key channels and write
    w_t = sigmoid(write_t) on value channels (see gdn2_oracle_run in
    kda_oracle.c). erase and write are [S,H,D]; everything else as in
    kda_reference. Returns 'o' and, when dO is given, 'dq','dk','dv','dg',
    'derase','dwrite','dA_log','ddt_bias' (plus 'hT' / 'dh0' with states)."""
    q = _f64(q)
    if q.ndim != 3:
        raise ValueError("q must be [S,H,D]")
    S, H, D = q.shape
    k = _f64(k, (S, H, D)); v = _f64(v, (S, H, D)); g = _f64(g, (S, H, D))
    erase = _f64(erase, (S, H, D)); write = _f64(write, (S, H, D))
    A_log = _f64(A_log, (H,)); dt_bias = _f64(dt_bias, (H, D))
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    if cu.ndim != 1 or cu.size < 1 or cu[0] != 0 or cu[-1] != S:
        raise ValueError("cu_seqlens must start at 0 and end at S")
    N = cu.size - 1
    want_state = want_state or h0 is not None or dht is not None
    h0 = None if h0 is None else _f64(h0, (N, H, D, D))
    dht = None if dht is None else _f64(dht, (N, H, D, D))
    out = {}
    hT = dh0 = None
    if want_state:
        hT = out["hT"] = np.zeros((N, H, D, D))
        if dO is not None:
            dh0 = out["dh0"] = np.zeros((N, H, D, D))
    o = np.zeros((S, H, D), np.float64) if want_o else None
    if want_o:
        out["o"] = o
    G = {}
    if dO is not None:
        dO = _f64(dO, (S, H, D))
        G = dict(dq=np.zeros((S, H, D)), dk=np.zeros((S, H, D)), dv=np.zeros((S, H, D)),
                 dg=np.zeros((S, H, D)), derase=np.zeros((S, H, D)), dwrite=np.zeros((S, H, D)),
                 dA_log=np.zeros((H,)), ddt_bias=np.zeros((H, D)))
        out.update(G)
    if threads is None:
        threads = os.cpu_count() or 1
    lib = _load()
    fp = ctypes.c_double
    rc = lib.gdn2_oracle_run(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, D,
        _ptr(q, fp), _ptr(k, fp), _ptr(v, fp), _ptr(g, fp), _ptr(erase, fp), _ptr(write, fp),
        _ptr(A_log, fp), _ptr(dt_bias, fp), float(scale), float(lower_bound), float(eps),
        _ptr(dO, fp), _ptr(o, fp), _ptr(G.get("dq"), fp), _ptr(G.get("dk"), fp),
        _ptr(G.get("dv"), fp), _ptr(G.get("dg"), fp), _ptr(G.get("derase"), fp),
        _ptr(G.get("dwrite"), fp), _ptr(G.get("dA_log"), fp), _ptr(G.get("ddt_bias"), fp),
        _ptr(h0, fp), _ptr(hT, fp), _ptr(dht, fp), _ptr(dh0, fp), int(threads))
    if rc != 0:
        raise RuntimeError(f"gdn2_oracle_run failed with code {rc}")
    return out
