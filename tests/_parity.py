"""Helpers for GPU-vs-oracle parity tests (test-only)."""
import numpy as np
import torch

import oracle
from recompute_kda_chunkwise_gb300 import kda as K

OUT_NAMES = ["o", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"]
# bf16 inputs: max|x - ref| <= 2e-2 * RMS(ref); fp32 inputs: <= 1e-4 * RMS(ref)
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def run_gpu(inp, scale=1.0, lower=-5.0, eps=1e-6, flags=0):
    o, ctx = K.kda_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                       inp["dt_bias"], inp["cu_seqlens"], scale=scale, lower_bound=lower, eps=eps,
                       flags=flags)
    r = K.kda_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
                  inp["cu_seqlens"], inp["dO"], ctx, scale=scale, lower_bound=lower, eps=eps,
                  flags=flags)
    torch.cuda.synchronize()
    r["o"] = o
    return r, ctx


def to_dev(inp, device="cuda"):
    return {k: (v.to(device) if v is not None else None) for k, v in inp.items()}


# Significant bits of the stored output type: storing the exact value r in
# that type alone errs by up to half an ulp of r's binade,
# 2^(floor(log2|r|) - bits).
SIG_BITS = {torch.bfloat16: 8, torch.float32: 24}


def half_ulp(r: np.ndarray, bits: int) -> np.ndarray:
    a = np.abs(r)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - bits).astype(np.int64)), 0.0)


def compare(gpu: dict, ref: dict, tol: float, heads=None, names=OUT_NAMES, rel: float = 0.0):
    """Per tensor: the computation error beyond the output's own rounding,
    max(|x - ref| - half_ulp(ref, dtype) - rel * |ref|), divided by
    RMS(ref), must be <= tol. Returns the worst ratio per name. ``rel`` is an
    extra per-element relative allowance (zero for the configurations'
    parity tests)."""
    report = {}
    for n in names:
        x = gpu[n]
        bits = SIG_BITS[x.dtype]
        if heads is not None:
            idx = torch.tensor(heads, device=x.device)
            x = x.index_select(0 if n in ("dA_log", "ddt_bias") else 1, idx)
        x = x.detach().double().cpu().numpy()
        r = ref[n]
        assert x.shape == r.shape, (n, x.shape, r.shape)
        assert np.all(np.isfinite(x)), f"{n} has non-finite values"
        rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
        err = float(np.max(np.abs(x - r) - half_ulp(r, bits) - rel * np.abs(r))) if r.size else 0.0
        err = max(err, 0.0)
        ratio = err / rms if rms > 0 else err
        report[n] = ratio
    bad = {n: v for n, v in report.items() if not v <= tol}
    assert not bad, f"parity failure (tol {tol}): {bad}; all: {report}"
    return report


def oracle_for(inp, heads=None, scale=1.0, lower=-5.0, eps=1e-6, threads=None):
    cpu = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    if heads is None:
        return oracle.kda_reference(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"],
                                    cpu["A_log"], cpu["dt_bias"], cpu["cu_seqlens"], cpu["dO"],
                                    scale=scale, lower_bound=lower, eps=eps, threads=threads)
    return oracle.kda_reference_heads(cpu, heads, scale=scale, lower_bound=lower, eps=eps,
                                      threads=threads)
