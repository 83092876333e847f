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


# Raw max|x - ref| / RMS(ref) of the last compare() per tensor, beside the
# adjusted ratio the bar applies to (printed by compare()).
LAST_RAW = {}


def _errors(x: np.ndarray, r: np.ndarray, bits: int):
    """(max(|x - ref| - half_ulp(ref)), max|x - ref|, sum ref^2, count)."""
    if not r.size:
        return 0.0, 0.0, 0.0, 0
    d = np.abs(x - r)
    return (float(np.max(d - half_ulp(r, bits))), float(np.max(d)), float(np.sum(r * r)), r.size)


def compare(gpu: dict, ref: dict, tol: float, heads=None, names=OUT_NAMES):
    """Per tensor: the computation error beyond the output's own rounding,
    max(|x - ref| - half_ulp(ref, dtype)), divided by RMS(ref), must be
    <= tol. Returns the worst ratio per name; the raw max|x - ref| / RMS(ref)
    is printed beside it (and kept in LAST_RAW)."""
    report, raw = {}, {}
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
        err, err_raw, ss, cnt = _errors(x, r, bits)
        rms = float(np.sqrt(ss / cnt)) if cnt else 0.0
        report[n] = max(err, 0.0) / rms if rms > 0 else max(err, 0.0)
        raw[n] = err_raw / rms if rms > 0 else err_raw
    LAST_RAW.clear()
    LAST_RAW.update(raw)
    print("parity (adjusted / raw max-err over RMS): " +
          ", ".join(f"{n} {report[n]:.3e} / {raw[n]:.3e}" for n in names))
    bad = {n: v for n, v in report.items() if not v <= tol}
    assert not bad, f"parity failure (tol {tol}): {bad}; all: {report}; raw: {raw}"
    return report


def compare_heads_streaming(gpu: dict, inp: dict, heads, tol: float, *, group: int = 16,
                            scale: float = 1.0, names=OUT_NAMES):
    """compare() over many heads of a large problem, ``group`` heads at a
    time, so that the oracle's fp64 results never sit in host memory for
    every head at once. The bar is the same: per tensor, the worst error
    over all checked heads against the RMS over all checked heads."""
    heads = list(heads)
    acc = {n: [0.0, 0.0, 0.0, 0] for n in names}
    for s in range(0, len(heads), group):
        hs = heads[s:s + group]
        ref = oracle_for(inp, heads=hs, scale=scale)
        for n in names:
            x = gpu[n]
            idx = torch.tensor(hs, device=x.device)
            x = x.index_select(0 if n in ("dA_log", "ddt_bias") else 1, idx).detach().double().cpu().numpy()
            assert x.shape == ref[n].shape, (n, x.shape, ref[n].shape)
            assert np.all(np.isfinite(x)), f"{n} has non-finite values"
            e, er, ss, cnt = _errors(x, ref[n], SIG_BITS[gpu[n].dtype])
            a = acc[n]
            a[0], a[1], a[2], a[3] = max(a[0], e), max(a[1], er), a[2] + ss, a[3] + cnt
        del ref
    report, raw = {}, {}
    for n, (e, er, ss, cnt) in acc.items():
        rms = (ss / cnt) ** 0.5 if cnt else 0.0
        report[n] = max(e, 0.0) / rms if rms > 0 else max(e, 0.0)
        raw[n] = er / rms if rms > 0 else er
    LAST_RAW.clear()
    LAST_RAW.update(raw)
    print(f"parity over {len(heads)} heads (adjusted / raw max-err over RMS): " +
          ", ".join(f"{n} {report[n]:.3e} / {raw[n]:.3e}" for n in names))
    bad = {n: v for n, v in report.items() if not v <= tol}
    assert not bad, f"parity failure (tol {tol}): {bad}; all: {report}; raw: {raw}"
    return report


def oracle_for(inp, heads=None, scale=1.0, lower=-5.0, eps=1e-6, threads=None):
    cpu = {k: (v.cpu() if v is not None else None) for k, v in inp.items()}
    if heads is None:
        return oracle.kda_reference(cpu["q"], cpu["k"], cpu["v"], cpu["g"], cpu["beta"],
                                    cpu["A_log"], cpu["dt_bias"], cpu["cu_seqlens"], cpu["dO"],
                                    scale=scale, lower_bound=lower, eps=eps, threads=threads)
    return oracle.kda_reference_heads(cpu, heads, scale=scale, lower_bound=lower, eps=eps,
                                      threads=threads)
