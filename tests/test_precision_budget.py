"""Error budget of the kernels' operand roundings, from an fp64 emulation of
the chunk algebra (not the kernels; CPU only).

The output o = (Qh Gamma) H + M U~ of a chunk ("KDA at the production shape
...", section 2.1: the aqk / akk / w / u / v_new / intra / inter / state-update
op table) is formed here three ways on the same synthetic head (N(0,1) inputs,
A_log = dt_bias = 0, scale 1, 8192 tokens):
- exactly, in fp64;
- with the roundings both tensor-core forwards apply to their fp16 operands
  (the state H and Qh Gamma of the state part, -W and H of U~ = U - W H,
  U~ and Kbar of the state update);
- with those plus single-pass tf32 operands in the Abar / M products, formed
  per 16-token column block referenced at the block's end, as the 64-token
  forward forms them: its fp32 operands go to the tf32 MMA as they are, and
  a tf32 MMA reads fp32 data with the low 13 mantissa bits dropped
  (truncation); rounding them to nearest first is the alternative compared
  (the 16-token forward forms Abar / M from hi + lo tf32 parts, which this
  emulation takes as exact).
Each is stored as bf16 and measured the way the parity tests measure it:
max(|x - ref| - half an ulp of ref) / RMS(ref).

What it shows: the tf32 Abar / M operands, not the fp16 state operands, set
the 64-token forward's output error. Truncated, they give about 1e-2 of RMS
on a head, the size the GPU parity runs measure (1.3e-2 on a 16-head sample
of the long-context run); rounded to nearest they would give less than half
of that; the fp16 operands together give under 1e-3, the share the 16-token
forward's scheme stays at. All sit below the 2e-2 bar.

The backward (16-token chunks) is emulated the same way, with its roundings
grouped: the rebuilt chunk-start states kept as fp16 tiles, the fp16 copy of
dH' in its products, the other fp16 state-product operands, the plain-tf32
dV product, and the fp16 operands of the state rebuild. dv's error is the
tf32 product's alone; dg's comes from the fp16 state side.
"""
import numpy as np
import pytest

C16, C64, BLOCK, D, TOKENS = 16, 64, 16, 128, 8192


def _bf16(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _tf32(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0xFFF + ((b >> 13) & 1)) >> 13) << 13
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _tf32_truncated(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    return (b & np.uint32(0xFFFFE000)).view(np.float32).astype(np.float64)


def _fp16(x):
    return np.asarray(x, dtype=np.float16).astype(np.float64)


def _exact(x):
    return x


def _pair_matrix(X, Y, G, strict, rnd):
    """sum_i X_ri Y_si e^{G_ri - G_si}, per 16-token column block J with the
    reference B_J = G at the end of J (row operand X e^{G - B_J}, column
    operand Y e^{B_J - G}, each rounded by rnd); s < r (strict) or s <= r."""
    n = X.shape[0]
    out = np.zeros((n, n))
    for j0 in range(0, n, BLOCK):
        j1 = min(n, j0 + BLOCK)
        ref = G[j1 - 1]
        col = rnd(Y[j0:j1] * np.exp(ref - G[j0:j1]))
        row = rnd(X[j0:] * np.exp(G[j0:] - ref))
        out[j0:, j0:j1] = row @ col.T
    r, s = np.indices((n, n))
    return np.where(s < r if strict else s <= r, out, 0.0)


def _forward(inp, C, op16, op_am):
    q, k, v, a, b = inp
    S = q.shape[0]
    H = np.zeros((D, D))
    o = np.zeros((S, D))
    for c0 in range(0, S, C):
        sl = slice(c0, min(S, c0 + C))
        n = sl.stop - sl.start
        qh = q[sl] / np.sqrt((q[sl] ** 2).sum(1, keepdims=True) + 1e-6)
        kh = k[sl] / np.sqrt((k[sl] ** 2).sum(1, keepdims=True) + 1e-6)
        beta = 1.0 / (1.0 + np.exp(-b[sl]))
        G = np.cumsum(-5.0 / (1.0 + np.exp(-a[sl])), axis=0)
        Abar = _pair_matrix(kh, kh, G, True, op_am) * beta[:, None]
        M = _pair_matrix(qh, kh, G, False, op_am)
        Tp = np.linalg.inv(np.eye(n) + Abar) * beta[None, :]
        W = Tp @ (kh * np.exp(G))
        U = Tp @ v[sl]
        Ut = U + op16(-W) @ op16(H)
        o[sl] = op16(qh * np.exp(G)) @ op16(H) + M @ Ut
        Kbar = kh * np.exp(G[-1] - G)
        H = np.exp(G[-1])[:, None] * H + op16(Kbar).T @ op16(Ut)
    return o


def _adjusted_error(x, ref):
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    half_ulp = np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)
    return np.maximum(np.abs(x - ref) - half_ulp, 0.0).max() / np.sqrt((ref ** 2).mean())


@pytest.fixture(scope="module")
def head():
    rng = np.random.default_rng(20260)
    q, k, v, a = (_bf16(rng.standard_normal((TOKENS, D))) for _ in range(4))
    b = _bf16(rng.standard_normal(TOKENS))
    return q, k, v, a, b


def test_chunk_size_leaves_the_exact_output_unchanged(head):
    # the blocked references keep the 64-token chunk in range: same o as C = 16
    o16 = _forward(head, C16, _exact, _exact)
    o64 = _forward(head, C64, _exact, _exact)
    assert np.abs(o16 - o64).max() <= 1e-9 * np.abs(o16).max()


def test_tf32_abar_m_operands_set_the_64_token_forwards_output_error(head):
    ref = _forward(head, C64, _exact, _exact)
    fp16_only = _adjusted_error(_bf16(_forward(head, C64, _fp16, _exact)), ref)
    rounded = _adjusted_error(_bf16(_forward(head, C64, _fp16, _tf32)), ref)
    truncated = _adjusted_error(_bf16(_forward(head, C64, _fp16, _tf32_truncated)), ref)
    c16 = _adjusted_error(_bf16(_forward(head, C16, _fp16, _exact)), ref)
    assert truncated > 1.5 * rounded, (truncated, rounded)
    assert rounded > 3.0 * fp16_only, (rounded, fp16_only)
    assert truncated > 5.0 * c16, (truncated, c16)
    assert 5e-3 < truncated < 2e-2 and fp16_only < 1e-3 and c16 < 1e-3, (truncated, fp16_only, c16)


def _backward(inp, dO_all, rH, rdH, rop, rdv, rupd):
    """Gradients of the 16-token backward with its operand roundings: the
    rebuilt chunk-start states as fp16 tiles (rH), the fp16 copy of dH' in
    its products (rdH), the fp16 operands of the other state products (rop:
    Kbar, Qh Gamma, -W, U~, dU~), the plain-tf32 dV = T'^T dU~ (rdv), and
    the fp16 operands of the state rebuild (rupd). Returns dq, dk, dv, dg."""
    q, k, v, a, b = inp
    S = q.shape[0]

    def chunk(t0):
        sl = slice(t0, t0 + C16)
        nq = np.sqrt((q[sl] ** 2).sum(1) + 1e-6)
        nk = np.sqrt((k[sl] ** 2).sum(1) + 1e-6)
        xq, xk = q[sl] / nq[:, None], k[sl] / nk[:, None]
        sg = 1.0 / (1.0 + np.exp(-a[sl]))
        beta = 1.0 / (1.0 + np.exp(-b[sl]))
        G = np.cumsum(-5.0 * sg, axis=0)
        c = dict(xq=xq, xk=xk, nq=nq, nk=nk, sg=sg, beta=beta, G=G, gam=np.exp(G[-1]), V=v[sl])
        c["Qg"], c["Kg"] = xq * np.exp(G), xk * np.exp(G)
        c["Ki"], c["Kb"] = xk * np.exp(-G), xk * np.exp(G[-1] - G)
        c["Xw"], c["Xu"] = beta[:, None] * c["Kg"], beta[:, None] * c["V"]
        c["M"] = np.tril(c["Qg"] @ c["Ki"].T)
        c["T"] = np.linalg.inv(np.eye(C16) + np.tril(c["Xw"] @ c["Ki"].T, -1))
        c["W"], c["U"] = c["T"] @ c["Xw"], c["T"] @ c["Xu"]
        return c

    starts, H = [], np.zeros((D, D))
    for t0 in range(0, S, C16):
        c = chunk(t0)
        starts.append(H)
        Ut = c["U"] + rupd(-c["W"]) @ rupd(H)
        H = c["gam"][:, None] * H + rupd(c["Kb"]).T @ rupd(Ut)
    out = {n: np.zeros((S, D)) for n in ("dq", "dk", "dv", "dg")}
    dH = np.zeros((D, D))
    for i in reversed(range(len(starts))):
        t0 = i * C16
        c, Hc, dO = chunk(t0), rH(starts[i]), dO_all[t0:t0 + C16]
        Ut = c["U"] + rop(-c["W"]) @ Hc
        dHo = rdH(dH)
        dUt = c["M"].T @ dO + rop(c["Kb"]) @ dHo
        dKb = rop(Ut) @ dHo.T
        dgam = (Hc * dH).sum(1)
        dW = -rop(dUt) @ Hc.T
        dQg = dO @ Hc.T
        dH = c["gam"][:, None] * dH + rop(c["Qg"]).T @ dO - rop(c["W"]).T @ rop(dUt)
        dM = np.tril(dO @ Ut.T)
        dT = np.tril(dW @ c["Xw"].T + dUt @ c["Xu"].T, -1)
        dA = np.tril(-(c["T"].T @ dT @ c["T"].T), -1)
        dXw = c["T"].T @ dW + dA @ c["Ki"]
        dXu = rdv(c["T"].T) @ rdv(dUt)
        dKi = dA.T @ c["Xw"] + dM.T @ c["Qg"]
        dQg = dQg + dM @ c["Ki"]
        dKg = c["beta"][:, None] * dXw
        e, ei, eb = np.exp(c["G"]), np.exp(-c["G"]), np.exp(c["G"][-1] - c["G"])
        dxq, dxk = dQg * e, dKg * e + dKi * ei + dKb * eb
        dG = dQg * c["Qg"] + dKg * c["Kg"] - dKi * c["Ki"] - dKb * c["Kb"]
        dg = np.cumsum(dG[::-1], 0)[::-1] + (dKb * c["Kb"]).sum(0) + dgam * c["gam"]
        sl, xq, xk = slice(t0, t0 + C16), c["xq"], c["xk"]
        out["dq"][sl] = (dxq - xq * (xq * dxq).sum(1, keepdims=True)) / c["nq"][:, None]
        out["dk"][sl] = (dxk - xk * (xk * dxk).sum(1, keepdims=True)) / c["nk"][:, None]
        out["dv"][sl] = c["beta"][:, None] * dXu
        out["dg"][sl] = dg * -5.0 * c["sg"] * (1.0 - c["sg"])
    return out


def test_backward_error_sources(head):
    # dv's error is its plain-tf32 product's; dg's comes from the fp16 state
    # side (the rebuilt state tiles and the rebuild's fp16 operands), not
    # from the tf32 product
    rng = np.random.default_rng(20261)
    dO = _bf16(rng.standard_normal((TOKENS, D)))
    ref = _backward(head, dO, *([_exact] * 5))
    err = lambda g: {n: _adjusted_error(_bf16(g[n]), ref[n]) for n in ref}
    full = err(_backward(head, dO, _fp16, _fp16, _fp16, _tf32, _fp16))
    dv_only = err(_backward(head, dO, _exact, _exact, _exact, _tf32, _exact))
    no_dv = err(_backward(head, dO, _fp16, _fp16, _fp16, _exact, _fp16))
    assert dv_only["dv"] > 0.8 * full["dv"] and no_dv["dv"] < 0.5 * full["dv"], (full, dv_only, no_dv)
    assert no_dv["dg"] > 0.8 * full["dg"] and dv_only["dg"] < 1e-4 * full["dg"], (full, dv_only, no_dv)
    assert max(full.values()) < 2e-2, full
