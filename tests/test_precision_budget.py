"""Error budget of the forward's operand roundings, from an fp64 emulation of
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
