"""fp32 range of the intra-chunk factors (CPU only).

"KDA at the production shape ...", section 3(a): the inverse-decay factor of
k leaves fp32 range once the cumulative log-decay passes about -88, which at
the -5 gate floor limits a factored chunk to 17 tokens. Two facts follow, and
both kernel families are built on them:
  * factored as (k e^G)(k e^-G)^T, a 16-token chunk stays finite in fp32 at
    the floor (the 16-token chunks of the backward and of the D = 64 kernels),
    while a 64-token chunk does not;
  * a 64-token chunk evaluated in 16-token column blocks J, each referenced
    at the end of its block (column operand k e^(B_J - G), row operand
    k e^(G - B_J)), stays finite and accurate (the forward's sub-block
    references).
"""
import numpy as np


def _chunk(C, D=16, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((C, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    g = np.full((C, D), -5.0)           # every gate at the -5 floor
    G = np.cumsum(g, 0)                  # inclusive cumulative log-decay
    exact = np.zeros((C, C))
    for r in range(C):
        for s in range(r):
            exact[r, s] = np.sum(k[r] * k[s] * np.exp(G[r] - G[s]))
    return k, G, exact


def _factored_fp32(k, G):
    k32, G32 = k.astype(np.float32), G.astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        rows = k32 * np.exp(G32)
        cols = k32 * np.exp(-G32)
        return np.tril(rows @ cols.T, -1)


def _sub_block_fp32(k, G, B=16):
    C = k.shape[0]
    k32, G32 = k.astype(np.float32), G.astype(np.float32)
    out = np.zeros((C, C), np.float32)
    for J in range(C // B):
        ref = G32[B * J + B - 1]                        # end of column block J
        cols = k32[B * J:B * J + B] * np.exp(ref - G32[B * J:B * J + B])
        rows = k32[B * J:] * np.exp(G32[B * J:] - ref)  # row blocks I >= J
        out[B * J:, B * J:B * J + B] = rows @ cols.T
    return np.tril(out, -1)


def test_sixteen_token_chunk_factors_in_fp32_at_the_floor():
    k, G, exact = _chunk(16)
    got = _factored_fp32(k, G)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, exact, rtol=1e-4, atol=1e-6)


def test_sixty_four_token_chunk_does_not_factor_in_fp32():
    k, G, _ = _chunk(64)
    assert not np.all(np.isfinite(_factored_fp32(k, G)))


def test_sub_block_references_keep_a_sixty_four_token_chunk_in_range():
    k, G, exact = _chunk(64)
    got = _sub_block_fp32(k, G)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, exact, rtol=1e-4, atol=1e-6)
