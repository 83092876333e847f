"""Pins for the oracle's GDN-2 mode (channel-wise erase and write gates),
checked against things other than itself:

* the KDA special case: erase = write = beta on every channel reproduces the
  (separately pinned) KDA oracle, and the two gate gradients summed over
  channels give dbeta;
* explicit_forward_gdn2: the recurrence with explicit D x D transition
  matrices, and float64 autograd through it for all nine gradients and the
  state gradient;
* central finite differences of the oracle's own forward;
* closed forms: no erasing (erase gate 0) is gated linear attention with a
  per-channel write gate; no writing (write gate 0) from a zero state gives
  zero output and zero gradients.
"""
import numpy as np
import torch
from scipy.special import expit

import oracle
from tests._explicit import explicit_forward_gdn2

NAMES = ["q", "k", "v", "g", "erase", "write", "A_log", "dt_bias"]
GRADS = dict(q="dq", k="dk", v="dv", g="dg", erase="derase", write="dwrite", A_log="dA_log",
             dt_bias="ddt_bias")


def rand_problem(lengths, H, D, param_std=0.5, seed=0):
    rng = np.random.default_rng(seed)
    S = int(sum(lengths))
    p = {n: rng.standard_normal((S, H, D)) for n in ["q", "k", "v", "g", "erase", "write", "dO"]}
    p["A_log"] = rng.standard_normal(H) * param_std
    p["dt_bias"] = rng.standard_normal((H, D)) * param_std
    p["cu_seqlens"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return p


def run(p, dO=True, **kw):
    return oracle.gdn2_reference(p["q"], p["k"], p["v"], p["g"], p["erase"], p["write"],
                                 p["A_log"], p["dt_bias"], p["cu_seqlens"],
                                 p["dO"] if dO else None, **kw)


def test_equal_gates_reduce_to_kda():
    # 300 + 40 tokens: the first sequence crosses the oracle's 256-token
    # state segments in the reverse loop
    p = rand_problem([300, 40], H=2, D=8, seed=11)
    beta = np.random.default_rng(12).standard_normal((340, 2))
    p["erase"] = p["write"] = np.repeat(beta[:, :, None], 8, axis=2)
    got = run(p, scale=0.5)
    ref = oracle.kda_reference(p["q"], p["k"], p["v"], p["g"], beta, p["A_log"], p["dt_bias"],
                               p["cu_seqlens"], p["dO"], scale=0.5)
    for n in ["o", "dq", "dk", "dv", "dg", "dA_log", "ddt_bias"]:
        np.testing.assert_allclose(got[n], ref[n], rtol=1e-10, atol=1e-12, err_msg=n)
    np.testing.assert_allclose(got["derase"].sum(-1) + got["dwrite"].sum(-1), ref["dbeta"],
                               rtol=1e-10, atol=1e-12)


def test_forward_and_backward_match_autograd_of_explicit_form():
    p = rand_problem([4, 6, 1], H=2, D=5, seed=13)
    rng = np.random.default_rng(14)
    h0 = rng.standard_normal((3, 2, 5, 5)) * 0.5
    dht = rng.standard_normal((3, 2, 5, 5)) * 0.5
    t = {n: torch.tensor(p[n], dtype=torch.float64, requires_grad=True) for n in NAMES}
    th0 = torch.tensor(h0, requires_grad=True)
    fin = []
    o = explicit_forward_gdn2(t["q"], t["k"], t["v"], t["g"], t["erase"], t["write"], t["A_log"],
                              t["dt_bias"], p["cu_seqlens"], scale=0.7, h0=th0, final_states=fin)
    loss = (o * torch.tensor(p["dO"])).sum() + (fin[0] * torch.tensor(dht)).sum()
    loss.backward()
    out = run(p, scale=0.7, h0=h0, dht=dht)
    np.testing.assert_allclose(out["o"], o.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["hT"], fin[0].detach().numpy(), rtol=1e-11, atol=1e-12)
    for iname, gname in GRADS.items():
        np.testing.assert_allclose(out[gname], t[iname].grad.numpy(), rtol=1e-9, atol=1e-11,
                                   err_msg=gname)
    np.testing.assert_allclose(out["dh0"], th0.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_backward_matches_central_finite_differences():
    p = rand_problem([3, 5], H=2, D=4, seed=15)
    out = run(p)
    h = 1e-6

    def loss(pp):
        return float((run(pp, dO=False)["o"] * pp["dO"]).sum())

    for iname, gname in GRADS.items():
        x = p[iname]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            pp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
            pp[iname][idx] += h
            lp = loss(pp)
            pp[iname][idx] -= 2 * h
            lm = loss(pp)
            fd[idx] = (lp - lm) / (2 * h)
        an = out[gname]
        scale = np.abs(an).max() + 1e-3
        assert np.abs(fd - an).max() <= 1e-6 * scale, (gname, np.abs(fd - an).max(), scale)


def _normalise(x, eps=1e-6):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def test_no_erasing_is_gated_linear_attention_with_a_write_gate():
    # erase gate 0: S_t = Diag(alpha_t) S_{t-1} + k_t (w_t * v_t)^T, so
    # o_t = sum_{s<=t} sum_i q_t[i] (prod_{u=s+1..t} alpha_u[i]) k_s[i] (w_s * v_s)
    p = rand_problem([7], H=2, D=6, seed=16)
    p["erase"][:] = -1e4
    out = run(p, dO=False)["o"]
    qh, kh = _normalise(p["q"]), _normalise(p["k"])
    z = np.exp(p["A_log"])[None, :, None] * (p["g"] + p["dt_bias"][None])
    alpha = np.exp(-5.0 * expit(z))
    wv = expit(p["write"]) * p["v"]
    ref = np.zeros_like(out)
    for t in range(7):
        for s in range(t + 1):
            decay = np.prod(alpha[s + 1:t + 1], axis=0) if t > s else np.ones((2, 6))
            ref[t] += ((qh[t] * decay * kh[s]).sum(-1))[:, None] * wv[s]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_no_writing_gives_zero_output_and_gradients():
    p = rand_problem([5, 2], H=2, D=4, seed=17)
    p["write"][:] = -1e4  # sigmoid -> exactly 0 in double
    out = run(p)
    for name in ["o", "dq", "dk", "dv", "dg", "derase", "dwrite", "dA_log", "ddt_bias"]:
        assert np.all(out[name] == 0.0), name
