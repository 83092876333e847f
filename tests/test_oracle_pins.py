"""Pins for the fp64 oracle, checked against things other than itself.

* explicit_forward: the recurrence as written with explicit D x D transition
  matrices (a different evaluation order and formula than the oracle's
  rank-one form);
* torch float64 autograd through that explicit form (independent backward);
* central finite differences of the oracle's own forward (backward <-> forward);
* closed forms: beta = 0, single token with no decay, length-1 sequences,
  the delta rule's overwrite property, one-hot keys (gated linear attention
  with per-channel decay), zero rows;
* invariants: scale invariance of the L2 norm, linearity in v / scale / dO,
  packing, head independence, the A_log / dt_bias chain-rule identities.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from tests._explicit import explicit_forward

RNG = np.random.default_rng(1234)


def rand_problem(lengths, H, D, param_std=0.5, gate_mean=0.0, seed=0):
    rng = np.random.default_rng(seed)
    S = int(sum(lengths))
    p = dict(
        q=rng.standard_normal((S, H, D)), k=rng.standard_normal((S, H, D)),
        v=rng.standard_normal((S, H, D)),
        g=rng.standard_normal((S, H, D)) + gate_mean,
        beta=rng.standard_normal((S, H)),
        A_log=rng.standard_normal(H) * param_std, dt_bias=rng.standard_normal((H, D)) * param_std,
        dO=rng.standard_normal((S, H, D)),
    )
    p["cu_seqlens"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return p


def run(p, dO=True, **kw):
    return oracle.kda_reference(p["q"], p["k"], p["v"], p["g"], p["beta"], p["A_log"],
                                p["dt_bias"], p["cu_seqlens"], p["dO"] if dO else None, **kw)


def torch_inputs(p):
    return {k: torch.tensor(v, dtype=torch.float64) for k, v in p.items() if k != "cu_seqlens"}


@pytest.mark.parametrize("scale", [1.0, 0.125])
def test_forward_matches_explicit_transition_matrices(scale):
    p = rand_problem([5, 1, 7], H=2, D=6, seed=1)
    t = torch_inputs(p)
    ref = explicit_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                           p["cu_seqlens"], scale=scale).numpy()
    out = run(p, dO=False, scale=scale)["o"]
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_backward_matches_autograd_of_explicit_form():
    p = rand_problem([4, 6], H=2, D=5, seed=2)
    t = torch_inputs(p)
    names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias"]
    for n in names:
        t[n].requires_grad_(True)
    o = explicit_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                         p["cu_seqlens"], scale=0.7)
    (o * t["dO"]).sum().backward()
    out = run(p, scale=0.7)
    pairs = dict(dq="q", dk="k", dv="v", dg="g", dbeta="beta", dA_log="A_log", ddt_bias="dt_bias")
    for gname, iname in pairs.items():
        ref = t[iname].grad.numpy()
        np.testing.assert_allclose(out[gname], ref, rtol=1e-9, atol=1e-11, err_msg=gname)


def test_backward_matches_central_finite_differences():
    p = rand_problem([3, 5], H=2, D=4, seed=3)
    out = run(p)
    h = 1e-6
    grads = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", A_log="dA_log", dt_bias="ddt_bias")

    def loss(pp):
        return float((run(pp, dO=False)["o"] * pp["dO"]).sum())

    for iname, gname in grads.items():
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


def test_beta_zero_gives_zero_output_and_gradients():
    p = rand_problem([6, 3], H=2, D=4, seed=4)
    p["beta"][:] = -1e4  # sigmoid -> exactly 0 in double
    out = run(p)
    for name in ["o", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"]:
        assert np.all(out[name] == 0.0), name


def _normalise(x, eps=1e-6):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


def test_single_token_without_decay_is_plain_delta_rule():
    p = rand_problem([1], H=3, D=8, param_std=0.0, seed=5)
    p["g"][:] = -1e4  # sigmoid(z) -> 0, so g = 0 and alpha = 1
    out = run(p, dO=False)["o"]
    qh, kh = _normalise(p["q"]), _normalise(p["k"])
    beta = expit(p["beta"])
    ref = (beta * (qh * kh).sum(-1))[..., None] * p["v"]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_length_one_sequences_reduce_to_single_steps():
    lengths = [1] * 7
    p = rand_problem(lengths, H=2, D=5, seed=6)  # any gate: S_0 = 0 so decay never acts
    out = run(p, dO=False)["o"]
    qh, kh = _normalise(p["q"]), _normalise(p["k"])
    ref = (expit(p["beta"]) * (qh * kh).sum(-1))[..., None] * p["v"]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_same_key_overwrites_state():
    # g = 0, beta = 1, one shared key: S_t = kh v_t^T exactly, o_t = (qh_t . kh) v_t
    T, D = 9, 6
    p = rand_problem([T], H=1, D=D, param_std=0.0, seed=7)
    p["g"][:] = -1e4
    p["beta"][:] = 1e4
    p["k"][:] = p["k"][0:1]
    out = run(p, dO=False, eps=0.0)["o"]  # eps = 0 so |kh| = 1 exactly
    qh, kh = _normalise(p["q"], 0.0), _normalise(p["k"], 0.0)
    ref = (qh * kh).sum(-1)[..., None] * p["v"]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("gate_mean", [0.0, 6.0])  # 6.0 pushes the gate to the -5 bound
def test_one_hot_keys_give_gated_linear_attention(gate_mean):
    # beta = 1 and orthonormal keys e_t: row t of the state is overwritten by
    # v_t and then decays channel-wise, so
    #   o_t = sum_{s<=t} qh_t[s] * prod_{u=s+1..t} alpha_u[s] * v_s
    T, D, H = 6, 8, 2
    p = rand_problem([T], H=H, D=D, gate_mean=gate_mean, seed=8)
    p["beta"][:] = 1e4
    p["k"][:] = 0
    for t in range(T):
        p["k"][t, :, t] = 3.0  # any positive multiple normalises to e_t
    eps = 0.0
    out = run(p, dO=False, eps=eps)["o"]
    qh = _normalise(p["q"], eps)
    z = np.exp(p["A_log"])[None, :, None] * (p["g"] + p["dt_bias"][None])
    alpha = np.exp(-5.0 * expit(z))
    ref = np.zeros_like(out)
    for h in range(H):
        for t in range(T):
            for s in range(t + 1):
                decay = np.prod(alpha[s + 1:t + 1, h, s])
                ref[t, h] += qh[t, h, s] * decay * p["v"][s, h]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)
    if gate_mean > 0:
        assert alpha.min() > np.exp(-5.0) and alpha.max() < 1.0


def test_l2_norm_scale_invariance_and_output_scale_linearity():
    p = rand_problem([7, 4], H=2, D=5, seed=9)
    base = run(p, dO=False, eps=0.0)["o"]
    p2 = dict(p)
    p2["q"] = p["q"] * 3.5
    p2["k"] = p["k"] * 0.25
    np.testing.assert_allclose(run(p2, dO=False, eps=0.0)["o"], base, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(run(p, dO=False, eps=0.0, scale=0.3)["o"], 0.3 * base,
                               rtol=1e-12, atol=1e-13)


def test_linear_in_v_and_gradients_linear_in_dO():
    p = rand_problem([8], H=2, D=4, seed=10)
    a = run(p)
    p2 = dict(p)
    p2["v"] = -2.0 * p["v"]
    p2["dO"] = 0.5 * p["dO"]
    b = run(p2)
    np.testing.assert_allclose(b["o"], -2.0 * a["o"], rtol=1e-12, atol=1e-13)
    p3 = dict(p)
    p3["dO"] = 3.0 * p["dO"]
    c = run(p3)
    for n in ["dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"]:
        np.testing.assert_allclose(c[n], 3.0 * a[n], rtol=1e-11, atol=1e-12, err_msg=n)


def test_packing_and_head_independence():
    lengths = [5, 3, 6]
    p = rand_problem(lengths, H=3, D=4, seed=11)
    full = run(p)
    cu = p["cu_seqlens"]
    # each sequence alone
    for n in range(len(lengths)):
        sl = slice(cu[n], cu[n + 1])
        q = {k: (v[sl] if k in ("q", "k", "v", "g", "beta", "dO") else v) for k, v in p.items()}
        q["cu_seqlens"] = np.array([0, lengths[n]])
        part = run(q)
        for name in ["o", "dq", "dk", "dv", "dg", "dbeta"]:
            np.testing.assert_allclose(part[name], full[name][sl], rtol=1e-13, atol=1e-15)
    # each head alone, via the head-subset helper
    inp = dict(p)
    sub = oracle.kda_reference_heads(inp, [2, 0])
    for name in ["o", "dq", "dk", "dv", "dg"]:
        np.testing.assert_allclose(sub[name], full[name][:, [2, 0]], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sub["dA_log"], full["dA_log"][[2, 0]], rtol=1e-13, atol=1e-15)


def test_gate_parameter_gradients_are_sums_of_raw_gate_gradients():
    # chain rule identities of the gate's affine argument:
    #   d dt_bias[h,i] = sum_t d a[t,h,i];  d A_log[h] = sum_{t,i} d a[t,h,i]*(a+dt_bias)[t,h,i]
    p = rand_problem([6, 5], H=2, D=4, seed=12)
    out = run(p)
    np.testing.assert_allclose(out["ddt_bias"], out["dg"].sum(0), rtol=1e-12, atol=1e-14)
    ref = (out["dg"] * (p["g"] + p["dt_bias"][None])).sum((0, 2))
    np.testing.assert_allclose(out["dA_log"], ref, rtol=1e-11, atol=1e-13)


def test_zero_query_row_gives_zero_output_and_finite_gradient():
    p = rand_problem([5], H=1, D=4, seed=13)
    p["q"][2] = 0.0
    out = run(p)
    assert np.all(out["o"][2] == 0.0)
    assert np.all(np.isfinite(out["dq"]))


def test_empty_sequences_are_skipped():
    p = rand_problem([0, 4, 0, 3], H=2, D=4, seed=14)
    full = run(p)
    q = dict(p)
    q["cu_seqlens"] = np.array([0, 4, 7])
    ref = run(q)
    for name in ["o", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias"]:
        np.testing.assert_allclose(full[name], ref[name], rtol=0, atol=0)


def test_backward_across_stored_state_segments():
    # sequences longer than the oracle's 256-token state segments, so the
    # reverse loop rebuilds states from stored ones more than once
    p = rand_problem([300, 530], H=1, D=3, seed=15)
    t = torch_inputs(p)
    for n in ["q", "k", "v", "g", "beta", "A_log", "dt_bias"]:
        t[n].requires_grad_(True)
    o = explicit_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                         p["cu_seqlens"])
    (o * t["dO"]).sum().backward()
    out = run(p)
    np.testing.assert_allclose(out["o"], o.detach().numpy(), rtol=1e-10, atol=1e-12)
    pairs = dict(dq="q", dk="k", dv="v", dg="g", dbeta="beta", dA_log="A_log", ddt_bias="dt_bias")
    for gname, iname in pairs.items():
        np.testing.assert_allclose(out[gname], t[iname].grad.numpy(), rtol=1e-8, atol=1e-10,
                                   err_msg=gname)


# ---- initial state h0, final state hT and their gradients ----

def rand_states(p, seed, scale=0.5):
    rng = np.random.default_rng(seed)
    N = len(p["cu_seqlens"]) - 1
    H, D = p["q"].shape[1], p["q"].shape[2]
    return rng.standard_normal((N, H, D, D)) * scale, rng.standard_normal((N, H, D, D))


def test_final_state_and_state_gradients_match_autograd_of_explicit_form():
    p = rand_problem([4, 0, 6], H=2, D=5, seed=21)
    h0, dht = rand_states(p, 22)
    t = torch_inputs(p)
    th0 = torch.tensor(h0, requires_grad=True)
    names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias"]
    for n in names:
        t[n].requires_grad_(True)
    fin = []
    o = explicit_forward(t["q"], t["k"], t["v"], t["g"], t["beta"], t["A_log"], t["dt_bias"],
                         p["cu_seqlens"], scale=0.7, h0=th0, final_states=fin)
    ((o * t["dO"]).sum() + (fin[0] * torch.tensor(dht)).sum()).backward()
    out = run(p, scale=0.7, h0=h0, dht=dht)
    np.testing.assert_allclose(out["o"], o.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["hT"], fin[0].detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["dh0"], th0.grad.numpy(), rtol=1e-9, atol=1e-11)
    pairs = dict(dq="q", dk="k", dv="v", dg="g", dbeta="beta", dA_log="A_log", ddt_bias="dt_bias")
    for gname, iname in pairs.items():
        np.testing.assert_allclose(out[gname], t[iname].grad.numpy(), rtol=1e-9, atol=1e-11,
                                   err_msg=gname)
    # the empty sequence passes its state through, and its gradient back
    np.testing.assert_array_equal(out["hT"][1], h0[1])
    np.testing.assert_array_equal(out["dh0"][1], dht[1])


def test_splitting_a_sequence_through_its_state_changes_nothing():
    # running [0, T) equals running [0, T1) and then [T1, T) from the first
    # part's final state; in the backward the second part's dh0 is the first
    # part's dhT (the recurrence is a composition of per-token maps)
    T, T1 = 11, 4
    p = rand_problem([T], H=2, D=4, seed=23)
    h0, dht = rand_states(p, 24)
    full = run(p, h0=h0, dht=dht)

    def part(a, b):
        q = {k: (v[a:b] if k not in ("A_log", "dt_bias", "cu_seqlens") else v) for k, v in p.items()}
        q["cu_seqlens"] = np.array([0, b - a], np.int64)
        return q

    second_h0 = run(part(0, T1), dO=False, h0=h0)["hT"]
    second = run(part(T1, T), h0=second_h0, dht=dht)
    first = run(part(0, T1), h0=h0, dht=second["dh0"])
    np.testing.assert_allclose(second["hT"], full["hT"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(np.concatenate([first["o"], second["o"]]), full["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(first["dh0"], full["dh0"], rtol=1e-11, atol=1e-12)
    for g in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(np.concatenate([first[g], second[g]]), full[g], rtol=1e-11,
                                   atol=1e-12, err_msg=g)
    for g in ("dA_log", "ddt_bias"):
        np.testing.assert_allclose(first[g] + second[g], full[g], rtol=1e-11, atol=1e-12, err_msg=g)


def test_beta_zero_decays_the_initial_state_channel_by_channel():
    # beta = 0 (raw beta -> -inf): S_t = Diag(alpha_t) S_{t-1}, so
    # hT = Diag(prod_t alpha_t) h0, o_t = S_t^T qh_t, dh0 = Diag(prod alpha) dhT
    p = rand_problem([5], H=1, D=3, seed=25)
    p["beta"][:] = -1e4
    h0, dht = rand_states(p, 26)
    out = run(p, h0=h0, dht=dht, dO=False)
    z = np.exp(p["A_log"])[None, :, None] * (p["g"] + p["dt_bias"][None])
    alpha = np.exp(-5.0 * expit(z))  # [T,H,D]
    decay = alpha[:, 0].prod(0)
    np.testing.assert_allclose(out["hT"][0, 0], decay[:, None] * h0[0, 0], rtol=1e-12, atol=1e-14)
    qh = p["q"] / np.sqrt((p["q"] ** 2).sum(-1, keepdims=True) + 1e-6)
    St = h0[0, 0].copy()
    for t in range(5):
        St = alpha[t, 0][:, None] * St
        np.testing.assert_allclose(out["o"][t, 0], St.T @ qh[t, 0], rtol=1e-11, atol=1e-13)
    p["dO"][:] = 0.0
    g = run(p, h0=h0, dht=dht)
    np.testing.assert_allclose(g["dh0"][0, 0], decay[:, None] * dht[0, 0], rtol=1e-12, atol=1e-14)


def test_zero_state_arguments_match_the_stateless_run():
    p = rand_problem([3, 7], H=2, D=4, seed=27)
    N, H, D = 2, 2, 4
    z = np.zeros((N, H, D, D))
    a, b = run(p), run(p, h0=z, dht=z)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
