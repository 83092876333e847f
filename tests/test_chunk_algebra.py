"""The chunked algebra the CUDA kernels evaluate, checked in float64 against
the oracle's token recurrence (CPU only).

Per chunk of C tokens, with G the chunk-local inclusive cumulative log-decay
(Gamma = e^G, gamma = Gamma_{C-1}), H the chunk-start state and the gates
written per channel (Be on key channels, Wr on value channels; KDA is
Be = Wr = beta on every channel):
    Xw = Be*Kh*Gamma,  Xu = Wr*V,  Ki = Kh/Gamma,  Kbar = Kh*gamma/Gamma
    Abar = tril(Xw Ki^T, -1),  M = tril((Qh*Gamma) Ki^T),  T = (I + Abar)^-1
    W = T Xw,  U = T Xu,  U~ = U - W H,  O = (Qh*Gamma) H + M U~
    H' = diag(gamma) H + Kbar^T U~
and the backward
    dU~ = M^T dO + Kbar dH',  dH = diag(gamma) dH' + (Qh*Gamma)^T dO - W^T dU~
    dW = -dU~ H^T,  dT = dW Xw^T + dU~ Xu^T,  dA = -T^T dT T^T (strictly lower)
    dXw = T^T dW + dA Ki,  dXu = T^T dU~,  dKi = dA^T Xw,
followed by the elementwise chain rules. This is the decomposition of the
op table in "KDA at the production shape ...", section 2.1. A slip in any
term shows up here as a mismatch with the token recurrence, before any GPU
runs. The test shares no code with the CUDA library or the oracle.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle


def _problem(lengths, H, D, seed, channel):
    rng = np.random.default_rng(seed)
    S = int(sum(lengths))
    p = {n: rng.standard_normal((S, H, D)) for n in ["q", "k", "v", "g", "dO"]}
    if channel:
        p["erase"] = rng.standard_normal((S, H, D))
        p["write"] = rng.standard_normal((S, H, D))
    else:
        p["beta"] = rng.standard_normal((S, H))
    p["A_log"] = rng.standard_normal(H) * 0.3
    p["dt_bias"] = rng.standard_normal((H, D)) * 0.3
    p["cu"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return p


def _chunked(p, C, scale, lower=-5.0, eps=1e-6):
    """Chunked forward + backward of every (sequence, head); returns the
    oracle's output names."""
    S, H, D = p["q"].shape
    channel = "erase" in p
    out = {n: np.zeros((S, H, D)) for n in ["o", "dq", "dk", "dv", "dg"]}
    if channel:
        out["derase"] = np.zeros((S, H, D))
        out["dwrite"] = np.zeros((S, H, D))
    else:
        out["dbeta"] = np.zeros((S, H))
    out["dA_log"] = np.zeros(H)
    out["ddt_bias"] = np.zeros((H, D))
    cu = p["cu"]
    for n in range(len(cu) - 1):
        bos, T = int(cu[n]), int(cu[n + 1] - cu[n])
        if T == 0:
            continue
        for h in range(H):
            eA = np.exp(p["A_log"][h])

            def prologue(t0, rows):
                sl = slice(bos + t0, bos + t0 + rows)
                pad = lambda x: np.concatenate([x, np.zeros((C - rows,) + x.shape[1:])])
                q, k, v = pad(p["q"][sl, h]), pad(p["k"][sl, h]), pad(p["v"][sl, h])
                nq = np.sqrt((q * q).sum(1) + eps)
                nk = np.sqrt((k * k).sum(1) + eps)
                z = eA * (pad(p["g"][sl, h]) + p["dt_bias"][h])
                sg = expit(z)
                gl = lower * sg * (np.arange(C) < rows)[:, None]
                if channel:
                    Be = pad(expit(p["erase"][sl, h]))
                    Wr = pad(expit(p["write"][sl, h]))
                else:
                    b = pad(expit(p["beta"][sl, h])[:, None])
                    Be, Wr = np.repeat(b, D, 1), np.repeat(b, D, 1)
                c = dict(xq=q / nq[:, None], xk=k / nk[:, None], nq=nq, nk=nk, V=v, z=z, sg=sg, Be=Be, Wr=Wr,
                         rows=rows, t0=t0)
                G = np.cumsum(gl, 0)
                c["G"], c["gam"] = G, np.exp(G[-1])
                c["Qg"] = scale * c["xq"] * np.exp(G)
                c["Kg"] = c["xk"] * np.exp(G)
                c["Ki"] = c["xk"] * np.exp(-G)
                c["Kb"] = c["xk"] * np.exp(G[-1] - G)
                c["Xw"], c["Xu"] = Be * c["Kg"], Wr * v
                c["Abar"] = np.tril(c["Xw"] @ c["Ki"].T, -1)
                c["M"] = np.tril(c["Qg"] @ c["Ki"].T)
                c["T"] = np.linalg.inv(np.eye(C) + c["Abar"])
                c["W"], c["U"] = c["T"] @ c["Xw"], c["T"] @ c["Xu"]
                return c

            nch = (T + C - 1) // C
            Hs, Hst = [], np.zeros((D, D))
            for ci in range(nch):
                t0 = ci * C
                c = prologue(t0, min(C, T - t0))
                Hs.append(Hst)
                Ut = c["U"] - c["W"] @ Hst
                o = c["Qg"] @ Hst + c["M"] @ Ut
                out["o"][bos + t0:bos + t0 + c["rows"], h] = o[:c["rows"]]
                Hst = c["gam"][:, None] * Hst + c["Kb"].T @ Ut
            dH = np.zeros((D, D))
            for ci in reversed(range(nch)):
                t0 = ci * C
                c = prologue(t0, min(C, T - t0))
                rows, Hc = c["rows"], Hs[ci]
                Ut = c["U"] - c["W"] @ Hc
                dO = np.zeros((C, D))
                dO[:rows] = p["dO"][bos + t0:bos + t0 + rows, h]
                dUt = c["M"].T @ dO + c["Kb"] @ dH
                dQg = dO @ Hc.T
                dKb = Ut @ dH.T
                dgam = (Hc * dH).sum(1)
                dW = -dUt @ Hc.T
                dH = c["gam"][:, None] * dH + c["Qg"].T @ dO - c["W"].T @ dUt
                dM = np.tril(dO @ Ut.T)
                dT = np.tril(dW @ c["Xw"].T + dUt @ c["Xu"].T, -1)
                dA = np.tril(-(c["T"].T @ dT @ c["T"].T), -1)
                dXw = c["T"].T @ dW + dA @ c["Ki"]
                dXu = c["T"].T @ dUt
                dKi = dA.T @ c["Xw"] + dM.T @ c["Qg"]
                dQg = dQg + dM @ c["Ki"]
                dKg = c["Be"] * dXw
                # gradients w.r.t. the unit-norm rows and the cumulative log-decay
                e, ei, eb = np.exp(c["G"]), np.exp(-c["G"]), np.exp(c["G"][-1] - c["G"])
                dxq = scale * dQg * e
                dxk = dKg * e + dKi * ei + dKb * eb
                dG = dQg * c["Qg"] + dKg * c["Kg"] - dKi * c["Ki"] - dKb * c["Kb"]
                dGe = (dKb * c["Kb"]).sum(0) + dgam * c["gam"]
                dg = np.cumsum(dG[::-1], 0)[::-1] + dGe
                sl = slice(bos + t0, bos + t0 + rows)
                xq, xk = c["xq"], c["xk"]
                out["dq"][sl, h] = ((dxq - xq * (xq * dxq).sum(1, keepdims=True)) / c["nq"][:, None])[:rows]
                out["dk"][sl, h] = ((dxk - xk * (xk * dxk).sum(1, keepdims=True)) / c["nk"][:, None])[:rows]
                dz = dg * lower * c["sg"] * (1 - c["sg"])
                out["dg"][sl, h] = (eA * dz)[:rows]
                out["ddt_bias"][h] += (eA * dz)[:rows].sum(0)
                out["dA_log"][h] += (dz * c["z"])[:rows].sum()
                dBe, dWr = c["Kg"] * dXw, c["V"] * dXu
                out["dv"][sl, h] = (c["Wr"] * dXu)[:rows]
                if channel:
                    out["derase"][sl, h] = (dBe * c["Be"] * (1 - c["Be"]))[:rows]
                    out["dwrite"][sl, h] = (dWr * c["Wr"] * (1 - c["Wr"]))[:rows]
                else:
                    beta = c["Be"][:, 0]
                    dbeta = dBe.sum(1) + dWr.sum(1)
                    out["dbeta"][sl, h] = (dbeta * beta * (1 - beta))[:rows]
    return out


@pytest.mark.parametrize("channel", [False, True])
@pytest.mark.parametrize("C", [8, 16, 64])
def test_chunked_algebra_matches_the_token_recurrence(channel, C):
    p = _problem([1, 37, 0, 70], H=2, D=8, seed=100 + C, channel=channel)
    got = _chunked(p, C, scale=0.6)
    args = [p["q"], p["k"], p["v"], p["g"]]
    args += [p["erase"], p["write"]] if channel else [p["beta"]]
    run = oracle.gdn2_reference if channel else oracle.kda_reference
    ref = run(*args, p["A_log"], p["dt_bias"], p["cu"], p["dO"], scale=0.6)
    for name, val in got.items():
        np.testing.assert_allclose(val, ref[name], rtol=1e-9, atol=1e-11, err_msg=name)
