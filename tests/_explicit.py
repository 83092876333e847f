"""Independent brute-force forms used to pin the oracle (test-only helpers).

``explicit_forward`` evaluates the KDA recurrence literally as written in the
operator definition, with explicit D x D transition matrices:
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = S_t^T q_t,
in torch float64, so autograd through it gives an independent backward. It is
O(T D^3) and only meant for tiny shapes.
"""
import torch


def prologue(q, k, g, b, A_log, dt_bias, scale, lower, eps):
    qh = scale * q / torch.sqrt((q * q).sum(-1, keepdim=True) + eps)
    kh = k / torch.sqrt((k * k).sum(-1, keepdim=True) + eps)
    z = torch.exp(A_log)[None, :, None] * (g + dt_bias[None])
    alpha = torch.exp(lower * torch.sigmoid(z))
    beta = torch.sigmoid(b)
    return qh, kh, alpha, beta


def explicit_forward(q, k, v, g, b, A_log, dt_bias, cu, scale=1.0, lower=-5.0, eps=1e-6,
                     h0=None, final_states=None):
    """o [S,H,D]. h0 [N,H,D,D] (rows: key index) starts each recurrence
    (zero when None); when ``final_states`` is a list, the final states are
    appended to it as one [N,H,D,D] tensor."""
    S_, H, D = q.shape
    qh, kh, alpha, beta = prologue(q, k, g, b, A_log, dt_bias, scale, lower, eps)
    eye = torch.eye(D, dtype=q.dtype)
    outs = []
    finals = []
    cu = [int(x) for x in cu]
    for n in range(len(cu) - 1):
        for_heads = []
        fin_heads = []
        for h in range(H):
            S = torch.zeros(D, D, dtype=q.dtype) if h0 is None else h0[n, h]
            os_ = []
            for t in range(cu[n], cu[n + 1]):
                kk = kh[t, h][:, None]
                B = (eye - beta[t, h] * kk @ kk.T) @ torch.diag(alpha[t, h])
                S = B @ S + beta[t, h] * kk @ v[t, h][None, :]
                os_.append(S.T @ qh[t, h])
            for_heads.append(torch.stack(os_) if os_ else torch.zeros(0, D, dtype=q.dtype))
            fin_heads.append(S)
        outs.append(torch.stack(for_heads, 1))
        finals.append(torch.stack(fin_heads, 0))
    if final_states is not None:
        final_states.append(torch.stack(finals, 0))
    return torch.cat(outs, 0)


def explicit_forward_gdn2(q, k, v, g, erase, write, A_log, dt_bias, cu, scale=1.0, lower=-5.0,
                          eps=1e-6, h0=None, final_states=None):
    """GDN-2 written literally with explicit D x D transition matrices:
        S_t = (I - k_t (b_t * k_t)^T) Diag(exp g_t) S_{t-1} + k_t (w_t * v_t)^T,
        o_t = S_t^T q_t,
    with the channel-wise erase gate b = sigmoid(erase) on key channels and
    write gate w = sigmoid(write) on value channels (torch float64; tiny
    shapes only). Arguments as in ``explicit_forward``."""
    S_, H, D = q.shape
    qh, kh, alpha, _ = prologue(q, k, g, torch.zeros(S_, H, dtype=q.dtype), A_log, dt_bias, scale,
                                lower, eps)
    be, wg = torch.sigmoid(erase), torch.sigmoid(write)
    eye = torch.eye(D, dtype=q.dtype)
    outs, finals = [], []
    cu = [int(x) for x in cu]
    for n in range(len(cu) - 1):
        for_heads, fin_heads = [], []
        for h in range(H):
            S = torch.zeros(D, D, dtype=q.dtype) if h0 is None else h0[n, h]
            os_ = []
            for t in range(cu[n], cu[n + 1]):
                kk = kh[t, h][:, None]
                B = (eye - kk @ (be[t, h][:, None] * kk).T) @ torch.diag(alpha[t, h])
                S = B @ S + kk @ (wg[t, h] * v[t, h])[None, :]
                os_.append(S.T @ qh[t, h])
            for_heads.append(torch.stack(os_) if os_ else torch.zeros(0, D, dtype=q.dtype))
            fin_heads.append(S)
        outs.append(torch.stack(for_heads, 1))
        finals.append(torch.stack(fin_heads, 0))
    if final_states is not None:
        final_states.append(torch.stack(finals, 0))
    return torch.cat(outs, 0)
