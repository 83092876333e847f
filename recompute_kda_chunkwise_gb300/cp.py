"""Context parallelism: sequences cut in time, joined by the affine state prefix.

The recurrence is linear in its state, so for fixed inputs a piece of a
sequence maps its start state H to its end state as A H + B, with A the
piece's final state when it runs from the identity state with zero values
and B its final state when it runs from zero. Backwards, a piece's
start-state gradient is A^T (end-state gradient) + C, with C the initial-state
gradient of the piece's own backward from a zero end-state gradient. Given
every piece's map, ``kda_state_prefix`` (include/kda.h) gives each piece its
true start state or end-state gradient, and the pieces then run
independently. Every product runs in the CUDA library: this module only
cuts token ranges, allocates buffers, calls the C ABI in order and, across
ranks, gathers the maps.

Two forms:
* ``kda_fwd_pieces`` / ``kda_bwd_pieces`` (and ``gdn2_fwd_pieces`` /
  ``gdn2_bwd_pieces``): one GPU, each sequence cut into P pieces that run as
  P packed sequences of one launch (the split is checked against the
  whole-sequence oracle in the tests). GDN-2's recurrence is affine in its
  state in the same way; with zero values its write term vanishes, so its
  pieces' transitions come out of the same runs.
* ``kda_fwd_cp`` / ``kda_bwd_cp``: one piece of every sequence per rank of a
  ``torch.distributed`` group (rank r holds piece r); the maps are
  all-gathered, which is the split's one exchange step. ``fwd`` / ``bwd`` /
  ``prefix`` / ``gather`` are the library calls by default; the CPU tests of
  the exchange protocol substitute host versions for them.

The pages measure no such split: the page "KDA Memory with Recompute: FLA
vs cuDNN Frontend FROST", section "Measured peak allocated memory", leaves
every 256K-token case unmeasured, which are the lengths that call for it.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import kda as K


def piece_lengths(lengths, pieces: int):
    """Token counts of the pieces, sequence-major: sequence n of length T is
    cut into ``pieces`` contiguous pieces, the first T % pieces of them one
    token longer."""
    if pieces < 1:
        raise ValueError("pieces must be >= 1")
    out = []
    for T in lengths:
        base, extra = divmod(int(T), pieces)
        out.extend(base + (1 if p < extra else 0) for p in range(pieces))
    return out


def _cu(lengths, device):
    cu = [0]
    for T in lengths:
        cu.append(cu[-1] + int(T))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def _identity_states(count, H, D, device):
    return torch.eye(D, dtype=torch.float32, device=device).expand(count, H, D, D).contiguous()


@dataclass
class PiecesContext:
    """What the forward of a split problem hands its backward: the piece
    boundaries, every piece's transition A (to propagate state gradients)
    and the checkpoints of the pieces' forward."""
    pieces: int
    cu: torch.Tensor          # [N * P + 1] piece boundaries (device)
    A: torch.Tensor           # [N, P, H, D, D] piece transitions
    ctx: torch.Tensor         # ctx of the pieces' forward
    has_h0: bool


def _fwd_pieces(fwd, q, k, v, g, gates, A_log, dt_bias, lengths, pieces, h0, kw):
    N, P = len(lengths), int(pieces)
    S, H, D = q.shape
    cu = _cu(piece_lengths(lengths, P), q.device)
    # 1. every piece's map: transition (identity start, zero values) and offset (zero start)
    _, _, A = fwd(q, k, torch.zeros_like(v), g, *gates, A_log, dt_bias, cu, save_ctx=False,
                  h0=_identity_states(N * P, H, D, q.device), final_state=True, **kw)
    _, _, B = fwd(q, k, v, g, *gates, A_log, dt_bias, cu, save_ctx=False, final_state=True, **kw)
    # 2. the prefix: each piece's true start state, and the sequences' final states
    starts, hT = K.state_prefix(A.view(N, P, H, D, D), B.view(N, P, H, D, D), h0,
                                direction=K.KDA_PREFIX_FORWARD, layout="seq_major")
    # 3. the pieces from their true start states
    o, ctx = fwd(q, k, v, g, *gates, A_log, dt_bias, cu, h0=starts.view(N * P, H, D, D), **kw)
    return o, hT, PiecesContext(P, cu, A.view(N, P, H, D, D), ctx, h0 is not None)


def _bwd_pieces(bwd, q, k, v, g, gates, A_log, dt_bias, dO, pctx, dht, kw):
    N, P, H, D = pctx.A.shape[0], pctx.pieces, q.shape[1], q.shape[2]
    # 1. every piece's own start-state gradient (zero end-state gradient)
    C = bwd(q, k, v, g, *gates, A_log, dt_bias, pctx.cu, dO, pctx.ctx, want_dh0=True, **kw)["dh0"]
    # 2. the prefix backwards: each piece's true end-state gradient, and dh0
    ends, dh0 = K.state_prefix(pctx.A, C.view(N, P, H, D, D), dht, direction=K.KDA_PREFIX_BACKWARD,
                               layout="seq_major")
    # 3. the pieces' backward from their true end-state gradients
    r = bwd(q, k, v, g, *gates, A_log, dt_bias, pctx.cu, dO, pctx.ctx, dht=ends.view(N * P, H, D, D), **kw)
    r["dh0"] = dh0
    return r


def kda_fwd_pieces(q, k, v, g, beta, A_log, dt_bias, lengths, pieces: int, *, h0=None,
                   scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6):
    """Forward of N packed sequences (token counts ``lengths``), each cut
    into ``pieces`` pieces that run as independent sequences after the
    affine state prefix has given every piece its start state. Returns
    (o, hT, PiecesContext); hT [N, H, D, D] are the sequences' final states."""
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    return _fwd_pieces(K.kda_fwd, q, k, v, g, (beta,), A_log, dt_bias, lengths, pieces, h0, kw)


def kda_bwd_pieces(q, k, v, g, beta, A_log, dt_bias, dO, pctx: PiecesContext, *, dht=None,
                   scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6):
    """Backward matching ``kda_fwd_pieces``. Returns the dict of kda_bwd
    (dq, dk, dv, dg, dbeta, dA_log, ddt_bias) plus dh0 [N, H, D, D], the
    gradient of the sequences' initial states."""
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    return _bwd_pieces(K.kda_bwd, q, k, v, g, (beta,), A_log, dt_bias, dO, pctx, dht, kw)


def gdn2_fwd_pieces(q, k, v, g, erase, write, A_log, dt_bias, lengths, pieces: int, *, h0=None,
                    scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6):
    """``kda_fwd_pieces`` for GDN-2 (channel-wise erase and write gates, as in
    kda.gdn2_fwd)."""
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    return _fwd_pieces(K.gdn2_fwd, q, k, v, g, (erase, write), A_log, dt_bias, lengths, pieces, h0, kw)


def gdn2_bwd_pieces(q, k, v, g, erase, write, A_log, dt_bias, dO, pctx: PiecesContext, *, dht=None,
                    scale: float = 1.0, lower_bound: float = -5.0, eps: float = 1e-6):
    """Backward matching ``gdn2_fwd_pieces``: the dict of kda.gdn2_bwd plus
    dh0."""
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    return _bwd_pieces(K.gdn2_bwd, q, k, v, g, (erase, write), A_log, dt_bias, dO, pctx, dht, kw)


# ---- one piece per rank ----------------------------------------------------


def _gather_default(x, group):
    """[world, *x.shape]: every rank's x, in rank order (the split's one
    exchange: a piece's map, D x D per sequence and head)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x.contiguous(), group=group)
    return torch.stack(parts)


def _prefix_default(A_all, B_all, x0, direction):
    return K.state_prefix(A_all, B_all, x0, direction=direction, layout="piece_major")


def _gates(inp):
    """The problem's gate tensors and its entry points: GDN-2's erase and
    write gates when ``inp`` has them, else KDA's beta."""
    if "erase" in inp:
        return (inp["erase"], inp["write"]), K.gdn2_fwd, K.gdn2_bwd
    return (inp["beta"],), K.kda_fwd, K.kda_bwd


def _fwd_default(inp, h0, zero_values, kw):
    """This rank's piece forward: (o, ctx, hT); with zero_values the piece
    runs with v = 0 and no ctx (its transition)."""
    gates, fwd, _ = _gates(inp)
    v = torch.zeros_like(inp["v"]) if zero_values else inp["v"]
    r = fwd(inp["q"], inp["k"], v, inp["g"], *gates, inp["A_log"], inp["dt_bias"],
            inp["cu_seqlens"], save_ctx=not zero_values, h0=h0, final_state=True, **kw)
    return r[0], r[1], r[2]


def _bwd_default(inp, ctx, dht, kw):
    gates, _, bwd = _gates(inp)
    return bwd(inp["q"], inp["k"], inp["v"], inp["g"], *gates, inp["A_log"], inp["dt_bias"],
               inp["cu_seqlens"], inp["dO"], ctx, dht=dht, want_dh0=True, **kw)


def kda_fwd_cp(inp: dict, group=None, *, h0=None, scale: float = 1.0, lower_bound: float = -5.0,
               eps: float = 1e-6, fwd=_fwd_default, prefix=_prefix_default, gather=_gather_default,
               identity=None):
    """Forward with one piece of every sequence on each rank of ``group``
    (rank r holds piece r: the r-th contiguous token range of each of the N
    sequences, packed with its own cu_seqlens in ``inp``; GDN-2 when ``inp``
    holds "erase" and "write" instead of "beta"). h0 [N, H, D, D]
    is the sequences' initial state (the same tensor on every rank, or
    None). Returns (o, ctx, state) where state carries the gathered
    transitions for the backward and the sequences' final states."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    N = inp["cu_seqlens"].numel() - 1
    H, D = inp["q"].shape[1], inp["q"].shape[2]
    eye = identity if identity is not None else _identity_states(N, H, D, inp["q"].device)
    _, _, A = fwd(inp, eye, True, kw)          # transition of this rank's piece
    _, _, B = fwd(inp, None, False, kw)[:3]    # offset: from zero, with its values
    A_all, B_all = gather(A, group), gather(B, group)
    starts, hT = prefix(A_all, B_all, h0, K.KDA_PREFIX_FORWARD)
    o, ctx, _ = fwd(inp, starts[rank].contiguous(), False, kw)
    return o, ctx, {"A_all": A_all, "hT": hT}


def kda_bwd_cp(inp: dict, ctx, state: dict, group=None, *, dht=None, scale: float = 1.0,
               lower_bound: float = -5.0, eps: float = 1e-6, bwd=_bwd_default, prefix=_prefix_default,
               gather=_gather_default):
    """Backward matching ``kda_fwd_cp``: returns this rank's gradients (the
    parameter gradients dA_log / ddt_bias are this rank's share; their sum
    over ranks is the total) and dh0, the gradient of the sequences' initial
    states (the same on every rank)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    kw = dict(scale=scale, lower_bound=lower_bound, eps=eps)
    C = bwd(inp, ctx, None, kw)["dh0"]          # this piece's own start-state gradient
    C_all = gather(C, group)
    ends, dh0 = prefix(state["A_all"], C_all, dht, K.KDA_PREFIX_BACKWARD)
    r = bwd(inp, ctx, ends[rank].contiguous(), kw)
    r["dh0"] = dh0
    return r
