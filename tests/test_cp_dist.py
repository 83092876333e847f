"""The context-parallel exchange protocol on CPU (gloo, world_size 2): each
rank holds one piece of every sequence, runs kda_fwd_cp / kda_bwd_cp (the
same host code the GPU ranks run: map, all-gather, prefix, piece run) with
the fp64 oracle standing in for the piece runs and a float64 loop for the
prefix, and the assembled result must equal the oracle on the whole
sequences. This checks the gather order, the index each rank takes and the
prefix directions; the CUDA prefix kernel itself is checked on the GPU."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_fwd(inp, h0, zero_values, kw):
    import oracle
    v = torch.zeros_like(inp["v"]) if zero_values else inp["v"]
    r = oracle.kda_reference(inp["q"], inp["k"], v, inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
                             inp["cu_seqlens"], h0=h0, want_state=True, **kw)
    # the piece's "ctx" is its start state: the oracle's backward re-runs from it
    return torch.from_numpy(r["o"]), h0, torch.from_numpy(r["hT"])


def _oracle_bwd(inp, ctx, dht, kw):
    import oracle
    r = oracle.kda_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
                             inp["cu_seqlens"], inp["dO"], h0=ctx, dht=dht, want_state=True, **kw)
    return {n: torch.from_numpy(x) for n, x in r.items()}


def _prefix64(A_all, B_all, x0, direction):
    """x_{p+1} = A_p x_p + B_p (forward) / x_{p-1} = A_p^T x_p + B_p
    (backward) over [P, N, H, D, D] maps, in float64."""
    A, B = A_all.double(), B_all.double()
    P = A.shape[0]
    x = torch.zeros_like(A[0]) if x0 is None else x0.double()
    xs = torch.empty_like(A)
    order = range(P) if direction == 0 else range(P - 1, -1, -1)
    for p in order:
        xs[p] = x
        M = A[p] if direction == 0 else A[p].transpose(-1, -2)
        x = M @ x + B[p]
    return xs, x


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from recompute_kda_chunkwise_gb300 import Workload, make_inputs, make_states
    from recompute_kda_chunkwise_gb300 import cp as CP
    lengths = (37, 70, 11)
    w = Workload("cp_dist", lengths, 2, 8, "f32", seed=8500, param_std=0.5, scale=8 ** -0.5,
                 gate_mean=-3.0)
    full = make_inputs(w)
    st = make_states(w)
    # this rank's piece of every sequence, packed with its own boundaries
    pl = CP.piece_lengths(lengths, world)
    cu = np.cumsum([0] + list(lengths))
    rows, mine = [], []
    for n in range(len(lengths)):
        start = int(cu[n]) + sum(pl[n * world:n * world + rank])
        rows.append(torch.arange(start, start + pl[n * world + rank]))
        mine.append(pl[n * world + rank])
    idx = torch.cat(rows)
    inp = {n: full[n][idx] for n in ("q", "k", "v", "g", "beta", "dO")}
    inp.update(A_log=full["A_log"], dt_bias=full["dt_bias"],
               cu_seqlens=torch.tensor(np.cumsum([0] + mine), dtype=torch.int32))
    kw = dict(scale=w.scale)
    eye = torch.eye(w.D, dtype=torch.float64).expand(len(lengths), w.H, w.D, w.D).contiguous()
    o, ctx, state = CP.kda_fwd_cp(inp, h0=st["h0"].double(), fwd=_oracle_fwd, prefix=_prefix64,
                                  identity=eye, **kw)
    r = CP.kda_bwd_cp(inp, ctx, state, dht=st["dht"].double(), bwd=_oracle_bwd, prefix=_prefix64, **kw)
    res = {"idx": idx, "o": o}
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        res[n] = r[n]
    for n in ("dA_log", "ddt_bias"):  # each rank's share; the total is the sum over ranks
        t = r[n].clone()
        dist.all_reduce(t)
        res[n] = t
    res["dh0"], res["hT"] = r["dh0"], state["hT"]
    out.put((rank, {k: v.numpy() for k, v in res.items()}))
    dist.destroy_process_group()


def test_cp_protocol_two_ranks_matches_the_whole_sequence():
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from recompute_kda_chunkwise_gb300 import Workload, make_inputs, make_states
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    lengths = (37, 70, 11)
    w = Workload("cp_dist", lengths, 2, 8, "f32", seed=8500, param_std=0.5, scale=8 ** -0.5, gate_mean=-3.0)
    full = make_inputs(w)
    st = make_states(w)
    ref = oracle.kda_reference(full["q"], full["k"], full["v"], full["g"], full["beta"], full["A_log"],
                               full["dt_bias"], full["cu_seqlens"], full["dO"], scale=w.scale,
                               h0=st["h0"], dht=st["dht"])
    for n in ("o", "dq", "dk", "dv", "dg", "dbeta"):
        x = np.zeros_like(ref[n])
        for rank in (0, 1):
            x[got[rank]["idx"]] = got[rank][n]
        np.testing.assert_allclose(x, ref[n], rtol=1e-9, atol=1e-10, err_msg=n)
    for rank in (0, 1):
        for n in ("dA_log", "ddt_bias", "dh0", "hT"):
            np.testing.assert_allclose(got[rank][n], ref[n], rtol=1e-9, atol=1e-10, err_msg=n)


def test_piece_lengths_cover_each_sequence_in_order():
    # every sequence's tokens, cut into contiguous pieces sequence-major; the
    # first T % P pieces take one token more, and empty pieces are allowed
    import pytest
    from recompute_kda_chunkwise_gb300 import cp as CP
    assert CP.piece_lengths([10, 3, 0], 4) == [3, 3, 2, 2, 1, 1, 1, 0, 0, 0, 0, 0]
    assert CP.piece_lengths([7], 1) == [7]
    for lengths, P in [([1029, 700, 2049, 3], 5), ([131072], 2), ([1], 3)]:
        pl = CP.piece_lengths(lengths, P)
        assert len(pl) == len(lengths) * P
        assert [sum(pl[n * P:(n + 1) * P]) for n in range(len(lengths))] == list(lengths)
        assert all(max(pl[n * P:(n + 1) * P]) - min(pl[n * P:(n + 1) * P]) <= 1 for n in range(len(lengths)))
    with pytest.raises(ValueError):
        CP.piece_lengths([4], 0)
