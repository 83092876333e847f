"""Context-parallel split on one GPU: sequences cut in time into P pieces,
joined by the affine state prefix (kda_state_prefix), checked element by
element against the fp64 oracle run on the whole sequences (o, every input
gradient, the final states and the initial-state gradient, plain bars), and
the prefix kernel alone against a float64 evaluation of its recurrence."""
import numpy as np
import pytest
import torch

import oracle
from recompute_kda_chunkwise_gb300 import Workload, make_inputs, make_states
from recompute_kda_chunkwise_gb300 import cp as CP
from recompute_kda_chunkwise_gb300 import kda as K
from tests._parity import OUT_NAMES, TOL, compare, to_dev

pytestmark = pytest.mark.gpu

ARGS = ("q", "k", "v", "g", "beta", "A_log", "dt_bias")


@pytest.mark.parametrize("dtype,D,pieces,states", [
    ("bf16", 128, 2, True), ("bf16", 128, 3, False), ("f32", 64, 3, True), ("bf16", 128, 5, True)])
def test_pieces_match_the_whole_sequence_oracle(dtype, D, pieces, states):
    # pieces cross chunk (64 / 16 tokens) and checkpoint (1024 tokens)
    # boundaries at odd offsets; one sequence is shorter than the piece count
    # allows for (3 tokens in 5 pieces: some pieces are empty)
    lengths = (1029, 700, 2049, 3) if pieces == 5 else (1029, 700, 2049)
    w = Workload(f"cp_{dtype}_d{D}_p{pieces}", lengths, 3, D, dtype, seed=8300 + D + pieces,
                 param_std=0.5, scale=D ** -0.5, gate_mean=-2.0)
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w)) if states else {"h0": None, "dht": None}
    args = [inp[n] for n in ARGS]
    o, hT, pctx = CP.kda_fwd_pieces(*args, list(lengths), pieces, h0=st["h0"], scale=w.scale)
    r = CP.kda_bwd_pieces(*args, inp["dO"], pctx, dht=st["dht"], scale=w.scale)
    torch.cuda.synchronize()
    r["o"], r["hT"] = o, hT
    cpu = {k_: (v_.cpu() if v_ is not None else None) for k_, v_ in inp.items()}
    ref = oracle.kda_reference(*[cpu[n] for n in ARGS], cpu["cu_seqlens"], cpu["dO"], scale=w.scale,
                               h0=None if st["h0"] is None else st["h0"].cpu(),
                               dht=None if st["dht"] is None else st["dht"].cpu(), want_state=True)
    compare(r, ref, TOL[inp["q"].dtype], names=OUT_NAMES + ["hT", "dh0"])


@pytest.mark.parametrize("dtype,D,pieces,states", [("bf16", 128, 3, True), ("f32", 64, 2, True)])
def test_gdn2_pieces_match_the_whole_sequence_oracle(dtype, D, pieces, states):
    # GDN-2 (channel-wise erase / write gates) cut the same way; bf16 D = 128
    # runs the tensor-core forward, fp32 D = 64 the CUDA-core kernels
    lengths = (1029, 700, 2049)
    w = Workload(f"cp_gdn2_{dtype}_d{D}_p{pieces}", lengths, 3, D, dtype, seed=8350 + D + pieces,
                 param_std=0.5, scale=D ** -0.5, gate_mean=-2.0, gates="channel")
    inp = to_dev(make_inputs(w))
    st = to_dev(make_states(w)) if states else {"h0": None, "dht": None}
    names = ("q", "k", "v", "g", "erase", "write", "A_log", "dt_bias")
    args = [inp[n] for n in names]
    o, hT, pctx = CP.gdn2_fwd_pieces(*args, list(lengths), pieces, h0=st["h0"], scale=w.scale)
    r = CP.gdn2_bwd_pieces(*args, inp["dO"], pctx, dht=st["dht"], scale=w.scale)
    torch.cuda.synchronize()
    r["o"], r["hT"] = o, hT
    cpu = {k_: (v_.cpu() if v_ is not None else None) for k_, v_ in inp.items()}
    ref = oracle.gdn2_reference(*[cpu[n] for n in names], cpu["cu_seqlens"], cpu["dO"], scale=w.scale,
                                h0=None if st["h0"] is None else st["h0"].cpu(),
                                dht=None if st["dht"] is None else st["dht"].cpu(), want_state=True)
    gnames = ["o", "dq", "dk", "dv", "dg", "derase", "dwrite", "dA_log", "ddt_bias", "hT", "dh0"]
    compare(r, ref, TOL[inp["q"].dtype], names=gnames)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("layout", ["seq_major", "piece_major"])
def test_state_prefix_kernel_against_float64(D, layout):
    N, P, H = 3, 4, 2
    gen = torch.Generator().manual_seed(8400 + D)
    shape = (N, P, H, D, D) if layout == "seq_major" else (P, N, H, D, D)
    A = torch.randn(shape, generator=gen) / D ** 0.5
    B = torch.randn(shape, generator=gen)
    x0 = torch.randn((N, H, D, D), generator=gen)
    Ad, Bd, x0d = A.double().numpy(), B.double().numpy(), x0.double().numpy()
    if layout == "piece_major":  # to [N][P] for the reference loop
        Ad, Bd = Ad.transpose(1, 0, 2, 3, 4), Bd.transpose(1, 0, 2, 3, 4)
    for direction in (K.KDA_PREFIX_FORWARD, K.KDA_PREFIX_BACKWARD):
        xs, x_end = K.state_prefix(A.cuda(), B.cuda(), x0.cuda(), direction=direction, layout=layout)
        torch.cuda.synchronize()
        xs = xs.double().cpu().numpy()
        if layout == "piece_major":
            xs = xs.transpose(1, 0, 2, 3, 4)
        want = np.zeros_like(Ad)
        x = x0d.copy()
        order = range(P) if direction == K.KDA_PREFIX_FORWARD else range(P - 1, -1, -1)
        for p in order:
            want[:, p] = x
            M = Ad[:, p] if direction == K.KDA_PREFIX_FORWARD else np.swapaxes(Ad[:, p], -1, -2)
            x = M @ x + Bd[:, p]
        scale = np.abs(want).max()
        assert np.abs(xs - want).max() <= 1e-5 * scale, (direction, np.abs(xs - want).max(), scale)
        assert np.abs(x_end.double().cpu().numpy() - x).max() <= 1e-5 * np.abs(x).max()


def test_state_prefix_rejects_bad_arguments():
    A = torch.zeros((1, 2, 1, 64, 64), device="cuda")
    with pytest.raises(K.KdaError):
        K.load_library()
        st = K.load_library().kda_state_prefix(1, 2, 1, 96, 0, 1, 2, K._ptr(A), K._ptr(A), None,
                                               K._ptr(A), None, None)
        K._check(st, "kda_state_prefix")
    with pytest.raises(K.KdaError):  # overlapping matrices (piece stride 0)
        st = K.load_library().kda_state_prefix(1, 2, 1, 64, 0, 0, 2, K._ptr(A), K._ptr(A), None,
                                               K._ptr(A), None, None)
        K._check(st, "kda_state_prefix")
