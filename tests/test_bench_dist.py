"""The benchmark's multi-rank host logic on CPU (gloo, world_size 2): the
timed value is the max over ranks and the barrier lets all ranks through.
Each rank runs an independent replica, so there is no data-path collective
to test."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), KDA_BENCH_BACKEND="gloo")
    import bench
    r, ws, local = bench.dist_setup()
    assert (r, ws, local) == (rank, world, rank)
    bench.barrier()
    m = bench.max_over_ranks(10.0 + 5.0 * rank)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, m))


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def test_algorithmic_bytes_match_per_token_head_formula():
    import bench
    from recompute_kda_chunkwise_gb300 import WORKLOADS
    w = WORKLOADS["mbs1_128k_h96_d128_bf16"]
    f, b = bench.algorithmic_bytes(w)
    # bf16: (10D + 2) forward + (18D + 4) backward bytes per token-head
    assert f + b == w.total_tokens * w.H * (28 * w.D + 6)


def test_gdn2_algorithmic_bytes_and_sample():
    # GDN-2: q, k, v, g, erase, write read and o written forward (14D bytes
    # per token-head in bf16); the backward re-reads the six inputs, reads dO
    # and writes six gradients (26D)
    import bench
    from recompute_kda_chunkwise_gb300 import WORKLOADS, make_inputs
    w = WORKLOADS["gdn2_mbs8_8k_h16_d128_bf16"]
    f, b = bench.algorithmic_bytes(w)
    assert f == w.total_tokens * w.H * 14 * w.D and b == w.total_tokens * w.H * 26 * w.D
    assert bench.gate_names(w) == ["erase", "write"]
    small = WORKLOADS["gdn2_b10_t512_h12_d64_f32"]
    sl = bench.make_sample(small, make_inputs(small), 100, 3)
    assert sl["erase"].shape == (100, 3, 64) and sl["write"].shape == (100, 3, 64)
    assert "beta" not in sl
    rate, dt = bench.oracle_sample(small, sl, 2)
    assert rate > 0 and dt > 0


def test_reference_arm_prints_its_line(capsys):
    # --impl reference times the oracle on host cores only (no GPU): one JSON
    # line with impl, cpu_baseline and a zero-copy e2e
    import json
    import bench
    for name in ["tiny_t256_h2_d64_bf16", "gdn2_b10_t512_h12_d64_f32"]:
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-sample-tokens", "64",
                    "--workload", name])
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
        assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
        assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
        assert line["config"]["workload"] == name


def test_traffic_records_follow_their_kernels_sources(tmp_path, monkeypatch):
    import json
    import bench
    # a record keyed by the current hash of its kernel family's own sources
    # is used; every family names its sources
    rec = {k: {"w": {"dram_bytes_per_launch": 1e9 + i, "source_hash": bench.kernel_files_hash(k)}}
           for i, k in enumerate(bench.KERNEL_SOURCES)}
    path = str(tmp_path / "traffic.json")
    with open(path, "w") as f:
        json.dump(rec, f)
    for i, k in enumerate(bench.KERNEL_SOURCES):
        assert bench.ncu_traffic(k, "w", path) == 1e9 + i
    # a change to a kernel's own sources voids its record, and only its record
    real = bench.kernel_files_hash
    monkeypatch.setattr(bench, "kernel_files_hash",
                        lambda k: "changed" if k == "kda_bwd_tc" else real(k))
    assert bench.ncu_traffic("kda_bwd_tc", "w", path) is None
    assert bench.ncu_traffic("kda_fwd_tc", "w", path) is not None
    # unknown kernels and workloads have no record
    assert bench.ncu_traffic("kda_fwd_tc", "no_such_workload", path) is None
    assert bench.ncu_traffic("no_such_kernel", "w", path) is None


def test_bench_flags_from_the_command_line():
    import argparse
    import bench
    from recompute_kda_chunkwise_gb300 import kda as K
    ns = argparse.Namespace
    assert bench.call_flags(ns(force_simt=False, chunk16=False)) == 0
    assert bench.call_flags(ns(force_simt=True, chunk16=False)) == K.KDA_FLAG_FORCE_SIMT
    assert bench.call_flags(ns(force_simt=False, chunk16=True)) == K.KDA_FLAG_CHUNK16
    # the 16-token forward exists for KDA only, and not in the context-parallel split
    for extra in (["--workload", "gdn2_mbs8_8k_h16_d128_bf16"], ["--pieces", "2"]):
        with pytest.raises(SystemExit) as e:
            bench.main(["--chunk16", *extra])
        assert e.value.code == 2
