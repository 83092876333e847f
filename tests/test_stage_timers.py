"""The tracing build (kernel stage timers compiled in with -DKDA_STAGE_TIMERS).

CPU: it compiles and exports its two counter accessors, which the default
library does not have. GPU: the counters of one forward + backward count every
chunk step of every CTA role.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np

import pytest

from recompute_kda_chunkwise_gb300 import build as kbuild


def _exports(path):
    lib = ctypes.CDLL(path)
    return [hasattr(lib, n) for n in ("kda_fwd_stage_timers", "kda_bwd_stage_timers")]


def test_tracing_build_exports_its_counters_and_the_default_build_does_not():
    traced = kbuild.build(stage_timers=True)
    assert os.path.dirname(traced) != os.path.dirname(kbuild.LIB)
    assert _exports(traced) == [True, True]
    assert _exports(kbuild.build()) == [False, False]


_CHILD = """
import sys
import numpy as np
from recompute_kda_chunkwise_gb300 import stage_timers
from recompute_kda_chunkwise_gb300.inputs import Workload
w = Workload("stage_timer_check", (2500, 1100), 2, 128, "bf16", seed=9300, param_std=0.3)
fb, bb, times = stage_timers.measure(w, iters=2)
np.savez(sys.argv[1], fb=fb, bb=bb, times=np.array(times))
"""


@pytest.mark.gpu
def test_stage_counters_count_every_chunk_step(tmp_path):
    # a process of its own: this one may already hold the default library
    out = tmp_path / "stages.npz"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CHILD, str(out)], cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    d = np.load(out)
    fb, bb, times = d["fb"], d["bb"], d["times"]
    # 2 sequences x 2 heads: 4 items, split mode in both directions (the spare
    # SMs run as helpers)
    items = 4
    fwd_chunks = sum((n + 63) // 64 for n in (2500, 1100)) * 2   # 64-token chunks, all items
    bwd_chunks = sum((n + 15) // 16 for n in (2500, 1100)) * 2   # 16-token chunks, all items
    # the forward's main CTAs step through every chunk of their item
    assert fb[:items, 31].sum() == fwd_chunks
    # the backward's reverse CTAs walk every chunk once in the reverse pass
    assert bb[:items, 31].sum() == bwd_chunks
    # helpers took part in both directions, and every counted step has cycles
    assert fb[items:, 31].sum() > 0 and bb[items:, 31].sum() > 0
    assert (fb[:, :31].sum(axis=1) > 0).sum() >= items and (bb[:, :31].sum(axis=1) > 0).sum() >= items
    assert times[0] > 0 and times[1] > 0
