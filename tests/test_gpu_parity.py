"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every test seals on the GPU and on the oracle from the same seeded inputs,
compares the sealed state, then steps both token by token and compares each
sampled output row and the counters (tolerances in parity_util).  Full-size
workloads run their whole launch (all groups, one launch per token) and
compare a sample of groups against the oracle, plus counter properties that
hold for every group.
"""
import numpy as np
import pytest

from parity_util import ParityRun
from streaming_nystr_landmark_gb300.workloads import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


def _run(wl, sample, dev, steps=None, check_every=None, n_groups=None,
         host_all=None):
    run = ParityRun(wl, sample, dev, n_groups=n_groups, host_all=host_all)
    try:
        run.seal()
        run.check_state()
        run.check_counters_all()
        steps = wl.steps if steps is None else steps
        for n in range(steps):
            run.step()
            if check_every and (n + 1) % check_every == 0:
                run.check_counters_all()
        run.check_counters_all()
        run.check_state()
        assert run.flagged <= max(2, 0.01 * run.checked), (run.flagged, run.checked)
        print(f"[parity] {wl.name}: {run.checked} rows, worst row error "
              f"{run.worst:.2e}, flagged {run.flagged}")
        return run
    finally:
        run.close()


def test_single_head_workload(cuda_device):
    """1 group, H=1, d=64, m=8, w=16, sink=4, t=64, 64 decode tokens."""
    _run(WORKLOADS["single"], [0], cuda_device)


def test_one_layer_workload(cuda_device):
    """8 KV groups x 2 heads, d=128, m=32, w=128, sink=4, t=256, 256 tokens."""
    _run(WORKLOADS["layer"], range(8), cuda_device)


@pytest.mark.parametrize("m", [8, 16, 32, 64])
@pytest.mark.parametrize("rect", ["agg", "fm"])
def test_sweep_workload_full_size(cuda_device, m, rect):
    """2048 groups per launch, t=512, 512 tokens; 3 groups checked."""
    wl = WORKLOADS[f"sweep_m{m}_{rect}"]
    _run(wl, [0, 1027, wl.n_groups - 1], cuda_device, check_every=128)


def test_batch64_workload_full_size(cuda_device):
    """64 seq x 28 layers x 8 groups = 14336 groups per launch, t=256, all
    1024 tokens; 8 groups checked: spread over sequences and layers, and
    the first, second and last groups of the launch's first CTA (the
    persistent kernel's 304 CTAs take groups c, c + 304, ...)."""
    wl = WORKLOADS["batch64"]
    _run(wl, [0, 1, 304, 608, 8 * 28 * 17 + 8 * 5 + 3, 8 * 28 * 40 + 7,
              wl.n_groups - 304, wl.n_groups - 1],
         cuda_device, check_every=256)


def test_long_context_workload_full_size(cuda_device):
    """512 groups x 8 heads, m=64, t=32768 (sealed in one call), 2048
    tokens; four groups checked against the oracle's sequential replay: the
    eight-head kernel runs 256 CTAs of two groups (c and c + 256), so
    groups 0 and 256 are one CTA's first and second, 131 and 509 two
    others'."""
    wl = WORKLOADS["long"]
    _run(wl, [0, 131, 256, wl.n_groups - 3], cuda_device, check_every=512)


@pytest.mark.parametrize("geo", [
    # name, H, d, dv, m, w, sink, t, rect, groups
    ("three_heads", 3, 32, 32, 8, 12, 4, 70, 0, 5),
    ("nine_heads_two_tiles", 9, 16, 16, 8, 10, 2, 40, 1, 3),
    ("no_sinks", 2, 32, 32, 8, 16, 0, 64, 0, 4),
    ("window_of_one", 1, 16, 16, 4, 1, 4, 40, 0, 3),
    ("d_ne_dv", 2, 64, 32, 8, 16, 4, 100, 0, 5),
    ("m_eff_below_budget", 2, 32, 32, 32, 64, 4, 160, 0, 3),
    ("wide_head", 1, 256, 256, 16, 32, 4, 200, 0, 2),
    ("ragged_tail_129_groups", 2, 32, 32, 8, 16, 4, 64, 0, 129),
    # Tensor-core seal replay (>= 256 keys to fold, m >= 32) on an uneven
    # geometry: 2 heads of 48 landmarks in the first CTA's 128 rows, 1 in
    # the second, d = 96 (three 32-element chunk groups), dv = 64.
    ("tc_replay_uneven", 3, 96, 64, 48, 64, 4, 400, 0, 3),
])
def test_edge_geometries(cuda_device, geo):
    name, H, d, dv, m, w, sink, t, rect, groups = geo
    wl = Workload(name, H, d, dv, m, w, sink, rect, t, 40, 1, 1, groups,
                  "unit2", seed=77)
    sample = range(groups) if groups <= 8 else [0, 63, 64, groups - 1]
    _run(wl, sample, cuda_device, n_groups=groups, host_all=groups <= 8)
