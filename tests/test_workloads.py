"""Host-side checks of the seeded synthetic inputs (no method arithmetic)."""
import numpy as np
import pytest

from streaming_nystr_landmark_gb300.workloads import (
    WORKLOADS, GroupInputs, host_prompt_batch, host_token_batch)


def test_workload_geometry():
    assert WORKLOADS["batch64"].n_groups == 64 * 28 * 8
    assert WORKLOADS["layer"].n_groups == 8
    assert WORKLOADS["long"].n_groups == 512
    assert sum(k.startswith("sweep_") for k in WORKLOADS) == 8
    wl = WORKLOADS["batch64"]
    assert wl.group_coords(0) == (0, 0, 0)
    assert wl.group_coords(wl.n_groups - 1) == (63, 27, 7)
    assert wl.group_coords(8 * 28 + 9) == (1, 1, 1)
    for wl in WORKLOADS.values():
        # every configured prompt takes the landmark path with m_eff = m
        assert wl.t > wl.w + wl.sink + 8 and wl.t // 8 >= wl.m


def test_group_streams_independent_and_deterministic():
    wl = WORKLOADS["layer"]
    q1, k1, v1, g1 = host_prompt_batch(wl, [3, 5])
    q2, k2, v2, g2 = host_prompt_batch(wl, [5])
    np.testing.assert_array_equal(q1[1], q2[0])
    np.testing.assert_array_equal(k1[1], k2[0])
    a = host_token_batch(g1, 0)
    b = host_token_batch(g2, 0)
    np.testing.assert_array_equal(a[0][1], b[0][0])
    assert not np.array_equal(q1[0], q1[1])
    assert q1.dtype == np.float32 and q1.shape == (2, 2, 256, 128)


def test_token_order_enforced():
    gi = GroupInputs(WORKLOADS["single"], 0)
    gi.prompt()
    gi.token(0)
    with pytest.raises(ValueError):
        gi.token(2)


@pytest.mark.parametrize("name,norm", [("single", 2.0), ("layer", 3.0)])
def test_key_mean_offset(name, norm):
    wl = WORKLOADS[name]
    _, k, _, _ = host_prompt_batch(wl, [0])
    mean = k[0].astype(np.float64).mean(axis=0)
    assert abs(np.linalg.norm(mean) - norm) < 0.35 * np.sqrt(wl.d / wl.t) + 0.3


def test_walk_moves_slowly():
    wl = WORKLOADS["long"].with_(t=2048, steps=8)
    gi = GroupInputs(wl, 0)
    _, k, _ = gi.prompt()
    early = k[:512].astype(np.float64).mean(0)
    late = k[-512:].astype(np.float64).mean(0)
    # 1536 steps of norm 0.01 in random directions: drift ~ 0.01*sqrt(1536)
    assert np.linalg.norm(late - early) < 1.5
    t0 = gi.token(0)
    assert t0[1].shape == (128,)
