"""The oracle worker pool used by the full-size parity runs: spawned workers
that rebuild their groups' inputs from the seeded streams give exactly the
outputs of oracles stepped in this process, and a failure in a worker
surfaces here as an error instead of a wait."""
import numpy as np
import pytest

from oracle import NystromOracle
from oracle_pool import OraclePool
from parity_util import GUARD_BAND, UNDERFLOW_GAP
from streaming_nystr_landmark_gb300.workloads import (Workload, host_prompt_batch,
                                                      host_token_batch)


def _wl():
    return Workload("pool", 2, 16, 16, 8, 16, 4, 0, 64, 6, 1, 1, 5, "unit2", seed=3)


def test_pool_matches_in_process_oracles():
    wl = _wl()
    groups = [0, 2, 3, 4]
    pool = OraclePool(wl, groups, 2, GUARD_BAND, UNDERFLOW_GAP)
    try:
        pool.ready()
        qh, kh, vh, gens = host_prompt_batch(wl, groups)
        local = []
        for i in range(len(groups)):
            o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.rect)
            o.prefill(qh[i], kh[i], vh[i])
            local.append(o)
        for n in range(wl.steps):
            pool.start_step(n)
            refs, flags, diag = pool.finish_step()
            tq, tk, tv = host_token_batch(gens, n)
            assert refs.shape == (len(groups), wl.heads_per_kv, wl.dv)
            for i, o in enumerate(local):
                assert np.array_equal(refs[i], o.step(tq[i], tk[i], tv[i]))
                want = [abs(dg.margin) < GUARD_BAND or dg.near_gap > UNDERFLOW_GAP
                        for dg in o.diags[-1]]
                assert list(flags[i]) == want
                assert np.array_equal(diag[i], [[dg.kappa, dg.margin, dg.near_gap]
                                                for dg in o.diags[-1]])
    finally:
        pool.close()


def test_pool_hands_over_prompts_and_token_streams():
    wl = _wl()
    groups = [4, 1]
    pool = OraclePool(wl, groups, 2, GUARD_BAND, UNDERFLOW_GAP, send_prompts=True)
    try:
        got = list(pool.prompts())
        pool.ready()
        qh, kh, vh, gens = host_prompt_batch(wl, groups)
        assert [x[0] for x in got] == groups
        for i, (g, q, k, v, gi) in enumerate(got):
            assert np.array_equal(q, qh[i]) and np.array_equal(k, kh[i])
            assert np.array_equal(v, vh[i])
        theirs = [x[4] for x in got]
        for n in range(3):
            a, b = host_token_batch(theirs, n), host_token_batch(gens, n)
            assert all(np.array_equal(x, y) for x, y in zip(a, b))
    finally:
        pool.close()


def test_worker_failure_is_reported():
    """A state comparison that fails in a worker (here: regions of the
    wrong shape) raises in the parent."""
    pool = OraclePool(_wl(), [1], 1, GUARD_BAND, UNDERFLOW_GAP)
    try:
        pool.ready()
        with pytest.raises(AssertionError):
            pool.compare_state({"ints": np.zeros((2, 8), np.int32)}, 1e-5)
    finally:
        pool.close()
