"""The decode kernel's bounded waits, made to run out on purpose.

nys_debug_stall_once makes the next launch's first CTA withhold one ring
stage: no copy is issued for it, so that CTA's consumer warps wait on a stage
that never fills.  Each wait gives up after its time limit, the CTA marks the
status word of every group it had left and returns; nothing faults and the
CUDA context stays usable.  The test checks that exactly that CTA's groups
report the stale status, that every other group stepped exactly as on an
untouched twin handle, and that a re-seal clears the status.
"""
import numpy as np
import pytest

from streaming_nystr_landmark_gb300 import nys
from streaming_nystr_landmark_gb300.workloads import (Workload, host_prompt_batch,
                                                      host_token_batch)

pytestmark = pytest.mark.gpu

GROUPS = 700  # more than one wave of CTAs, so the first CTA owns several groups


def _status(st):
    return st.region("ints")[:, 5].cpu().numpy()


def test_stalled_stage_times_out_and_marks_its_groups(cuda_device):
    import torch
    wl = Workload("stall", 2, 128, 128, 32, 128, 4, 0, 160, 4, 1, 1, GROUPS,
                  "unit2", seed=19)
    gids = range(GROUPS)
    q, k, v, gens = host_prompt_batch(wl, gids)
    q, k, v = (torch.from_numpy(a).to(cuda_device) for a in (q, k, v))
    states = [nys.NystromStates(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d, wl.dv,
                                GROUPS, wl.rect, cuda_device) for _ in range(2)]
    a, b = states
    try:
        for st in states:
            st.seal(q, k, v)
        toks = [tuple(torch.from_numpy(x).to(cuda_device)
                      for x in host_token_batch(gens, n)) for n in range(3)]
        outs = [torch.zeros((GROUPS, 2, 128), device=cuda_device) for _ in range(2)]

        # One clean token on both, then the stalled one on `a`.
        for st, o in zip(states, outs):
            st.step(*toks[0], o)
        a.debug_stall_once(3)
        for st, o in zip(states, outs):
            st.step(*toks[1], o)
        torch.cuda.synchronize()  # the stalled CTA returned: the context is alive

        sa, sb = _status(a), _status(b)
        assert not sb.any()
        bad = np.flatnonzero(sa)
        assert bad.size > 0 and bad[0] == 0, bad[:8]
        if bad.size > 1:  # a grid-stride set: group 0 and every grid after it
            stride = int(bad[1])
            assert np.array_equal(bad, np.arange(0, GROUPS, stride))
        assert a.query(0)[0]["status"] == 1
        good = np.setdiff1d(np.arange(GROUPS), bad)
        # Every group the stalled CTA did not own stepped bit for bit as on b.
        for name in ("win_k", "t_hat", "t_lo", "z_hat", "z_lo", "m_max", "far_len"):
            ra, rb = a.region(name), b.region(name)
            assert torch.equal(ra[good], rb[good]), name
        assert torch.equal(outs[0][good], outs[1][good])

        # A re-seal clears the status; both handles then agree everywhere.
        for st in states:
            st.seal(q, k, v)
        assert not _status(a).any()
        for st, o in zip(states, outs):
            st.step(*toks[0], o)
        torch.cuda.synchronize()
        assert not _status(a).any()
        assert torch.equal(outs[0], outs[1])
    finally:
        for st in states:
            st.close()


def test_stalled_replay_times_out_and_marks_its_group(cuda_device):
    """The tensor-core seal replay's bounded waits: its first CTA withholds
    its first MMAs (nys_debug_stall_replay_once), waits out its 2 s limit,
    marks its group (status 3), frees its tensor memory and returns."""
    import torch
    # m >= 32 and 300 - 16 - 4 = 280 keys to fold: the tensor-core replay.
    wl = Workload("replay_stall", 2, 32, 32, 32, 16, 4, 0, 300, 4, 1, 1, 4,
                  "unit2", seed=23)
    q, k, v, _ = host_prompt_batch(wl, range(4))
    q, k, v = (torch.from_numpy(a).to(cuda_device) for a in (q, k, v))
    states = [nys.NystromStates(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d, wl.dv,
                                4, wl.rect, cuda_device) for _ in range(2)]
    a, b = states
    try:
        a.debug_stall_replay_once()
        for st in states:
            st.seal(q, k, v)
        torch.cuda.synchronize()  # the stalled CTA returned: the context is alive
        assert list(_status(a)) == [3, 0, 0, 0]
        assert not _status(b).any()
        assert a.query(0)[0]["status"] == 3
        for name in ("t_hat", "t_lo", "z_hat", "z_lo", "m_max", "mu", "k_tilde"):
            assert torch.equal(a.region(name)[1:], b.region(name)[1:]), name
        a.seal(q, k, v)  # a fresh seal clears the status
        torch.cuda.synchronize()
        assert not _status(a).any()
        for name in ("t_hat", "t_lo", "z_hat", "z_lo", "m_max", "mu"):
            assert torch.equal(a.region(name), b.region(name)), name
    finally:
        for st in states:
            st.close()
