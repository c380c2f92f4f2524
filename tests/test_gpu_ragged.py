"""One batched seal over prompts of different lengths (nys_seal_ragged).

Each group keeps its own prompt length and effective landmark count
(m_eff = clamp(t/8, 4, m) per group); the sealed state of every group must
match the oracle sealed on that group's prompt alone, be bit-identical to
sealing the group by itself with nys_seal, and decode correctly afterwards."""
import numpy as np
import pytest

from oracle import NystromOracle
from parity_util import OUT_TOL, compare_group_state, read_state, row_err
from streaming_nystr_landmark_gb300 import nys
from streaming_nystr_landmark_gb300.workloads import GroupInputs, Workload

pytestmark = pytest.mark.gpu

TS = [70, 96, 200, 133, 300, 41, 257]   # m_eff 8, 12, 25, 16, 32, 5, 32


def _groups(cuda_device, rect):
    import torch
    H, d, m, w, sink = 2, 32, 32, 16, 4
    gens, qs, ks, vs = [], [], [], []
    for g, t in enumerate(TS):
        wl = Workload("ragged", H, d, d, m, w, sink, rect, t, 16, 1, 1, len(TS),
                      "unit2", seed=31)
        gi = GroupInputs(wl, g)
        q, k, v = gi.prompt()
        gens.append(gi)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    qp = dev(np.concatenate([q.reshape(-1, d) for q in qs]))
    kp = dev(np.concatenate(ks))
    vp = dev(np.concatenate(vs))
    return (H, d, m, w, sink), gens, (qs, ks, vs), (qp, kp, vp)


@pytest.mark.parametrize("rect", [0, 1])
def test_ragged_seal_matches_oracle_and_separate_seals(cuda_device, rect):
    import torch
    (H, d, m, w, sink), gens, (qs, ks, vs), (qp, kp, vp) = _groups(cuda_device, rect)
    n = len(TS)
    st = nys.NystromStates(m, w, sink, H, d, d, n, rect, cuda_device)
    st.seal_ragged(TS, qp, kp, vp)
    torch.cuda.synchronize()
    reg = read_state(st)
    oracles = []
    for g, t in enumerate(TS):
        o = NystromOracle(m, w, sink, H, rect)
        o.prefill(qs[g], ks[g], vs[g])
        oracles.append(o)
        compare_group_state(reg, g, o)
        assert reg["ints"][g][3] == t
    # Bit-identical to sealing each group alone (same kernels, same inputs).
    for g, t in enumerate(TS):
        one = nys.NystromStates(m, w, sink, H, d, d, 1, rect, cuda_device)
        one.seal(torch.from_numpy(qs[g][None]).to(cuda_device),
                 torch.from_numpy(ks[g][None]).to(cuda_device),
                 torch.from_numpy(vs[g][None]).to(cuda_device))
        for name in ("k_tilde", "q_tilde", "mu", "t_hat", "t_lo", "z_hat", "z_lo",
                     "m_max", "win_k", "win_v", "sink_k", "ints", "far_len"):
            assert torch.equal(one.region(name)[0], st.region(name)[g]), (g, name)
        one.close()
    # Decode all groups together afterwards.
    worst = 0.0
    for step in range(16):
        toks = [gi.token(step) for gi in gens]
        tq = torch.from_numpy(np.stack([x[0] for x in toks])).to(cuda_device)
        tk = torch.from_numpy(np.stack([x[1] for x in toks])).to(cuda_device)
        tv = torch.from_numpy(np.stack([x[2] for x in toks])).to(cuda_device)
        out = torch.empty((n, H, d), device=cuda_device)
        st.step(tq, tk, tv, out)
        got = out.cpu().numpy().astype(np.float64)
        for g, o in enumerate(oracles):
            ref = o.step(*toks[g])
            for h in range(H):
                worst = max(worst, row_err(got[g, h], ref[h]))
    assert worst <= OUT_TOL, worst
    st.close()


def test_ragged_seal_rejects_short_prompt(cuda_device):
    import torch
    st = nys.NystromStates(8, 16, 4, 1, 16, 16, 2, 0, cuda_device)
    k = torch.zeros((64 + 28, 16), device=cuda_device)
    with pytest.raises(nys.NysError) as ei:
        st.seal_ragged([64, 28], torch.zeros((92, 16), device=cuda_device), k,
                       torch.zeros_like(k))
    assert ei.value.code == nys.NYS_E_EXACT_ONLY
    st.close()
