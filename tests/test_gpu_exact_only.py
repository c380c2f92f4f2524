"""Exact-only (short-prompt) groups on the GPU.

A prompt of t <= w + sink + 8 keys takes the page's exact-only mode: all keys
stay exact, the window grows with every token, and each output is softmax
attention over every key so far.  Here such groups share a handle (and every
launch) with landmark-path groups; both kinds are checked against the oracle,
the exact ones additionally against brute-force softmax attention, and a token
that would overflow exact_cap is refused before anything runs."""
import numpy as np
import pytest

from oracle import NystromOracle, score_scale
from parity_util import OUT_TOL, row_err
from streaming_nystr_landmark_gb300 import nys
from streaming_nystr_landmark_gb300.workloads import (Workload, host_prompt_batch,
                                                      host_token_batch)

pytestmark = pytest.mark.gpu


def _softmax_attention(q, keys, vals, scale):
    lg = keys.astype(np.float64) @ q.astype(np.float64) * scale
    p = np.exp(lg - lg.max())
    return (p @ vals.astype(np.float64)) / p.sum()


@pytest.mark.parametrize("heads", [1, 2])
def test_exact_only_groups_beside_landmark_groups(cuda_device, heads):
    import torch
    H, d, m, w, sink, cap = heads, 32, 8, 16, 4, 40
    n_exact, n_land = 3, 3
    t_exact, t_land = 20, 64          # 20 <= w + sink + 8 = 28 < 64
    wl_e = Workload("exact", H, d, d, m, w, sink, 0, t_exact, 20, 1, 1, n_exact, "unit2", seed=41)
    wl_l = Workload("land", H, d, d, m, w, sink, 0, t_land, 20, 1, 1, n_land, "unit2", seed=42)
    st = nys.NystromStates(m, w, sink, H, d, d, n_exact + n_land, 0, cuda_device, exact_cap=cap)
    qe, ke, ve, ge = host_prompt_batch(wl_e, range(n_exact))
    ql, kl, vl, gl = host_prompt_batch(wl_l, range(n_land))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    # exact groups interleave with landmark groups: 0 L 1 L 2 L -> seal one by one
    order = []
    for i in range(n_exact):
        order += [("e", i), ("l", i)]
    oracles, keys, vals = [], [], []
    for g, (kind, i) in enumerate(order):
        q, k, v = (qe, ke, ve) if kind == "e" else (ql, kl, vl)
        st.seal(dev(q[i:i + 1]), dev(k[i:i + 1]), dev(v[i:i + 1]), g0=g, n=1)
        o = NystromOracle(m, w, sink, H)
        o.prefill(q[i], k[i], v[i])
        assert o.exact_only == (kind == "e")
        oracles.append(o)
        keys.append(list(k[i]))
        vals.append(list(v[i]))
    torch.cuda.synchronize()
    info, far = st.query(0)
    assert info["mode"] == 2 and info["win_len"] == t_exact and far == [0] * H
    steps = cap - t_exact               # fill the exact groups to capacity
    for n in range(steps):
        te = host_token_batch(ge, n)
        tl = host_token_batch(gl, n)
        toks = [(te if kind == "e" else tl) for kind, _ in order]
        tq = np.stack([toks[g][0][i] for g, (_, i) in enumerate(order)])
        tk = np.stack([toks[g][1][i] for g, (_, i) in enumerate(order)])
        tv = np.stack([toks[g][2][i] for g, (_, i) in enumerate(order)])
        out = torch.empty((len(order), H, d), device=cuda_device)
        st.step(dev(tq), dev(tk), dev(tv), out)
        got = out.cpu().numpy().astype(np.float64)
        for g, o in enumerate(oracles):
            ref = o.step(tq[g], tk[g], tv[g])
            keys[g].append(tk[g])
            vals[g].append(tv[g])
            for h in range(H):
                assert row_err(got[g, h], ref[h]) <= OUT_TOL, (n, g, h)
                if order[g][0] == "e":
                    exact = _softmax_attention(tq[g][h], np.array(keys[g]), np.array(vals[g]),
                                               score_scale(d))
                    assert row_err(got[g, h], exact) <= OUT_TOL, (n, g, h)
    info, _ = st.query(0)
    assert info["win_len"] == cap
    ints = st.region("ints").cpu().numpy()
    assert np.all(ints[:, 5] == 0)
    # One more token would exceed exact_cap: refused on the host.
    out = torch.empty((len(order), H, d), device=cuda_device)
    z = torch.zeros((len(order), H, d), device=cuda_device)
    with pytest.raises(nys.NysError) as ei:
        st.step(z, z[:, 0].contiguous(), z[:, 0].contiguous(), out)
    assert ei.value.code == nys.NYS_E_CAPACITY
    # Re-sealing an exact group on a long prompt turns it into a landmark group.
    st.seal(dev(ql[:1]), dev(kl[:1]), dev(vl[:1]), g0=0, n=1)
    torch.cuda.synchronize()
    assert st.query(0)[0]["mode"] == 1
    st.close()


def test_exact_only_needs_capacity(cuda_device):
    import torch
    st = nys.NystromStates(8, 16, 4, 1, 16, 16, 1, 0, cuda_device, exact_cap=10)
    k = torch.zeros((1, 20, 16), device=cuda_device)
    with pytest.raises(nys.NysError) as ei:      # 20 keys > exact_cap = 10
        st.seal(torch.zeros((1, 1, 20, 16), device=cuda_device), k, k.clone())
    assert ei.value.code == nys.NYS_E_RANGE
    st.close()
