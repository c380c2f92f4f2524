"""GPU-side ABI behaviour: error codes on a live device, sub-range and empty
launches, the non-finite ridge fallback, large finite landmark logits, and the
step kernel alone on a state uploaded from the oracle."""
import numpy as np
import pytest

from oracle import NystromOracle
from parity_util import (OUT_TOL, compare_group_state, read_state, row_err,
                         step_oracles_and_compare)
from streaming_nystr_landmark_gb300 import nys
from streaming_nystr_landmark_gb300.workloads import (Workload, host_prompt_batch,
                                                      host_token_batch)

pytestmark = pytest.mark.gpu


def _small(device, groups=6, **kw):
    wl = Workload("abi", 2, 32, 32, 8, 16, 4, 0, 64, 8, 1, 1, groups, "unit2",
                  seed=5).with_(**kw)
    st = nys.NystromStates(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d, wl.dv,
                           groups, wl.rect, device)
    return wl, st


def _to(dev, *arrs):
    import torch
    return [torch.from_numpy(a).to(dev) for a in arrs]


def test_error_codes_on_device(cuda_device):
    import torch
    wl, st = _small(cuda_device)
    q, k, v, gens = host_prompt_batch(wl, range(6))
    q, k, v = _to(cuda_device, q, k, v)
    tq, tk, tv = _to(cuda_device, *host_token_batch(gens, 0))
    out = torch.empty((6, 2, 32), device=cuda_device)
    with pytest.raises(nys.NysError) as ei:
        st.step(tq, tk, tv, out)
    assert ei.value.code == nys.NYS_E_NOT_SEALED
    short = 16 + 4 + 8
    with pytest.raises(nys.NysError) as ei:
        st.seal(q[:, :, :short].contiguous(), k[:, :short].contiguous(),
                v[:, :short].contiguous())
    assert ei.value.code == nys.NYS_E_EXACT_ONLY
    st.seal(q, k, v)
    raw = torch.empty(6 * 32 + 1, device=cuda_device)
    bad = raw[1:].view(6, 32)
    with pytest.raises(nys.NysError) as ei:
        nys.nys_step_batch(st.handle, 0, 6, tq.data_ptr(), bad.data_ptr(),
                           tv.data_ptr(), out.data_ptr())
    assert ei.value.code == nys.NYS_E_ALIGN
    with pytest.raises(nys.NysError) as ei:
        nys.nys_step_batch(st.handle, 4, 3, tq.data_ptr(), tk.data_ptr(),
                           tv.data_ptr(), out.data_ptr())
    assert ei.value.code == nys.NYS_E_RANGE
    # Empty launches are valid no-ops.
    nys.nys_step_batch(st.handle, 6, 0, tq.data_ptr(), tk.data_ptr(),
                       tv.data_ptr(), out.data_ptr())
    st.step(tq, tk, tv, out)
    torch.cuda.synchronize()
    info, far = st.query(3)
    assert info == {"mode": 1, "m_eff": 8, "t": 64, "win_len": 16,
                    "win_head": (64 - 4 + 1) % 16, "status": 0}
    assert far == [64 - 4 - 16 + 1] * 2
    st.close()


def test_subrange_leaves_other_groups_untouched(cuda_device):
    import torch
    wl, st = _small(cuda_device)
    q, k, v, gens = host_prompt_batch(wl, range(6))
    st.seal(*_to(cuda_device, q, k, v))
    before = {n: st.region(n).clone() for n in ("win_k", "t_hat", "z_hat", "ints",
                                                  "far_len")}
    th = host_token_batch(gens, 0)
    tq, tk, tv = _to(cuda_device, *th)
    out = torch.zeros((3, 2, 32), device=cuda_device)
    st.step(tq[2:5].contiguous(), tk[2:5].contiguous(), tv[2:5].contiguous(), out,
            g0=2, n=3)
    torch.cuda.synchronize()
    for name, old in before.items():
        new = st.region(name)
        for g in (0, 1, 5):
            assert torch.equal(new[g], old[g]), (name, g)
        assert not torch.equal(new[2:5], old[2:5]), name
    # The stepped groups match the oracle.
    for i, g in enumerate(range(2, 5)):
        o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv)
        o.prefill(q[g], k[g], v[g])
        ref = o.step(th[0][g], th[1][g], th[2][g])
        for h in range(2):
            assert row_err(out[i, h].cpu().numpy().astype(np.float64), ref[h]) <= OUT_TOL
    st.close()


def test_overflowing_landmark_kernel_takes_ridge_fallback(cuda_device):
    """Prompt logits past exp's f64 range make A infinite: every Cholesky
    attempt fails and M falls back to I / mean diag = 0, on both sides."""
    import torch
    wl, st = _small(cuda_device, groups=2)
    rng = np.random.default_rng(3)
    t = wl.t
    q = np.full((2, 2, t, 32), 30.0, np.float32)
    k = (30.0 + rng.random((2, t, 32))).astype(np.float32)
    v = rng.standard_normal((2, t, 32)).astype(np.float32)
    st.seal(*_to(cuda_device, q, k, v))
    torch.cuda.synchronize()
    mu = st.region("mu").cpu().numpy()
    for g in range(2):
        o = NystromOracle(wl.m, wl.w, wl.sink, 2)
        o.prefill(q[g], k[g], v[g])
        for h in range(2):
            assert o.hs[h].ridge.fallback
            np.testing.assert_array_equal(mu[g, h], o.hs[h].mu.astype(np.float32))
        tq = rng.standard_normal((2, 32)).astype(np.float32)
        tk = rng.standard_normal(32).astype(np.float32)
        tv = rng.standard_normal(32).astype(np.float32)
        ref = o.step(tq, tk, tv)
        out = torch.empty((1, 2, 32), device=cuda_device)
        st.step(*_to(cuda_device, tq[None], tk[None], tv[None]), out, g0=g, n=1)
        for h in range(2):
            assert row_err(out[0, h].cpu().numpy().astype(np.float64), ref[h]) <= OUT_TOL
    st.close()


def test_large_landmark_logits_sum_gram_in_f64(cuda_device):
    """Landmark logits of 60 (A up to e^60, finite): past the +-41 bound of
    the double-float A^T A, so the pinv sums A^T A in f64; the sealed state
    and a decode step still match the oracle.  Every prompt segment is
    constant (keys and queries alpha e_b in segment b), so the landmarks are
    alpha e_b and A = J + (e^60 - 1) I is well conditioned."""
    import torch
    wl, st = _small(cuda_device, groups=2)
    t, d, m, H = wl.t, wl.d, wl.m, wl.heads_per_kv
    scale = float(np.float32(1.0) / np.sqrt(np.float32(d)))
    alpha = np.float32(np.sqrt(60.0 / scale))
    seg = np.arange(t) * m // t  # segment of each prompt position (t = 8 m)
    rng = np.random.default_rng(11)
    q = np.zeros((2, H, t, d), np.float32)
    q[:, :, np.arange(t), seg] = alpha
    k = np.zeros((2, t, d), np.float32)
    k[:, np.arange(t), seg] = alpha
    v = rng.standard_normal((2, t, wl.dv)).astype(np.float32)
    st.seal(*_to(cuda_device, q, k, v))
    torch.cuda.synchronize()
    reg = read_state(st)
    for g in range(2):
        o = NystromOracle(m, wl.w, wl.sink, H)
        o.prefill(q[g], k[g], v[g])
        for h in range(H):
            assert not o.hs[h].ridge.fallback
        compare_group_state(reg, g, o)
        tq = rng.standard_normal((H, d)).astype(np.float32)
        tk = rng.standard_normal(d).astype(np.float32)
        tv = rng.standard_normal(wl.dv).astype(np.float32)
        ref = o.step(tq, tk, tv)
        out = torch.empty((1, H, wl.dv), device=cuda_device)
        st.step(*_to(cuda_device, tq[None], tk[None], tv[None]), out, g0=g, n=1)
        for h in range(H):
            assert row_err(out[0, h].cpu().numpy().astype(np.float64), ref[h]) <= OUT_TOL
    st.close()


def test_step_kernel_on_uploaded_oracle_state(cuda_device):
    """Isolate the step kernel: write the oracle's sealed state into the
    device buffer through the layout, then step both."""
    import torch
    wl, st = _small(cuda_device, groups=3, heads_per_kv=3, m=8, w=16)
    q, k, v, gens = host_prompt_batch(wl, range(3))
    oracles = []
    for g in range(3):
        o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv)
        o.prefill(q[g], k[g], v[g])
        oracles.append(o)
        me = o.m_eff
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(cuda_device)
        st.region("win_k")[g] = f32(o.win_k)
        st.region("win_v")[g] = f32(o.win_v)
        st.region("sink_k")[g] = f32(o.sink_k)
        st.region("sink_v")[g] = f32(o.sink_v)
        st.region("k_tilde")[g, :me] = f32(o.k_tilde)
        for h, hs in enumerate(o.hs):
            st.region("q_tilde")[g, h, :me] = f32(hs.q_tilde)
            st.region("mu")[g, h, :me, :me] = f32(hs.mu)
            st.region("t_hat")[g, h, :me] = f32(hs.t_hat)
            st.region("z_hat")[g, h, :me] = f32(hs.z_hat)
            st.region("m_max")[g, h, :me] = f32(hs.m_max)
            st.region("far_len")[g, h] = hs.far_len
        st.region("ints")[g, :5] = torch.tensor(
            [o.win_head, o.win_len, me, wl.t, 1], dtype=torch.int32)
    st.mark_sealed()
    for n in range(20):
        tq, tk, tv = host_token_batch(gens, n)
        out = torch.empty((3, 3, 32), device=cuda_device)
        st.step(*_to(cuda_device, tq, tk, tv), out)
        got = out.cpu().numpy().astype(np.float64)
        for g, o in enumerate(oracles):
            ref = o.step(tq[g], tk[g], tv[g])
            for h in range(3):
                assert row_err(got[g, h], ref[h]) <= OUT_TOL, (n, g, h)
    st.close()


def test_host_pipeline_matches_direct_steps(cuda_device):
    """The pipelined host path (copies on a side stream, double-buffered
    device staging) yields exactly the outputs of plain launches on device
    inputs, token after token."""
    import torch
    wl, st_a = _small(cuda_device, groups=5)
    _, st_b = _small(cuda_device, groups=5)
    q, k, v, gens = host_prompt_batch(wl, range(5))
    qd, kd, vd = _to(cuda_device, q, k, v)
    st_a.seal(qd, kd, vd)
    st_b.seal(qd, kd, vd)
    pipe = st_b.host_pipeline()
    outs_host = []
    outs_dev = []
    for n in range(12):
        tq, tk, tv = host_token_batch(gens, n)
        hq, hk, hv = [torch.from_numpy(a).pin_memory() for a in (tq, tk, tv)]
        hout = torch.empty((5, 2, 32), pin_memory=True)
        pipe.submit(hq, hk, hv, hout)
        outs_host.append(hout)
        out = torch.empty((5, 2, 32), device=cuda_device)
        st_a.step(*_to(cuda_device, tq, tk, tv), out)
        outs_dev.append(out)
    pipe.synchronize()
    for a, b in zip(outs_dev, outs_host):
        assert torch.equal(a.cpu(), b)
    st_a.close()
    st_b.close()


def test_per_layer_launches_and_graph_replay_match_fused(cuda_device):
    """A model steps one layer at a time: per-layer handles stepped with one
    launch each, eagerly or replayed from a CUDA graph, give bit-identical
    outputs and state to one fused launch over all layers' groups, and every
    output row of every token matches the fp64 oracle of its group."""
    import torch
    L, per = 3, 6
    wl = Workload("layers", 2, 32, 32, 8, 16, 4, 0, 64, 8, 1, 1, L * per, "unit2", seed=9)
    q, k, v, gens = host_prompt_batch(wl, range(L * per))
    oracles = []
    for g in range(L * per):
        o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.rect)
        o.prefill(q[g], k[g], v[g])
        oracles.append(o)
    mk = lambda n: nys.NystromStates(wl.m, wl.w, wl.sink, 2, 32, 32, n, 0, cuda_device)
    fused = mk(L * per)
    fused.seal(*_to(cuda_device, q, k, v))
    eager = [mk(per) for _ in range(L)]
    graphed = [mk(per) for _ in range(L)]
    for l in range(L):
        sl = slice(l * per, (l + 1) * per)
        for st in (eager[l], graphed[l]):
            st.seal(*_to(cuda_device, q[sl], k[sl], v[sl]))
    tq = torch.empty((L * per, 2, 32), device=cuda_device)
    tk = torch.empty((L * per, 32), device=cuda_device)
    tv = torch.empty((L * per, 32), device=cuda_device)
    out_f = torch.empty((L * per, 2, 32), device=cuda_device)
    out_e = torch.empty_like(out_f)
    out_g = torch.empty_like(out_f)

    def layered(states, out):
        for l, st in enumerate(states):
            sl = slice(l * per, (l + 1) * per)
            st.step(tq[sl], tk[sl], tv[sl], out[sl])

    # warm up the graphed handles once, outside capture, on token 0
    th = host_token_batch(gens, 0)
    for dst, src in zip((tq, tk, tv), th):
        dst.copy_(torch.from_numpy(src))
    fused.step(tq, tk, tv, out_f)
    layered(eager, out_e)
    layered(graphed, out_g)
    torch.cuda.synchronize()
    assert torch.equal(out_f, out_e) and torch.equal(out_f, out_g)
    step_oracles_and_compare(oracles, *th, [out_e.cpu().numpy(), out_g.cpu().numpy()])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layered(graphed, out_g)
    for n in range(1, 8):
        th = host_token_batch(gens, n)
        for dst, src in zip((tq, tk, tv), th):
            dst.copy_(torch.from_numpy(src))
        fused.step(tq, tk, tv, out_f)
        layered(eager, out_e)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_f, out_e), n
        assert torch.equal(out_f, out_g), n
        step_oracles_and_compare(oracles, *th, [out_e.cpu().numpy(), out_g.cpu().numpy()])
    for name in ("t_hat", "t_lo", "z_hat", "m_max", "far_len", "ints", "win_k"):
        whole = fused.region(name)
        for l in range(L):
            assert torch.equal(whole[l * per:(l + 1) * per], eager[l].region(name)), name
            assert torch.equal(whole[l * per:(l + 1) * per], graphed[l].region(name)), name
    for st in [fused] + eager + graphed:
        st.close()
