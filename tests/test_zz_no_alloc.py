"""nys_seal_static -- the seal that allocates nothing -- against nys_seal.

Some callers cannot allocate device memory once they are running: a serving
process that reserved all of its GPU memory at start-up, or a host
application whose own allocator must see every device buffer.  For them the
library offers nys_seal_static, which keeps the seal's f64 workspace in a
fixed 4 MiB array inside the library instead of calling cudaMallocAsync.  It
runs the same deterministic kernels as nys_seal, so the states it builds must
be bit-identical, and after its first call on a device (which looks the
array's address up) it must not change the device's free memory at all.
This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import pytest

pytestmark = pytest.mark.gpu

REGIONS = ("win_k", "win_v", "sink_k", "sink_v", "k_tilde", "q_tilde", "mu",
           "t_hat", "t_lo", "z_hat", "z_lo", "m_max", "far_len", "ints")


def _assert_same_state(ref, sta, what):
    import torch
    for name in REGIONS:
        assert torch.equal(ref.region(name), sta.region(name)), (what, name)


def test_static_seal_matches_allocating_seal_twice_in_a_row(cuda_device):
    import torch
    from streaming_nystr_landmark_gb300 import nys
    from streaming_nystr_landmark_gb300.workloads import (WORKLOADS,
                                                          host_prompt_batch,
                                                          host_token_batch)

    # 96 KiB of workspace per group: 100 groups need three passes through
    # the 4 MiB array within one call.
    wl = WORKLOADS["batch64"]
    n = 100
    geo = (wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d, wl.dv, n, wl.rect,
           cuda_device)
    for call, first_group in enumerate((0, 5000)):
        ref = nys.NystromStates(*geo)
        sta = nys.NystromStates(*geo)
        q, k, v, gens = host_prompt_batch(wl, range(first_group, first_group + n))
        q, k, v = [torch.from_numpy(a).to(cuda_device) for a in (q, k, v)]
        ref.seal(q, k, v)
        stream = torch.cuda.current_stream(cuda_device).cuda_stream
        torch.cuda.synchronize(cuda_device)
        free_before, _ = torch.cuda.mem_get_info(cuda_device)
        nys.nys_seal_static(sta.handle, 0, n, wl.t, q.data_ptr(), k.data_ptr(),
                            v.data_ptr(), stream)
        torch.cuda.synchronize(cuda_device)
        free_after, _ = torch.cuda.mem_get_info(cuda_device)
        if call > 0:
            # The first call on the device may load the library's module
            # (and with it the static array); later calls allocate nothing.
            assert free_after == free_before, (free_before, free_after)
        _assert_same_state(ref, sta, call)
        # Identical states decode identically.
        out_r = torch.empty((n, wl.heads_per_kv, wl.dv), device=cuda_device)
        out_s = torch.empty_like(out_r)
        for step in range(3):
            tq, tk, tv = [torch.from_numpy(a).to(cuda_device)
                          for a in host_token_batch(gens, step)]
            ref.step(tq, tk, tv, out_r)
            sta.step(tq, tk, tv, out_s)
            assert torch.equal(out_r, out_s), (call, step)
        ref.close()
        sta.close()


def test_static_seal_takes_short_prompts_like_nys_seal(cuda_device):
    """A prompt with t <= w + sink + 8 on a handle with an exact region is
    sealed in exact-only mode by both entry points, with identical states;
    without an exact region both refuse it with the same code."""
    import torch
    from streaming_nystr_landmark_gb300 import nys
    from streaming_nystr_landmark_gb300.workloads import (Workload,
                                                          host_prompt_batch,
                                                          host_token_batch)

    wl = Workload("short", 2, 32, 32, 8, 16, 4, 0, 20, 4, 1, 1, 4, "unit2",
                  seed=17)
    geo = (wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d, wl.dv, 4, wl.rect,
           cuda_device)
    q, k, v, gens = host_prompt_batch(wl, range(4))
    q, k, v = [torch.from_numpy(a).to(cuda_device) for a in (q, k, v)]
    stream = torch.cuda.current_stream(cuda_device).cuda_stream
    ref = nys.NystromStates(*geo, exact_cap=64)
    sta = nys.NystromStates(*geo, exact_cap=64)
    ref.seal(q, k, v)
    nys.nys_seal_static(sta.handle, 0, 4, wl.t, q.data_ptr(), k.data_ptr(),
                        v.data_ptr(), stream)
    torch.cuda.synchronize(cuda_device)
    for name in REGIONS + ("exact_k", "exact_v"):
        assert torch.equal(ref.region(name), sta.region(name)), name
    out_r = torch.empty((4, wl.heads_per_kv, wl.dv), device=cuda_device)
    out_s = torch.empty_like(out_r)
    for step in range(3):
        tq, tk, tv = [torch.from_numpy(a).to(cuda_device)
                      for a in host_token_batch(gens, step)]
        ref.step(tq, tk, tv, out_r)
        sta.step(tq, tk, tv, out_s)
        assert torch.equal(out_r, out_s), step
    ref.close()
    sta.close()
    bare = nys.NystromStates(*geo)
    for fn in (nys.nys_seal, nys.nys_seal_static):
        with pytest.raises(nys.NysError) as ei:
            fn(bare.handle, 0, 4, wl.t, q.data_ptr(), k.data_ptr(),
               v.data_ptr(), stream)
        assert ei.value.code == nys.NYS_E_EXACT_ONLY
    bare.close()


def test_static_seal_rejects_workspace_beyond_scratch(cuda_device):
    from streaming_nystr_landmark_gb300 import nys
    # (1 + 64) * 64 * 128 * 8 bytes = 4.06 MiB per group > 4 MiB.
    import torch
    st = nys.NystromStates(64, 16, 4, 64, 128, 128, 1, 0, cuda_device)
    t = 600
    q = torch.zeros((1, 64, t, 128), device=cuda_device)
    k = torch.zeros((1, t, 128), device=cuda_device)
    v = torch.zeros((1, t, 128), device=cuda_device)
    with pytest.raises(nys.NysError) as ei:
        nys.nys_seal_static(st.handle, 0, 1, t, q.data_ptr(), k.data_ptr(),
                            v.data_ptr())
    assert ei.value.code == nys.NYS_E_SCRATCH
    assert "static scratch" in nys.nys_strerror(nys.NYS_E_SCRATCH)
    st.close()
