"""nys_seal_static -- the seal that allocates nothing -- against nys_seal.

Some callers cannot allocate device memory once they are running: a serving
process that reserved all of its GPU memory at start-up, or a host
application whose own allocator must see every device buffer.  For them the
library offers nys_seal_static, which keeps the seal's f64 workspace in a
fixed 4 MiB array inside the library instead of calling cudaMallocAsync.  It
must seal exactly as nys_seal does.  This file is collected last on purpose,
so that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

from parity_util import LANDMARK_TOL, MU_TOL, OUT_TOL, row_err

pytestmark = pytest.mark.gpu


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
        nys.nys_seal_static(sta.handle, 0, n, wl.t, q.data_ptr(), k.data_ptr(),
                            v.data_ptr(), stream)
        torch.cuda.synchronize(cuda_device)
        for name in ("win_k", "win_v", "sink_k", "sink_v", "ints", "far_len"):
            assert torch.equal(ref.region(name), sta.region(name)), (call, name)
        for name in ("k_tilde", "q_tilde"):
            a, b = ref.region(name).double(), sta.region(name).double()
            scale = a.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
            assert float(((a - b).abs() / scale).max()) <= LANDMARK_TOL, (call, name)
        a, b = ref.region("mu").double(), sta.region("mu").double()
        rel = (a - b).flatten(2).norm(dim=2) / a.flatten(2).norm(dim=2)
        assert float(rel.max()) <= MU_TOL, call
        for got, want in ((sta.far_numerator(), ref.far_numerator()),
                          (sta.far_denominator(), ref.far_denominator())):
            assert np.abs(got - want).max() <= 1e-5 * np.abs(want).max(), call
        # The decode outputs of both states agree too.
        out_r = torch.empty((n, wl.heads_per_kv, wl.dv), device=cuda_device)
        out_s = torch.empty_like(out_r)
        for step in range(3):
            tq, tk, tv = [torch.from_numpy(a).to(cuda_device)
                          for a in host_token_batch(gens, step)]
            ref.step(tq, tk, tv, out_r)
            sta.step(tq, tk, tv, out_s)
            r, s = out_r.cpu().numpy(), out_s.cpu().numpy()
            for g in range(n):
                for h in range(wl.heads_per_kv):
                    assert row_err(s[g, h].astype(np.float64),
                                   r[g, h].astype(np.float64)) <= OUT_TOL
        ref.close()
        sta.close()


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
