"""The LayerKvCache o1 lifecycle (nys_o1_*): collect the prompt's queries one
position at a time, seal when the page's preconditions hold, then decode.

A layer sealed through the lifecycle must hold exactly the states a direct
nys_seal of the same groups builds, decode identically, and match the fp64
oracle run per (sequence, KV head) on the layer's own tensors; every failed
precondition must leave the layer unsealed (exact), as o1_seal returns false."""
import numpy as np
import pytest

from oracle import NystromOracle
from parity_util import step_oracles_and_compare

from streaming_nystr_landmark_gb300 import nys
from streaming_nystr_landmark_gb300.workloads import Workload, host_prompt_batch, host_token_batch

pytestmark = pytest.mark.gpu

B, NH, NKV, D, M, W, SINK, T = 3, 4, 2, 32, 8, 16, 4, 64
HPK = NH // NKV


def _inputs(cuda_device):
    import torch
    wl = Workload("o1", HPK, D, D, M, W, SINK, 0, T, 8, 1, 1, B * NKV, "unit2", seed=51)
    q, k, v, gens = host_prompt_batch(wl, range(B * NKV))   # groups g = b*NKV + kvh
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    # the layer's view: q_all[pos] = [B][NH][D], head h of sequence b is
    # query head h % HPK of group b*NKV + h // HPK
    q_layer = q.reshape(B, NKV, HPK, T, D).reshape(B, NH, T, D)
    return wl, gens, dev, q, k, v, q_layer


def test_lifecycle_matches_direct_seal_and_decode(cuda_device):
    import torch
    wl, gens, dev, q, k, v, q_layer = _inputs(cuda_device)
    layer = nys.O1Layer(M, W, SINK, D, D, B, NH, NKV, max_prompt=100, device=cuda_device)
    with pytest.raises(nys.NysError) as ei:
        layer.step(*[torch.zeros(s, device=cuda_device) for s in
                     ((B, NH, D), (B, NKV, D), (B, NKV, D), (B, NH, D))])
    assert ei.value.code == nys.NYS_E_NOT_SEALED
    for p in range(T):
        layer.push_q(dev(q_layer[:, :, p, :]))
    assert layer.memory_bytes() == B * NH * T * D * 4          # the trace so far
    assert not layer.sealed()
    assert layer.seal(dev(k.reshape(B, NKV, T, D)), dev(v.reshape(B, NKV, T, D)))
    assert layer.sealed()
    direct = nys.NystromStates(M, W, SINK, HPK, D, D, B * NKV, 0, cuda_device)
    direct.seal(dev(q), dev(k), dev(v))
    assert layer.memory_bytes() == nys.nys_memory_bytes(direct.cfg, B * NKV)
    layer.push_q(dev(q_layer[:, :, 0, :]))                     # no-op once sealed
    # the layer's states are the direct states, byte for byte
    import ctypes
    sp = ctypes.c_void_p(0)
    assert nys._lib.nys_o1_states(layer.handle, ctypes.byref(sp)) == 0
    base, lay = nys.nys_layout_of(sp.value)
    torch.cuda.synchronize()

    class _Raw:  # a view of the library-owned state buffer
        def __init__(self, ptr, n):
            self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1",
                                             "data": (ptr, False), "version": 2}

    ours = torch.as_tensor(_Raw(base, lay.total_bytes), device=cuda_device)
    theirs = direct.buf[direct._off:direct._off + lay.total_bytes]
    assert torch.equal(ours, theirs)
    # The oracle side reads the layer's own tensors and applies the page's
    # rule itself (Struct LayerKvCache, o1_step: query head h belongs to KV
    # group h / hpk): one oracle per (sequence b, KV head j), fed query heads
    # j*hpk .. j*hpk + hpk - 1 of sequence b.
    k_layer = k.reshape(B, NKV, T, D)
    v_layer = v.reshape(B, NKV, T, D)
    oracles = []
    for b in range(B):
        for j in range(NKV):
            o = NystromOracle(M, W, SINK, HPK, 0)
            o.prefill(np.stack([q_layer[b, h] for h in range(NH) if h // HPK == j]),
                      k_layer[b, j], v_layer[b, j])
            oracles.append(o)
    for n in range(8):
        tq, tk, tv = host_token_batch(gens, n)                   # per group
        q_all = dev(tq.reshape(B, NKV, HPK, D).reshape(B, NH, D))
        kn, vn = dev(tk.reshape(B, NKV, D)), dev(tv.reshape(B, NKV, D))
        out_l = torch.empty((B, NH, D), device=cuda_device)
        layer.step(q_all, kn, vn, out_l)
        out_d = torch.empty((B * NKV, HPK, D), device=cuda_device)
        direct.step(dev(tq), dev(tk), dev(tv), out_d)
        assert torch.equal(out_l.reshape(-1), out_d.reshape(-1)), n
        # Oracle inputs and outputs rebuilt from the layer view by the rule.
        ql, kl, vl = q_all.cpu().numpy(), kn.cpu().numpy(), vn.cpu().numpy()
        got = out_l.cpu().numpy()
        oq = np.stack([np.stack([ql[b, h] for h in range(NH) if h // HPK == j])
                       for b in range(B) for j in range(NKV)])
        og = np.stack([np.stack([got[b, h] for h in range(NH) if h // HPK == j])
                       for b in range(B) for j in range(NKV)])
        step_oracles_and_compare(oracles, oq, kl.reshape(B * NKV, D),
                                 vl.reshape(B * NKV, D), [og])
    layer.close()
    direct.close()


@pytest.mark.parametrize("case", ["fan_out", "short_trace", "not_dense", "no_exact_room"])
def test_failed_preconditions_keep_the_layer_exact(cuda_device, case):
    wl, gens, dev, q, k, v, q_layer = _inputs(cuda_device)
    nh, t = (3 if case == "fan_out" else NH), T
    kk, vv = k, v
    if case == "no_exact_room":
        t = 20                                                   # <= w + sink + 8
        kk, vv = k[:, :t], v[:, :t]
    layer = nys.O1Layer(M, W, SINK, D, D, B, nh, NKV, max_prompt=100, device=cuda_device)
    pushes = t - 1 if case == "short_trace" else t
    for p in range(pushes):
        layer.push_q(dev(np.ascontiguousarray(q_layer[:, :nh, p, :])))
    ok = layer.seal(dev(kk.reshape(B, NKV, t, D)), dev(vv.reshape(B, NKV, t, D)),
                    kv_dense=(case != "not_dense"))
    assert not ok and not layer.sealed()
    assert layer.memory_bytes() == B * nh * pushes * D * 4       # trace kept
    layer.close()


def test_trace_capacity(cuda_device):
    import torch
    layer = nys.O1Layer(M, W, SINK, D, D, 1, 2, 1, max_prompt=3, device=cuda_device)
    z = torch.zeros((1, 2, D), device=cuda_device)
    for _ in range(3):
        layer.push_q(z)
    with pytest.raises(nys.NysError) as ei:
        layer.push_q(z)
    assert ei.value.code == nys.NYS_E_RANGE
    layer.close()
