"""The low part of the far numerator does its job.

The state comparisons in the parity tests bound T^ at 1e-5 relative, far
above one f32 rounding, so they cannot tell a working low part from a broken
one (a low part stored in the wrong half of its word, or dropped).  Two
checks that can:

* Closed form.  With every prompt query zero, every query landmark is zero,
  every far logit is exactly 0 and every far weight exactly 1 (the running
  maximum is 0 from the first absorbed key on; nystrom.rs, far_insert), so
  each row of T^ is the plain sum of the absorbed values and Z^ their count.
  Integer prompt values make the seal's sums exact; small non-integer decode
  values then make every token's addition round.  hi + lo must match the f64
  sum far more closely than hi alone.
* Residual shape.  After a seal whose key blocks all add comparable amounts,
  each decoded low part is the rounding residual of its high part: at most
  about half an ulp, and a sizeable fraction of an ulp for many elements, in
  every column half (the tensor-core replay stores the two halves from
  different threads).
"""
import numpy as np
import pytest

from streaming_nystr_landmark_gb300 import nys

pytestmark = pytest.mark.gpu


def _ulp(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(x).astype(np.float64)


@pytest.mark.parametrize("heads,d,dv", [(2, 32, 32), (3, 20, 20)])
def test_decode_low_part_tracks_exact_sums(cuda_device, heads, d, dv):
    """(2, 32, 32) runs the TMA decode kernel, (3, 20, 20) the general one."""
    import torch
    G, m, w, sink, t, steps = 6, 8, 16, 4, 64, 300
    rng = np.random.default_rng(123)
    q = np.zeros((G, heads, t, d), np.float32)
    k = rng.standard_normal((G, t, d)).astype(np.float32)
    v = rng.integers(-8, 9, size=(G, t, dv)).astype(np.float32)
    st = nys.NystromStates(m, w, sink, heads, d, dv, G, 0, cuda_device)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    st.seal(dev(q), dev(k), dev(v))
    # Keys sink .. t-w-1 were absorbed by the seal; decode token n absorbs
    # the key w positions before it.
    hist = [v[:, j] for j in range(t)]
    absorbed = [v[:, j].astype(np.float64) for j in range(sink, t - w)]
    out = torch.empty((G, heads, dv), device=cuda_device)
    for n in range(steps):
        tq = rng.standard_normal((G, heads, d)).astype(np.float32)
        tk = rng.standard_normal((G, d)).astype(np.float32)
        tv = (rng.standard_normal((G, dv)) / 16).astype(np.float32)   # sums round
        st.step(dev(tq), dev(tk), dev(tv), out)
        absorbed.append(hist[t + n - w].astype(np.float64))
        hist.append(tv)
    ref = np.sum(absorbed, axis=0)                       # [G][dv], exact in f64
    torch.cuda.synchronize(cuda_device)
    z = st.region("z_hat").cpu().numpy()
    m_max = st.region("m_max").cpu().numpy()
    assert np.all(m_max == 0.0) and np.all(z == len(absorbed))
    hi = st.region("t_hat").double().cpu().numpy()
    full = st.far_numerator()
    err_hi = np.abs(hi - ref[:, None, None, :])
    err_full = np.abs(full - ref[:, None, None, :])
    # Each token's addition rounds hi by up to half an ulp and leaves the
    # residual in lo; lo is stored as bf16 (eight significant bits) at every
    # token, and those storage errors accumulate.  A CPU emulation of this
    # scenario gives err_full ~0.04 err_hi on average and at most ~0.02 ulp
    # of the row's largest sum; a lost or scrambled low part gives ~1 or more.
    assert err_full.mean() < 0.2 * err_hi.mean(), (err_hi.mean(), err_full.mean())
    row_ulp = _ulp(np.abs(ref).max(axis=1))[:, None, None, None]
    assert np.all(err_full <= 0.25 * row_ulp), float((err_full / row_ulp).max())
    st.close()


@pytest.mark.parametrize("t", [256, 600])
def test_sealed_low_parts_are_rounding_residuals(cuda_device, t):
    """t = 256 absorbs 236 keys on the CUDA-core replay, t = 600 absorbs 580
    on the tensor-core replay.  Small queries keep every weight near 1, so
    every key block adds a comparable amount and each fold rounds."""
    import torch
    G, H, d, dv, m, w, sink = 4, 2, 64, 64, 32, 16, 4
    rng = np.random.default_rng(t)
    q = (0.05 * rng.standard_normal((G, H, t, d))).astype(np.float32)
    k = rng.standard_normal((G, t, d)).astype(np.float32)
    v = rng.standard_normal((G, t, dv)).astype(np.float32)
    st = nys.NystromStates(m, w, sink, H, d, dv, G, 0, cuda_device)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda_device)
    st.seal(dev(q), dev(k), dev(v))
    torch.cuda.synchronize(cuda_device)
    hi = st.region("t_hat").double().cpu().numpy()
    lo = st.far_numerator() - hi
    st.close()
    keep = np.abs(hi) > 1e-30
    ratio = np.where(keep, np.abs(lo) / _ulp(np.where(keep, hi, 1.0)), 0.0)
    # A rounding residual is about half an ulp at most (one ulp allows for
    # Fast2Sum's last fold when the added block outweighs the sum).  With few
    # folds many residuals are exactly zero -- two f32 sums of similar size
    # often add exactly -- and the rest are a sizeable fraction of an ulp
    # (measured: 45% of them above 0.05 ulp after four folds, 80% after ten).
    # A lost low part, or one stored at a wrong scale, leaves none there.
    assert np.all(ratio <= 1.0), float(ratio.max())
    half = dv // 2
    for cols in (slice(0, half), slice(half, dv)):
        r = ratio[..., cols][keep[..., cols]]
        assert np.mean(r > 0.05) > 0.25, (cols, float(np.mean(r > 0.05)))
