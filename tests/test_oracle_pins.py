"""Pins of the fp64 oracle against things other than itself.

Each test ties one part of the oracle to a fact the operator's pages fix or to
mathematics that holds independently of it: golden tables worked by hand from
the rules in nystrom.rs, closed forms, brute-force softmax attention, an SVD
formula, and a second (materialised-weights) formulation of the operator.  A
plausible slip in the oracle -- a dropped term, a wrong sign or index, a
transposed M, an off-by-one in the ring or the far set -- fails at least one.
"""
import math

import numpy as np
import pytest

from conftest import read_golden
import oracle
from oracle import (AGGREGATE, FM, NystromOracle, direct_output,
                    effective_landmarks, is_exact_only, ridge_pinv,
                    cholesky_lower, score_scale, seg_means)

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def softmax_attention(q, keys, values, scale):
    """Textbook exact attention: softmax over all keys (fsum for stability)."""
    logits = [float(np.dot(q, kj)) * scale for kj in keys]
    mx = max(logits)
    w = [math.exp(x - mx) for x in logits]
    z = math.fsum(w)
    return np.array([math.fsum(wi * float(vj[c]) for wi, vj in zip(w, values))
                     for c in range(values.shape[1])]) / z


def _rand_prompt(rng, heads, t, d, dv, kshift=0.0):
    q = rng.standard_normal((heads, t, d)).astype(np.float32)
    k = (rng.standard_normal((t, d)) + kshift).astype(np.float32)
    v = rng.standard_normal((t, dv)).astype(np.float32)
    return q, k, v


# ---------------------------------------------------------------- tables
def test_constants_match_golden():
    rows = {r[0]: r[1] for r in read_golden("constants.txt")}
    assert oracle.RIDGE_REL == float(rows["RIDGE_REL"])
    assert oracle.DEN_EPS == float(rows["DEN_EPS"])
    assert oracle.EXACT_SLACK == int(rows["EXACT_SLACK"])
    assert oracle.RIDGE_TRIES == int(rows["RIDGE_TRIES"])
    assert (oracle.DEFAULT_M, oracle.DEFAULT_W, oracle.DEFAULT_SINK) == (
        int(rows["DEFAULT_M"]), int(rows["DEFAULT_W"]), int(rows["DEFAULT_SINK"]))
    assert rows["DEFAULT_RECT"] == "aggregate" and oracle.AGGREGATE == 0
    # Growth factor: after the fallback the ridge has been multiplied by
    # ten once per failed attempt.
    r = ridge_pinv(np.array([[np.inf, 0.0], [0.0, 1.0]]))
    assert r.fallback and r.tries == oracle.RIDGE_TRIES + 1
    assert r.lam == np.inf  # inf * 10**12 stays inf; finite case below
    r = ridge_pinv(np.array([[np.nan, 1.0], [1.0, 1.0]]))
    tiny = np.finfo(np.float64).tiny
    base = oracle.RIDGE_REL * tiny
    assert r.fallback
    assert r.lam == pytest.approx(base * float(rows["RIDGE_GROWTH"]) ** 12,
                                  rel=1e-12)


def test_landmark_budget_table():
    for t, m, m_eff in read_golden("landmark_budget.txt"):
        assert effective_landmarks(int(t), int(m)) == int(m_eff), (t, m)


def test_exact_only_threshold_table():
    for t, w, s, flag in read_golden("exact_only_threshold.txt"):
        assert is_exact_only(int(t), int(w), int(s)) == bool(int(flag))


def test_seg_means_against_hand_bounds():
    rng = np.random.default_rng(7)
    xs = rng.standard_normal((70, 5)).astype(np.float32)
    got = seg_means(xs, 8)
    for i, lo, hi in read_golden("seg_bounds_t70_m8.txt"):
        i, lo, hi = int(i), int(lo), int(hi)
        for c in range(5):
            want = math.fsum(float(x) for x in xs[lo:hi, c]) / (hi - lo)
            assert got[i, c] == pytest.approx(want, rel=1e-14, abs=1e-15)


@pytest.mark.parametrize("t,m", [(64, 8), (70, 8), (256, 32), (100, 7), (9, 4)])
def test_seg_means_partition(t, m):
    """Segments tile [0, t) in order; sizes differ by at most one; the means
    reweighted by segment size give back the column sums."""
    xs = np.random.default_rng(t * m).standard_normal((t, 3))
    bounds = [(i * t) // m for i in range(m + 1)]
    sizes = np.diff(bounds)
    assert bounds[0] == 0 and bounds[-1] == t
    assert sizes.min() >= 1 and sizes.max() - sizes.min() <= 1
    got = seg_means(xs, m)
    np.testing.assert_allclose((got * sizes[:, None]).sum(0), xs.sum(0),
                               rtol=1e-12, atol=1e-12)


def test_score_scale_is_f32():
    assert score_scale(128) == float(np.float32(1) / np.sqrt(np.float32(128)))
    assert score_scale(128) != 1.0 / math.sqrt(128.0)
    assert score_scale(64) == 0.125


# ---------------------------------------------------------------- pinv
def test_cholesky_against_library():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((9, 9))
    spd = a @ a.T + 9 * np.eye(9)
    np.testing.assert_allclose(cholesky_lower(spd), np.linalg.cholesky(spd),
                               rtol=1e-12, atol=1e-12)
    assert cholesky_lower(np.array([[1.0, 2.0], [2.0, 1.0]])) is None
    assert cholesky_lower(np.array([[0.0, 0.0], [0.0, 1.0]])) is None
    assert cholesky_lower(np.array([[np.nan, 0.0], [0.0, 1.0]])) is None
    assert cholesky_lower(np.array([[np.inf, 0.0], [0.0, 1.0]])) is None


@pytest.mark.parametrize("n,seed", [(4, 0), (8, 1), (32, 2), (64, 3)])
def test_ridge_pinv_matches_svd_formula(n, seed):
    """M = V diag(s/(s^2+lam)) U^T for A = U diag(s) V^T, lam as stated."""
    rng = np.random.default_rng(seed)
    qt = rng.standard_normal((n, 16)) / math.sqrt(8)
    kt = rng.standard_normal((n, 16)) / math.sqrt(8) + 0.3
    a = np.exp(qt @ kt.T * 0.25)
    r = ridge_pinv(a)
    assert r.tries == 1 and not r.fallback
    lam_expected = 1e-6 * np.trace(a.T @ a) / n
    assert r.lam == pytest.approx(lam_expected, rel=1e-13)
    u, s, vt = np.linalg.svd(a)
    ref = vt.T @ np.diag(s / (s * s + r.lam)) @ u.T
    scale = np.abs(ref).max()
    assert np.abs(r.m - ref).max() <= 1e-7 * scale
    # Residual identity M A = I - lam (A^T A + lam I)^-1.
    resid = np.eye(n) - r.lam * np.linalg.inv(a.T @ a + r.lam * np.eye(n))
    assert np.abs(r.m @ a - resid).max() <= 1e-6


def test_ridge_pinv_closed_forms():
    for alpha in (0.5, 2.0, 7.0):
        r = ridge_pinv(alpha * np.eye(4))
        np.testing.assert_allclose(r.m, np.eye(4) / (alpha * (1 + 1e-6)),
                                   rtol=1e-12)
    n = 5
    r = ridge_pinv(np.ones((n, n)))          # rank one: J
    lam = 1e-6 * n
    assert r.lam == pytest.approx(lam, rel=1e-14)
    np.testing.assert_allclose(r.m, np.ones((n, n)) / (n * n + lam), rtol=1e-9)


def test_ridge_pinv_fallback_paths():
    r = ridge_pinv(np.array([[np.inf, 0.0], [0.0, 1.0]]))
    assert r.fallback and np.all(r.m == 0.0)
    r = ridge_pinv(np.array([[np.nan, 1.0], [1.0, 1.0]]))
    tiny = np.finfo(np.float64).tiny
    assert r.fallback
    np.testing.assert_array_equal(r.m, np.eye(2) / tiny)


def test_ridge_pinv_duplicate_landmarks():
    """Two identical landmark rows make Au singular; the ridge keeps the
    solve well posed on the first attempt and M A stays a projector-like
    contraction (the SVD formula still holds)."""
    rng = np.random.default_rng(5)
    qt = rng.standard_normal((6, 8)) * 0.3
    qt[3] = qt[1]
    a = np.exp(qt @ qt.T)
    r = ridge_pinv(a)
    assert r.tries == 1 and np.all(np.isfinite(r.m))
    u, s, vt = np.linalg.svd(a)
    ref = vt.T @ np.diag(s / (s * s + r.lam)) @ u.T
    assert np.abs(r.m - ref).max() <= 1e-6 * np.abs(ref).max()


# ---------------------------------------------------------------- whole operator
@pytest.mark.parametrize("t,w,sink,steps,heads", [
    (28, 16, 4, 12, 1), (20, 16, 4, 30, 2), (9, 1, 0, 5, 1), (140, 128, 4, 3, 2)])
def test_exact_only_is_softmax_attention(t, w, sink, steps, heads):
    """t <= w + sink + 8: every key stays exact, so each output is plain
    softmax attention over all keys so far, before and after decode tokens."""
    rng = np.random.default_rng(t + steps)
    d = dv = 8
    q, k, v = _rand_prompt(rng, heads, t, d, dv, kshift=0.5)
    o = NystromOracle(m=8, w=w, sink=sink, heads=heads)
    o.prefill(q, k, v)
    assert o.exact_only and o.far_len(0) == 0
    keys, vals = list(k.astype(np.float64)), list(v.astype(np.float64))
    for n in range(steps):
        qa = rng.standard_normal((heads, d)).astype(np.float32)
        kn = rng.standard_normal(d).astype(np.float32)
        vn = rng.standard_normal(dv).astype(np.float32)
        out = o.step(qa, kn, vn)
        keys.append(kn.astype(np.float64))
        vals.append(vn.astype(np.float64))
        for h in range(heads):
            ref = softmax_attention(qa[h].astype(np.float64), np.array(keys),
                                    np.array(vals), score_scale(d))
            np.testing.assert_allclose(out[h], ref, rtol=1e-12, atol=1e-13)


def _run_oa_ob(rect, sink, heads=2, t=56, d=12, dv=10, m=8, w=9, steps=14,
               seed=0, kshift=0.7):
    rng = np.random.default_rng(seed)
    q, k, v = _rand_prompt(rng, heads, t, d, dv, kshift=kshift)
    o = NystromOracle(m=m, w=w, sink=sink, heads=heads, rect=rect)
    o.prefill(q, k, v)
    assert not o.exact_only
    k_hist = [x for x in k.astype(np.float64)]
    v_hist = [x for x in v.astype(np.float64)]
    results = []
    for n in range(steps):
        qa = rng.standard_normal((heads, d)).astype(np.float32)
        kn = (rng.standard_normal(d) + kshift).astype(np.float32)
        vn = rng.standard_normal(dv).astype(np.float32)
        out = o.step(qa, kn, vn)
        k_hist.append(kn.astype(np.float64))
        v_hist.append(vn.astype(np.float64))
        for h in range(heads):
            hs = o.hs[h]
            ref, far_w, keep = direct_output(
                qa[h], np.array(k_hist), np.array(v_hist), sink, w,
                o.k_tilde, hs.q_tilde, hs.mu, o.scale, rect)
            results.append((out[h], ref, far_w, keep, o.diags[-1][h]))
    return o, results


@pytest.mark.parametrize("rect", [AGGREGATE, FM])
@pytest.mark.parametrize("sink", [0, 4])
def test_streamed_equals_materialised(rect, sink):
    """The ring + delayed insertion + running-max far field + joint shift
    (streaming form) equals the explicitly materialised F M E far weights over
    the far set, for sink = 0 (the sink-free definition, near = last w keys)
    and sink = 4."""
    _, res = _run_oa_ob(rect, sink)
    for out, ref, _, keep, dg in res:
        assert dg.have_far == keep
        np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_fm_far_weights_nonnegative():
    _, res = _run_oa_ob(FM, 4, seed=3)
    for _, _, far_w, _, _ in res:
        assert far_w.size > 0 and np.all(far_w >= 0.0)


def test_aggregate_drops_far_iff_negative():
    """The guard keeps the far field exactly when the materialised far mass
    sum_Phi w^_j is >= 0; a dropped row is exact softmax over the near set
    (sinks + window) alone.  Running the same inputs with M and with -M makes
    both branches occur."""
    seen = set()
    for flip in (1.0, -1.0):
        rng = np.random.default_rng(11)
        heads, t, d, dv, m, w, sink = 1, 60, 8, 6, 8, 10, 3
        q, k, v = _rand_prompt(rng, heads, t, d, dv, kshift=0.4)
        o = NystromOracle(m=m, w=w, sink=sink, heads=heads)
        o.prefill(q, k, v)
        o.hs[0].mu = flip * o.hs[0].mu
        k_hist = list(k.astype(np.float64))
        v_hist = list(v.astype(np.float64))
        for n in range(12):
            qa = rng.standard_normal((1, d)).astype(np.float32)
            kn = rng.standard_normal(d).astype(np.float32)
            vn = rng.standard_normal(dv).astype(np.float32)
            out = o.step(qa, kn, vn)
            k_hist.append(kn.astype(np.float64))
            v_hist.append(vn.astype(np.float64))
            ref, far_w, keep = direct_output(
                qa[0], np.array(k_hist), np.array(v_hist), sink, w,
                o.k_tilde, o.hs[0].q_tilde, o.hs[0].mu, o.scale, AGGREGATE)
            assert keep == (far_w.sum() >= 0) == o.diags[-1][0].have_far
            seen.add(keep)
            np.testing.assert_allclose(out[0], ref, rtol=1e-11, atol=1e-13)
            if not keep:
                p = len(k_hist) - 1
                near = [j for j in range(p + 1) if j < sink or j > p - w]
                exact_near = softmax_attention(
                    qa[0].astype(np.float64), np.array(k_hist)[near],
                    np.array(v_hist)[near], o.scale)
                np.testing.assert_allclose(out[0], exact_near, rtol=1e-11,
                                           atol=1e-13)
    assert seen == {True, False}


@pytest.mark.parametrize("t,w,sink,heads", [(64, 16, 4, 1), (50, 9, 0, 3),
                                            (300, 128, 4, 2)])
def test_delayed_insertion_counts(t, w, sink, heads):
    """far_len equals the number of evictions -- t - sink - w after the seal,
    plus one per decode token -- for EVERY head, never heads times it; the
    ring head advances once per key."""
    rng = np.random.default_rng(t)
    d = dv = 4
    q, k, v = _rand_prompt(rng, heads, t, d, dv)
    o = NystromOracle(m=8, w=w, sink=sink, heads=heads)
    o.prefill(q, k, v)
    for n in range(0, 20):
        if n:
            o.step(rng.standard_normal((heads, d)), rng.standard_normal(d),
                   rng.standard_normal(dv))
        for h in range(heads):
            assert o.far_len(h) == t - sink - w + n
        assert o.win_len == w
        assert o.win_head == (t - sink + n) % w


def test_running_max_matches_unshifted_sums():
    """T^_i e^{m_i} and Z^_i e^{m_i} equal the plain (unshifted) f64 sums of
    exp(l_ij) and exp(l_ij) v_j over the far set, where those do not
    overflow."""
    rng = np.random.default_rng(2)
    heads, t, d, dv, m, w, sink = 2, 80, 6, 5, 8, 12, 2
    q, k, v = _rand_prompt(rng, heads, t, d, dv, kshift=1.0)
    o = NystromOracle(m=m, w=w, sink=sink, heads=heads)
    o.prefill(q, k, v)
    kk, vv = list(k.astype(np.float64)), list(v.astype(np.float64))
    for n in range(10):
        kn = rng.standard_normal(d).astype(np.float32)
        vn = rng.standard_normal(dv).astype(np.float32)
        o.step(rng.standard_normal((heads, d)), kn, vn)
        kk.append(kn.astype(np.float64))
        vv.append(vn.astype(np.float64))
    p = len(kk) - 1
    far = [j for j in range(sink, p - w + 1)]
    for hs in o.hs:
        logits = hs.q_tilde @ np.array(kk)[far].T * o.scale      # [m][|far|]
        z_ref = np.exp(logits).sum(axis=1)
        t_ref = np.exp(logits) @ np.array(vv)[far]
        np.testing.assert_allclose(hs.z_hat * np.exp(hs.m_max), z_ref,
                                   rtol=1e-12)
        np.testing.assert_allclose(hs.t_hat * np.exp(hs.m_max)[:, None], t_ref,
                                   rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hs.m_max, logits.max(axis=1), rtol=0,
                                   atol=0)


def test_running_max_survives_overflowing_logits():
    """Logits near 800 overflow exp() in f64; the shifted accumulators stay
    finite and the output is still a convex mix of values."""
    rng = np.random.default_rng(4)
    heads, t, d, dv, m, w, sink = 1, 48, 4, 3, 4, 8, 2
    q, k, v = _rand_prompt(rng, heads, t, d, dv)
    q = np.abs(q) * 0 + 40.0
    k = np.abs(k) * 0 + 10.0 + rng.random((t, d)).astype(np.float32)
    o = NystromOracle(m=m, w=w, sink=sink, heads=heads)
    o.prefill(q, k, v)
    hs = o.hs[0]
    logits = hs.q_tilde @ k[sink:t - w].astype(np.float64).T * o.scale
    assert logits.max() > 750
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp(logits).sum(axis=1)))
    assert np.all(np.isfinite(hs.z_hat)) and np.all(np.isfinite(hs.t_hat))
    assert np.all(hs.z_hat >= 1.0)        # the max term contributes exp(0)
    out = o.step(q[:, 0], k[-1], v[-1])
    assert np.all(np.isfinite(out))


def test_gqa_group_equals_independent_heads():
    """A group of H heads computes, per head, exactly what H single-head
    states fed the same keys/values and that head's own queries compute."""
    rng = np.random.default_rng(9)
    heads, t, d, dv = 3, 70, 8, 8
    q, k, v = _rand_prompt(rng, heads, t, d, dv, kshift=0.5)
    grp = NystromOracle(m=8, w=12, sink=4, heads=heads)
    grp.prefill(q, k, v)
    singles = []
    for h in range(heads):
        s = NystromOracle(m=8, w=12, sink=4, heads=1)
        s.prefill(q[h:h + 1], k, v)
        singles.append(s)
    for n in range(12):
        qa = rng.standard_normal((heads, d))
        kn, vn = rng.standard_normal(d), rng.standard_normal(dv)
        og = grp.step(qa, kn, vn)
        for h in range(heads):
            os_ = singles[h].step(qa[h:h + 1], kn, vn)
            np.testing.assert_allclose(og[h], os_[0], rtol=1e-14, atol=1e-15)
            assert grp.far_len(h) == singles[h].far_len(0)


def test_nystrom_reproduction_special_case():
    """Orthogonal landmarks: every prompt segment i holds keys alpha*e_i and
    queries beta*e_i, so K~ = alpha I, Q~ = beta I and Au = J + (c - 1) I with
    c = exp(alpha beta scale), which is well conditioned.  Every far key
    equals some landmark key, so the skeleton's far weights F M E_j equal the
    exact weights exp(q . k_j * scale) up to the ridge error
    lambda / (sigma_min^2 + lambda) ~ 1e-6; the output therefore equals exact
    softmax attention over ALL keys within that bound."""
    m = d = dv = 8
    t, w, sink = 64, 16, 4
    alpha = beta = 4.0
    eye = np.eye(d, dtype=np.float32)
    seg = np.repeat(np.arange(m), t // m)
    k = (alpha * eye[seg]).astype(np.float32)
    qh = (beta * eye[seg]).astype(np.float32)[None]
    rng = np.random.default_rng(21)
    v = rng.standard_normal((t, dv)).astype(np.float32)
    o = NystromOracle(m=m, w=w, sink=sink, heads=1)
    o.prefill(qh, k, v)
    np.testing.assert_allclose(o.k_tilde, alpha * np.eye(m), rtol=0, atol=0)
    np.testing.assert_allclose(o.hs[0].q_tilde, beta * np.eye(m), rtol=0,
                               atol=0)
    keys, vals = list(k.astype(np.float64)), list(v.astype(np.float64))
    worst = 0.0
    for n in range(40):
        qa = rng.standard_normal((1, d)).astype(np.float32)
        kn = (alpha * eye[rng.integers(m)]).astype(np.float32)
        vn = rng.standard_normal(dv).astype(np.float32)
        out = o.step(qa, kn, vn)
        keys.append(kn.astype(np.float64))
        vals.append(vn.astype(np.float64))
        ref = softmax_attention(qa[0].astype(np.float64), np.array(keys),
                                np.array(vals), o.scale)
        err = np.abs(out[0] - ref).max() / np.abs(ref).max()
        worst = max(worst, err)
    assert worst < 2e-5, worst
    assert o.far_len(0) == t - sink - w + 40
    # Au is symmetric here, so so is M: this case cannot tell M from its
    # transpose.  test_nystrom_reproduction_nonsymmetric below does.


def _nonsym_landmarks(m, alpha, beta, seed):
    """Key landmarks alpha*(I + 0.5 U) with U strictly upper triangular
    (entries in [0.5, 1]) and query landmarks beta*I: Au[i][j] =
    exp(q~_i . k~_j * scale) then has exp(0) = 1 below the diagonal and up to
    exp(alpha*beta*scale/2) above it -- far from symmetric, yet dominated by
    its diagonal and well conditioned."""
    rng = np.random.default_rng(seed)
    upper = np.triu(rng.uniform(0.5, 1.0, (m, m)), 1)
    k_t = (alpha * (np.eye(m) + 0.5 * upper)).astype(np.float32)
    q_t = (beta * np.eye(m)).astype(np.float32)
    return k_t, q_t


def test_nystrom_reproduction_nonsymmetric():
    """Nystrom reproduction with a NON-symmetric landmark kernel, which pins
    the orientation of M.  The prompt is segment-constant: segment b holds
    keys k~_b and queries q~_b, so seg_means returns exactly those rows.  The
    page builds Au with query landmarks as rows (nystrom.rs,
    ``NystromHead::seal``), solves G M = Au^T so that M's rows are key
    landmarks (``ridge_pinv``), and mixes u_b = sum_a F_a M[a][b]
    (``NystromHead::step``).  A far key equal to k~_b then gets the weight
    F (M Au) e_b, and M Au = (Au^T Au + lam I)^-1 Au^T Au is I up to the
    ridge error eps = lam / (sigma_min^2 + lam): every far weight equals the
    exact weight exp(q . k_j * scale) and the output equals softmax attention
    over all keys.  Building Au transposed, or mixing u = M F, replaces M Au
    by M^T Au, which is off the identity by several percent here.  Aggregate
    only: Fm clamps the negative entries of u = F Au^-1 and so leaves the
    reproduction identity by design."""
    rect = AGGREGATE
    m = d = dv = 8
    t, w, sink = 64, 16, 4
    alpha = beta = 4.0
    k_t, q_t = _nonsym_landmarks(m, alpha, beta, seed=5)
    seg = np.repeat(np.arange(m), t // m)
    k = k_t[seg]
    qh = q_t[seg][None]
    rng = np.random.default_rng(22)
    v = rng.standard_normal((t, dv)).astype(np.float32)
    o = NystromOracle(m=m, w=w, sink=sink, heads=1, rect=rect)
    o.prefill(qh, k, v)
    np.testing.assert_array_equal(o.k_tilde, k_t.astype(np.float64))
    np.testing.assert_array_equal(o.hs[0].q_tilde, q_t.astype(np.float64))
    scale = o.scale
    au = np.exp((q_t.astype(np.float64) @ k_t.astype(np.float64).T) * scale)
    assert np.abs(au - au.T).max() > 0.04 * np.abs(au).max()
    sv = np.linalg.svd(au, compute_uv=False)
    lam = 1e-6 * float(np.sum(au * au)) / m
    eps = lam / (sv[-1] ** 2 + lam)
    assert eps < 1e-5
    keys, vals = list(k.astype(np.float64)), list(v.astype(np.float64))
    worst = worst_w = 0.0
    for n in range(40):
        qa = rng.standard_normal((1, d)).astype(np.float32)
        kn = k_t[rng.integers(m)]
        vn = rng.standard_normal(dv).astype(np.float32)
        out = o.step(qa, kn, vn)
        keys.append(kn.astype(np.float64))
        vals.append(vn.astype(np.float64))
        q64 = qa[0].astype(np.float64)
        ref = softmax_attention(q64, np.array(keys), np.array(vals), scale)
        worst = max(worst, np.abs(out[0] - ref).max() / np.abs(ref).max())
        # The materialised far weights themselves are the exact ones.
        kh = np.array(keys)
        _, far_w, keep = direct_output(q64, kh, np.array(vals), sink, w,
                                       o.k_tilde, o.hs[0].q_tilde,
                                       o.hs[0].mu, scale, rect)
        p = kh.shape[0] - 1
        exact_w = np.exp((kh[sink:p - w + 1] @ q64) * scale)
        assert keep
        worst_w = max(worst_w,
                      np.abs(far_w - exact_w).max() / exact_w.max())
    # eps bounds |F (M Au - I) e_b| / |F|; M's f32 storage adds ~1e-7.
    assert worst_w < 10 * eps + 1e-6, (worst_w, eps)
    assert worst < 2e-5, worst
    assert o.far_len(0) == t - sink - w + 40


def test_joint_shift_covers_far_maxima():
    """Far logits ~800 above the near ones: the joint shift c_all must take
    the far maxima, or exp(f + m_max - c) overflows.  Prompt = small sink
    keys, huge far keys, then small window keys."""
    rng = np.random.default_rng(8)
    heads, t, d, dv, m, w, sink = 1, 40, 4, 3, 4, 6, 2
    q = np.full((heads, t, d), 40.0, dtype=np.float32)
    k = (0.01 * rng.standard_normal((t, d))).astype(np.float32)
    k[sink:t - w] += 10.0
    v = rng.standard_normal((t, dv)).astype(np.float32)
    o = NystromOracle(m=m, w=w, sink=sink, heads=heads)
    o.prefill(q, k, v)
    assert o.hs[0].m_max.max() > 700
    for n in range(3):
        out = o.step(np.full((1, d), 40.0),
                     0.01 * rng.standard_normal(d), rng.standard_normal(dv))
        dg = o.diags[-1][0]
        assert np.all(np.isfinite(out)), out
        assert dg.near_gap > 700          # the far maxima set the shift


def test_frozen_state_is_f32():
    """K~, Q~ and M are stored as f32 (nystrom.rs, prefill_shared and
    NystromHead::seal collect them `as f32`); the far field is fed by those
    stored values."""
    rng = np.random.default_rng(12)
    q, k, v = _rand_prompt(rng, 2, 64, 8, 8, kshift=0.5)
    o = NystromOracle(m=8, w=16, sink=4, heads=2)
    o.prefill(q, k, v)
    for arr in [o.k_tilde] + [h.q_tilde for h in o.hs] + [h.mu for h in o.hs]:
        np.testing.assert_array_equal(arr.astype(np.float32).astype(np.float64),
                                      arr)
    for h in o.hs:
        # M is the f32 rounding of the f64 solve, not a re-solve from the
        # rounded landmarks.
        assert np.abs(h.mu - h.ridge.m).max() <= 2 ** -23 * np.abs(h.ridge.m).max()
        assert not np.array_equal(h.mu, h.ridge.m)
