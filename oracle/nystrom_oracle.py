"""Plain fp64 CPU oracle for streaming Nystrom (landmark) attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
in ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import or run anything in this package.  The CUDA path never
calls it and it never calls the CUDA path: the two share no code, headers or
constants.  Inputs reach both sides from the seeded generators in
``streaming_nystr_landmark_gb300.workloads``, which hold none of the method's
arithmetic.

Source of truth: the docs.rs source view of ``cortiq_engine/src/nystrom.rs``
(cortiq-engine 0.5.71), cited below as "nystrom.rs, <item>", and the API page
"Struct NystromState" (cortiq-engine 0.5.21), cited as "NystromState docs,
<method>".  The functions restate the steps of those items in numpy, in the
order the page takes them, with these readings of what the page leaves open:

* Arithmetic is float64 throughout.  The page stores exactly three frozen
  quantities in f32 -- the key landmarks K~, the query landmarks Q~ and the
  mixing matrix M (nystrom.rs, ``prefill_shared`` and ``NystromHead::seal``) --
  and the oracle rounds exactly those three to f32 after computing them in
  f64, then uses the rounded values.  The score scale is the f32 value
  1/sqrt(d) computed in f32 (nystrom.rs, ``prefill_shared``), widened.
* The Au matrix is built from the f64 landmarks, before rounding (nystrom.rs,
  ``NystromHead::seal``).
* ``max`` in the ridge step follows f64::max: a NaN mean diagonal yields the
  other operand (np.fmax).

Every function here is pinned by the ``-m "not gpu"`` tests against closed
forms, brute force and independent library routines (see tests/test_oracle_*).
The approximation's fidelity to exact attention is PARITY UNPINNED: the pages'
only quality figures need a trained model and a text corpus.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
from scipy.linalg import solve_triangular

# nystrom.rs, const RIDGE_REL: lambda = RIDGE_REL * mean(diag(A^T A)).
RIDGE_REL = 1e-6
# nystrom.rs, const DEN_EPS: floor of the joint denominator.
DEN_EPS = 1e-30
# nystrom.rs, const EXACT_SLACK: prompts with t <= w + sink + EXACT_SLACK skip
# the skeleton.
EXACT_SLACK = 8
# nystrom.rs, ridge_pinv: the ridge grows tenfold on a failed Cholesky, at most
# twelve attempts in all.
RIDGE_TRIES = 12
# nystrom.rs, O1_DEFAULT_M / _W / _SINK.
DEFAULT_M, DEFAULT_W, DEFAULT_SINK = 32, 128, 4

# nystrom.rs, enum O1Rect.
AGGREGATE = 0
FM = 1


def score_scale(d: int) -> float:
    """1/sqrt(d) evaluated in f32 (nystrom.rs, ``prefill_shared``), widened."""
    return float(np.float32(1.0) / np.sqrt(np.float32(d)))


def f32_round(x: np.ndarray) -> np.ndarray:
    """Round to the nearest f32 and widen back: the page's f32 storage."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def effective_landmarks(t: int, m: int) -> int:
    """m_eff = clamp(t/8, 4, m) with integer division (nystrom.rs,
    ``prefill_shared``, the landmark clamp)."""
    return min(max(t // 8, 4), m)


def is_exact_only(t: int, w: int, sink: int) -> bool:
    """Short-prompt mode: t <= w + sink + EXACT_SLACK (nystrom.rs,
    ``prefill_shared``)."""
    return t <= w + sink + EXACT_SLACK


def seg_means(xs: np.ndarray, m: int) -> np.ndarray:
    """Contiguous segment means in f64 (nystrom.rs, ``seg_means``).

    Segment i covers rows [floor(i*t/m), floor((i+1)*t/m)); its mean is the
    f64 row sum times the reciprocal of the row count.
    """
    xs = np.asarray(xs, dtype=np.float64)
    t = xs.shape[0]
    out = np.zeros((m, xs.shape[1]), dtype=np.float64)
    for i in range(m):
        lo, hi = (i * t) // m, ((i + 1) * t) // m
        out[i] = xs[lo:hi].sum(axis=0) * (1.0 / (hi - lo))
    return out


def cholesky_lower(g: np.ndarray):
    """Lower Cholesky factor of a symmetric matrix, or None when a pivot is
    not strictly positive or not finite (nystrom.rs, ``cholesky``)."""
    n = g.shape[0]
    low = np.zeros_like(g, dtype=np.float64)
    for i in range(n):
        for j in range(i + 1):
            s = g[i, j] - float(np.dot(low[i, :j], low[j, :j]))
            if i == j:
                if not (s > 0.0) or not math.isfinite(s):
                    return None
                low[i, i] = math.sqrt(s)
            else:
                low[i, j] = s / low[j, j]
    return low


@dataclass
class RidgeResult:
    m: np.ndarray          # (A^T A + lambda I)^-1 A^T, f64
    lam: float             # the ridge that succeeded (or the last one tried)
    tries: int             # Cholesky attempts made (1..12), 13 = fallback used
    fallback: bool


def ridge_pinv(a: np.ndarray) -> RidgeResult:
    """Regularised pseudo-inverse of a square matrix (nystrom.rs,
    ``ridge_pinv``): M = (A^T A + lambda I)^-1 A^T with lambda =
    RIDGE_REL * max(mean diag(A^T A), f64 MIN_POSITIVE), solved through a
    Cholesky factor.  A failed factorisation multiplies lambda by ten, at most
    twelve attempts; after that M = I / max(mean diag, MIN_POSITIVE)."""
    a = np.asarray(a, dtype=np.float64)
    n = a.shape[0]
    with np.errstate(invalid="ignore", over="ignore"):
        ata = a.T @ a
        mean_diag = float(np.sum(np.diag(ata)) / n)
    tiny = float(np.finfo(np.float64).tiny)
    lam = RIDGE_REL * float(np.fmax(mean_diag, tiny))
    for attempt in range(1, RIDGE_TRIES + 1):
        with np.errstate(invalid="ignore", over="ignore"):
            g = ata + lam * np.eye(n)
        low = cholesky_lower(g)
        if low is not None:
            # G M = A^T, one right-hand side per column of A^T (= row of A).
            y = solve_triangular(low, a.T, lower=True)
            mm = solve_triangular(low.T, y, lower=False)
            return RidgeResult(mm, lam, attempt, False)
        lam *= 10.0
    fb = np.eye(n) / float(np.fmax(mean_diag, tiny))
    return RidgeResult(fb, lam, RIDGE_TRIES + 1, True)


@dataclass
class HeadState:
    """Private per-Q-head part (nystrom.rs, ``NystromHead``)."""
    q_tilde: np.ndarray = None   # [m_eff][d]   f32-rounded
    mu: np.ndarray = None        # [m_eff][m_eff] f32-rounded, rows = key landmark
    t_hat: np.ndarray = None     # [m_eff][dv]  at scale e^{-m_max}
    z_hat: np.ndarray = None     # [m_eff]
    m_max: np.ndarray = None     # [m_eff]
    far_len: int = 0
    ridge: RidgeResult = None


@dataclass
class StepDiag:
    """Per head and decode step: numbers the parity tests use to decide
    whether a row sits on a discontinuity of the method."""
    have_far: bool
    margin: float        # far_den / den: distance of the Aggregate guard
    near_gap: float      # c_all - c: near weights are exp(sigma - c_all)
    den: float           # final joint denominator (shifted frame)
    kappa: float         # cancellation factor of u = F^ M (max over b)


@dataclass
class NystromOracle:
    """One GQA group's state (nystrom.rs, ``NystromState`` = ``NystromGroup``
    shared by the group + one ``NystromHead`` per Q head).

    Lifecycle as on the NystromState docs: construct, ``prefill`` once, then
    ``step`` once per decode token.
    """
    m: int
    w: int
    sink: int
    heads: int = 1
    rect: int = AGGREGATE
    # shared part (nystrom.rs, NystromGroup)
    d: int = 0
    dv: int = 0
    m_eff: int = 0
    exact_only: bool = True
    scale: float = 0.0
    win_k: np.ndarray = None
    win_v: np.ndarray = None
    win_len: int = 0
    win_head: int = 0
    sink_k: np.ndarray = None
    sink_v: np.ndarray = None
    sink_len: int = 0
    k_tilde: np.ndarray = None
    hs: list = field(default_factory=list)
    diags: list = field(default_factory=list)

    def __post_init__(self):
        # nystrom.rs, new_group: the three constructor preconditions.
        if self.m < 4 or self.w < 1 or self.heads < 1:
            raise ValueError("need m >= 4, w >= 1, heads >= 1")
        if self.rect not in (AGGREGATE, FM):
            raise ValueError("rect must be AGGREGATE or FM")
        self.hs = [HeadState() for _ in range(self.heads)]

    # ------------------------------------------------------------ seal
    def prefill(self, qs, ks, vs):
        """Seal the prompt (nystrom.rs, ``prefill_group``).

        qs: [heads][t][d], ks: [t][d], vs: [t][dv].  Shared part first, then
        each head's landmarks and M, then a replay of positions sink..t-1
        through the window (delayed far insertion)."""
        qs = np.asarray(qs, dtype=np.float64)
        ks = np.asarray(ks, dtype=np.float64)
        vs = np.asarray(vs, dtype=np.float64)
        if qs.ndim == 2:
            qs = qs[None]
        if qs.shape[0] != self.heads:
            raise ValueError("one query block per head")
        t, d = ks.shape
        dv = vs.shape[1]
        if qs.shape[1:] != (t, d) or vs.shape[0] != t:
            raise ValueError("prompt shapes disagree")
        self.diags = []
        k_tilde64 = self._prefill_shared(ks, vs, t, d, dv)
        if k_tilde64 is None:
            for h in self.hs:          # nystrom.rs, seal_exact
                h.far_len = 0
            return
        for h, q in zip(self.hs, qs):
            self._seal_head(h, q, k_tilde64)
        for j in range(self.sink, t):
            self._advance(ks[j], vs[j])

    def _prefill_shared(self, ks, vs, t, d, dv):
        """nystrom.rs, ``NystromGroup::prefill_shared``."""
        self.d, self.dv = d, dv
        self.scale = score_scale(d)
        self.win_len = 0
        self.win_head = 0
        self.sink_len = 0
        self.exact_only = is_exact_only(t, self.w, self.sink)
        if self.exact_only:
            # Every prompt key stays an exact key; no sinks, no skeleton.
            self.win_k = ks.copy()
            self.win_v = vs.copy()
            self.win_len = t
            self.m_eff = 0
            return None
        self.sink_len = self.sink
        self.sink_k = ks[: self.sink].copy()
        self.sink_v = vs[: self.sink].copy()
        self.m_eff = effective_landmarks(t, self.m)
        k_tilde64 = seg_means(ks, self.m_eff)
        self.k_tilde = f32_round(k_tilde64)
        self.win_k = np.zeros((self.w, d))
        self.win_v = np.zeros((self.w, dv))
        return k_tilde64

    def _seal_head(self, h: HeadState, q, k_tilde64):
        """nystrom.rs, ``NystromHead::seal``: Q~ from this head's queries,
        Au = exp(Q~64 K~64^T * scale) in f64, M = ridge_pinv(Au) stored f32,
        empty far field with running max -inf."""
        q_tilde64 = seg_means(q, self.m_eff)
        h.q_tilde = f32_round(q_tilde64)
        with np.errstate(over="ignore"):
            au = np.exp((q_tilde64 @ k_tilde64.T) * self.scale)
        h.ridge = ridge_pinv(au)
        h.mu = f32_round(h.ridge.m)
        h.t_hat = np.zeros((self.m_eff, self.dv))
        h.z_hat = np.zeros(self.m_eff)
        h.m_max = np.full(self.m_eff, -np.inf)
        h.far_len = 0

    # ------------------------------------------------------------ decode
    def step(self, q_all, k, v):
        """One decode token for the whole group (nystrom.rs, ``step_group``):
        insert (k, v) once -- evicting into every head's far field -- and then
        compute every head's output.  q_all: [heads][d]; returns [heads][dv]."""
        if self.d == 0:
            raise RuntimeError("prefill must run before step")
        q_all = np.asarray(q_all, dtype=np.float64).reshape(self.heads, self.d)
        k = np.asarray(k, dtype=np.float64).reshape(self.d)
        v = np.asarray(v, dtype=np.float64).reshape(self.dv)
        self._advance(k, v)
        outs, diags = [], []
        for h, q in zip(self.hs, q_all):
            o, dg = self._head_output(h, q)
            outs.append(o)
            diags.append(dg)
        self.diags.append(diags)
        return np.stack(outs)

    def _advance(self, k, v):
        """nystrom.rs, ``NystromState::advance``.  A full ring is a GROUP
        eviction: every head absorbs the oldest slot once, then the slot is
        overwritten and the ring head moves on."""
        if self.exact_only:
            self.win_k = np.vstack([self.win_k, k[None]])
            self.win_v = np.vstack([self.win_v, v[None]])
            self.win_len += 1
        elif self.win_len == self.w:
            slot = self.win_head
            for h in self.hs:
                self._far_insert(h, slot)
            self.win_k[slot] = k
            self.win_v[slot] = v
            self.win_head = (self.win_head + 1) % self.w
        else:
            self.win_k[self.win_len] = k
            self.win_v[self.win_len] = v
            self.win_len += 1

    def _far_insert(self, h: HeadState, slot: int):
        """nystrom.rs, ``NystromHead::far_insert``: logits of the outgoing key
        against this head's query landmarks; where a logit beats the running
        max (strictly), the stored mass is rescaled by exp(old - new) (which is
        0 on the first insertion, old = -inf); then the key is added at weight
        exp(l - m_max)."""
        k_ev, v_ev = self.win_k[slot], self.win_v[slot]
        logit = (h.q_tilde @ k_ev) * self.scale
        grow = logit > h.m_max
        r = np.where(grow, np.exp(np.where(grow, h.m_max - logit, 0.0)), 1.0)
        h.z_hat *= r
        h.t_hat *= r[:, None]
        h.m_max = np.where(grow, logit, h.m_max)
        e = np.exp(logit - h.m_max)
        h.z_hat += e
        h.t_hat += e[:, None] * v_ev[None, :]
        h.far_len += 1

    def _head_output(self, h: HeadState, q):
        """nystrom.rs, ``NystromHead::step``: exact near logits over sinks and
        window, landmark row with its own shift f, mixing row u = F^ M (Fm
        clamps it at 0), one joint shift c_all, Aggregate guard on the far
        denominator, then a single division floored at DEN_EPS."""
        ns = self.sink_len
        rows_k = self.win_k[: self.win_len]
        rows_v = self.win_v[: self.win_len]
        if ns:
            rows_k = np.vstack([self.sink_k, rows_k])
            rows_v = np.vstack([self.sink_v, rows_v])
        sigma = (rows_k @ q) * self.scale
        c = float(np.max(sigma)) if sigma.size else -np.inf

        far_den, c_all, have_far, gains, kappa = 0.0, c, False, None, 0.0
        if h.far_len > 0:
            s = (self.k_tilde @ q) * self.scale
            f = float(np.max(s))
            fh = np.exp(s - f)
            terms = fh[:, None] * h.mu           # [a][b] = F^_a M[a][b]
            u = terms.sum(axis=0)
            with np.errstate(divide="ignore", invalid="ignore"):
                kap = np.abs(terms).sum(axis=0) / np.abs(u)
            kappa = float(np.nanmax(kap)) if kap.size else 0.0
            if self.rect == FM:
                u = np.maximum(u, 0.0)
            c_all = max(c, float(np.max(f + h.m_max)))
            gains = u * np.exp(f + h.m_max - c_all)
            far_den = float(gains @ h.z_hat)
            if far_den >= 0.0:
                have_far = True
            else:
                far_den = 0.0

        out = np.zeros(self.dv)
        if have_far:
            out += gains @ h.t_hat
        p = np.exp(sigma - c_all)
        out += p @ rows_v
        den = far_den + float(p.sum())
        total = max(den, DEN_EPS)
        margin = (far_den / total) if have_far else (
            -1.0 if h.far_len > 0 else 0.0)
        if h.far_len > 0 and not have_far:
            # Report how far below zero the dropped far denominator was,
            # relative to the near mass it was compared with.
            raw = float(gains @ h.z_hat)
            margin = raw / max(float(p.sum()), DEN_EPS)
        return out / total, StepDiag(have_far, margin, c_all - c, den, kappa)

    # ------------------------------------------------------------ queries
    def far_len(self, head: int) -> int:
        """Keys absorbed into one head's far field (NystromState docs,
        ``far_len``)."""
        return self.hs[head].far_len


# ---------------------------------------------------------------- O-B
def direct_output(q, k_hist, v_hist, sink, w, k_tilde, q_tilde, mu, scale,
                  rect=AGGREGATE):
    """Materialised-weights formulation of one head's output at the newest
    position p = len(k_hist) - 1 (nystrom.rs module doc: the operator formula,
    with the sink rule of the same doc and the rectifiers of ``O1Rect``).

    Near set N = {j < sink} U {p - w < j <= p}; far set Phi = {sink <= j <=
    p - w}.  Weights are built unshifted:
        e_j      = exp(q . k_j * scale)                   (j in N)
        F_a      = exp(q . k~_a * scale)
        u        = F M                 (Fm: clamped at 0 elementwise)
        E[b][j]  = exp(q~_b . k_j * scale)                (j in Phi)
        w^_j     = sum_b u_b E[b][j]
    The far field is kept iff sum_Phi w^_j >= 0, and
        out = (sum_N e_j v_j + keep sum_Phi w^_j v_j)
              / (sum_N e_j + keep sum_Phi w^_j).
    Returns (out, far_weights, keep)."""
    q = np.asarray(q, dtype=np.float64)
    k_hist = np.asarray(k_hist, dtype=np.float64)
    v_hist = np.asarray(v_hist, dtype=np.float64)
    p = k_hist.shape[0] - 1
    idx = np.arange(p + 1)
    near = (idx < sink) | (idx > p - w)
    far = ~near
    e = np.exp((k_hist[near] @ q) * scale)
    num = e @ v_hist[near]
    den = float(e.sum())
    far_w = np.zeros(0)
    keep = False
    if far.any():
        fvec = np.exp((k_tilde @ q) * scale)
        u = fvec @ mu
        if rect == FM:
            u = np.maximum(u, 0.0)
        big_e = np.exp((q_tilde @ k_hist[far].T) * scale)
        far_w = u @ big_e
        keep = float(far_w.sum()) >= 0.0
        if keep:
            num = num + far_w @ v_hist[far]
            den = den + float(far_w.sum())
    return num / den, far_w, keep
