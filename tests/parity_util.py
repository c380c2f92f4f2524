"""Drive the CUDA path and the fp64 oracle side by side on the same inputs.

The library runs every group of a workload in one launch per token.  Groups
listed in ``sample`` receive host-drawn inputs from the seeded per-group
streams, which the oracle also consumes; any other group receives
device-drawn filler of the same distribution, so full-size launches stay full
size while the oracle only runs the sampled groups.

Tolerances (an fp32 evaluation of the step, measured against the oracle
before any kernel existed, gives ~1.4e-5 per step on the m = 32 workloads;
the bounds leave room for that plus the state's accumulated rounding):
  outputs         row-normwise  max|o - o_ref| / max|o_ref| <= 1e-4, except
                  rows where the Aggregate guard sits within 1e-5 of its
                  threshold (either branch is then correct) or where the far
                  maxima sit > 80 above the near maximum (fp32 near weights
                  underflow by design of the joint shift);
  K~, Q~          <= 1e-6 relative to the row's max magnitude;
  M               <= 1e-5 normwise relative;
  T^, Z^, m_max   <= 1e-5, compared at a common scale (T^ and Z^ are the
                  device's hi + lo pairs);
  window, sinks   bit-exact (copies of the inputs);
  counters        bit-exact (far_len per head, win_head, win_len, m_eff, t).
"""
from __future__ import annotations

import numpy as np

from oracle import NystromOracle
from streaming_nystr_landmark_gb300.workloads import (DeviceFill, GroupInputs,
                                                      host_prompt_batch,
                                                      host_token_batch)

OUT_TOL = 1e-4
LANDMARK_TOL = 1e-6
MU_TOL = 1e-5
FAR_TOL = 1e-5
GUARD_BAND = 1e-5
UNDERFLOW_GAP = 80.0


def oracle_workers():
    """Oracle worker processes for a full-size run: the host's cores but two."""
    import os
    return max(1, min(16, (os.cpu_count() or 2) - 2))


def row_err(got, ref):
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


class ParityRun:
    """workers > 0: the sampled groups' oracles run in that many spawned
    processes (oracle_pool.OraclePool), stepped while the GPU steps."""

    def __init__(self, wl, sample, device, n_groups=None, host_all=None, workers=0):
        import torch
        from streaming_nystr_landmark_gb300.nys import NystromStates
        self.torch = torch
        self.wl = wl
        self.dev = device
        self.G = wl.n_groups if n_groups is None else n_groups
        self.sample = list(sample)
        self.host_all = (self.G <= 64) if host_all is None else host_all
        if self.host_all:
            self.sample = list(range(self.G))
        self.st = NystromStates(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.d,
                                wl.dv, self.G, wl.rect, device)
        self.flagged = 0
        self.checked = 0
        self.worst = 0.0
        self.worst_at = None  # (group, token, head, kappa, margin, near_gap)
        self.workers = workers
        self.pool = None
        self.oracles = []
        self.fill = None if self.host_all else DeviceFill(
            wl.with_(seqs=1, layers=1, kv_groups=self.G), device)

    # ------------------------------------------------------------ seal
    def seal(self):
        torch, wl, G = self.torch, self.wl, self.G
        if self.workers:
            from oracle_pool import OraclePool
            # The workers draw the sampled prompts, hand them over, and seal
            # their oracles while this process seals the GPU.
            self.pool = OraclePool(wl, self.sample, self.workers, GUARD_BAND, UNDERFLOW_GAP,
                                   send_prompts=not self.host_all)
        if self.host_all:
            qh, kh, vh, self.gens = host_prompt_batch(wl, self.sample)
            q = torch.from_numpy(qh).to(self.dev)
            k = torch.from_numpy(kh).to(self.dev)
            v = torch.from_numpy(vh).to(self.dev)
        else:
            q = torch.empty((G, wl.heads_per_kv, wl.t, wl.d), device=self.dev)
            k = torch.empty((G, wl.t, wl.d), device=self.dev)
            v = torch.empty((G, wl.t, wl.dv), device=self.dev)
            self.fill.prompt_into(q, k, v)
            # Host prompts of the sampled groups, a few at a time (a long
            # prompt is ~0.2 GB); the oracles below, if local, get theirs
            # regenerated from the same streams.
            if self.pool is not None:
                self.gens = []
                for g, qh, kh, vh, gi in self.pool.prompts():
                    q[g] = torch.from_numpy(qh).to(self.dev)
                    k[g] = torch.from_numpy(kh).to(self.dev)
                    v[g] = torch.from_numpy(vh).to(self.dev)
                    self.gens.append(gi)
            else:
                self.gens = []
                for c0 in range(0, len(self.sample), 4):
                    part = self.sample[c0:c0 + 4]
                    qh, kh, vh, gens = host_prompt_batch(wl, part)
                    idx = torch.tensor(part, device=self.dev)
                    q[idx] = torch.from_numpy(qh).to(self.dev)
                    k[idx] = torch.from_numpy(kh).to(self.dev)
                    v[idx] = torch.from_numpy(vh).to(self.dev)
                    self.gens += gens
        self.st.seal(q, k, v)
        torch.cuda.synchronize(self.dev)
        del q, k, v
        if self.pool is not None:
            self.pool.ready()
        else:
            self.oracles = []
            for g in self.sample:
                qh, kh, vh, _ = host_prompt_batch(wl, [g])
                o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.rect)
                o.prefill(qh[0], kh[0], vh[0])
                self.oracles.append(o)
        self.n_steps = 0

    # ------------------------------------------------------------ state
    def check_state(self, far_tol=FAR_TOL):
        """Compare every sampled group's device state with its oracle."""
        regs = read_state(self.st)
        if self.pool is not None:
            self.pool.compare_state(regs, far_tol)
            return
        for o, g in zip(self.oracles, self.sample):
            compare_group_state(regs, g, o, far_tol)

    # ------------------------------------------------------------ decode
    def step(self):
        torch, wl, G = self.torch, self.wl, self.G
        n = self.n_steps
        qh, kh, vh = host_token_batch(self.gens, n)
        if self.host_all:
            q = torch.from_numpy(qh).to(self.dev)
            k = torch.from_numpy(kh).to(self.dev)
            v = torch.from_numpy(vh).to(self.dev)
        else:
            q = torch.empty((1, G, wl.heads_per_kv, wl.d), device=self.dev)
            k = torch.empty((1, G, wl.d), device=self.dev)
            v = torch.empty((1, G, wl.dv), device=self.dev)
            self.fill.tokens_into(q, k, v)
            q, k, v = q[0], k[0], v[0]
            idx = torch.tensor(self.sample, device=self.dev)
            q[idx] = torch.from_numpy(qh).to(self.dev)
            k[idx] = torch.from_numpy(kh).to(self.dev)
            v[idx] = torch.from_numpy(vh).to(self.dev)
        if self.pool is not None:
            self.pool.start_step(n)  # the oracles step while the GPU does
        out = torch.empty((G, wl.heads_per_kv, wl.dv), device=self.dev)
        self.st.step(q, k, v, out)
        got = out[torch.tensor(self.sample, device=self.dev)].cpu().numpy()
        self.n_steps += 1
        if self.pool is not None:
            refs, flags, diag = self.pool.finish_step()
            for i in range(len(self.sample)):
                for h in range(wl.heads_per_kv):
                    self.checked += 1
                    if flags[i, h]:
                        self.flagged += 1
                        assert np.all(np.isfinite(got[i, h]))
                        continue
                    err = row_err(got[i, h].astype(np.float64), refs[i, h])
                    if err > self.worst:
                        self.worst = err
                        self.worst_at = (self.sample[i], n, h, *diag[i, h])
                    assert err <= OUT_TOL, (self.sample[i], h, n, err, tuple(diag[i, h]))
            return out
        for i, o in enumerate(self.oracles):
            ref = o.step(qh[i], kh[i], vh[i])
            for h in range(wl.heads_per_kv):
                dg = o.diags[-1][h]
                err = row_err(got[i, h].astype(np.float64), ref[h])
                self.checked += 1
                if abs(dg.margin) < GUARD_BAND or dg.near_gap > UNDERFLOW_GAP:
                    self.flagged += 1
                    assert np.all(np.isfinite(got[i, h]))
                    continue
                if err > self.worst:
                    self.worst = err
                    self.worst_at = (self.sample[i], n, h, dg.kappa, dg.margin, dg.near_gap)
                assert err <= OUT_TOL, (self.sample[i], h, n, err)
        return out

    def check_counters_all(self):
        """Properties that hold for every group at any size: counters follow
        the eviction count exactly."""
        wl = self.wl
        far = self.st.region("far_len").cpu().numpy()
        ints = self.st.region("ints").cpu().numpy()
        ev = wl.t - wl.sink - wl.w + self.n_steps
        assert np.all(far == ev), (far.min(), far.max(), ev)
        assert np.all(ints[:, 0] == (wl.t - wl.sink + self.n_steps) % wl.w)
        assert np.all(ints[:, 1] == wl.w)
        assert np.all(ints[:, 5] == 0), "a decode kernel reported a timed-out wait"

    def close(self):
        if self.pool is not None:
            self.pool.close()
            self.pool = None
        self.st.close()


def step_oracles_and_compare(oracles, tq, tk, tv, outs):
    """Step each group's oracle once (host token inputs tq [G][H][d],
    tk [G][d], tv [G][dv], group g feeding oracles[g]) and compare every
    array in `outs` ([G][H][dv] device results copied to the host) with the
    oracle's outputs row by row at OUT_TOL.  Rows on a discontinuity of the
    method (guard band, near-weight underflow) are only checked finite.
    Returns the worst row error."""
    worst = 0.0
    for g, o in enumerate(oracles):
        ref = o.step(tq[g], tk[g], tv[g])
        for h in range(ref.shape[0]):
            dg = o.diags[-1][h]
            flagged = abs(dg.margin) < GUARD_BAND or dg.near_gap > UNDERFLOW_GAP
            for got in outs:
                row = np.asarray(got[g][h], dtype=np.float64)
                if flagged:
                    assert np.all(np.isfinite(row)), (g, h)
                    continue
                err = row_err(row, ref[h])
                assert err <= OUT_TOL, (g, h, err)
                worst = max(worst, err)
    return worst


def read_state(st):
    """Host copies of every state region (T^ and Z^ as hi + lo)."""
    reg = {name: st.region(name).cpu().numpy() for name in (
        "win_k", "win_v", "sink_k", "sink_v", "k_tilde", "q_tilde", "mu",
        "m_max", "far_len", "ints")}
    reg["t_hat"] = st.far_numerator()
    reg["z_hat"] = st.far_denominator()
    return reg


def compare_group_state(reg, g, o, far_tol=FAR_TOL):
    """Device state of group g (from read_state) against oracle o."""
    me = o.m_eff
    ints = reg["ints"][g]
    assert ints[0] == o.win_head and ints[1] == o.win_len, (g, ints)
    assert ints[2] == me and ints[4] == 1, (g, ints)
    np.testing.assert_array_equal(reg["win_k"][g], o.win_k.astype(np.float32))
    np.testing.assert_array_equal(reg["win_v"][g], o.win_v.astype(np.float32))
    if o.sink_len:
        np.testing.assert_array_equal(reg["sink_k"][g], o.sink_k.astype(np.float32))
        np.testing.assert_array_equal(reg["sink_v"][g], o.sink_v.astype(np.float32))
    _close_rows(reg["k_tilde"][g][:me].astype(np.float64), o.k_tilde, LANDMARK_TOL,
                "k_tilde", g)
    for h, hs in enumerate(o.hs):
        assert reg["far_len"][g][h] == hs.far_len, (g, h)
        _close_rows(reg["q_tilde"][g][h][:me].astype(np.float64), hs.q_tilde,
                    LANDMARK_TOL, "q_tilde", g)
        mu = reg["mu"][g][h][:me, :me].astype(np.float64)
        rel = np.linalg.norm(mu - hs.mu) / np.linalg.norm(hs.mu)
        assert rel <= MU_TOL, ("mu", g, h, rel)
        mm = reg["m_max"][g][h][:me].astype(np.float64)
        assert np.all(np.abs(mm - hs.m_max) <= far_tol * np.maximum(1.0, np.abs(hs.m_max))), \
            ("m_max", g, h, np.abs(mm - hs.m_max).max())
        # Bring the device accumulators to the oracle's scale.
        rescale = np.exp(mm - hs.m_max)
        z = reg["z_hat"][g][h][:me].astype(np.float64) * rescale
        np.testing.assert_allclose(z, hs.z_hat, rtol=far_tol, atol=0)
        t = reg["t_hat"][g][h][:me].astype(np.float64) * rescale[:, None]
        for b in range(me):
            e = row_err(t[b], hs.t_hat[b])
            assert e <= far_tol, ("t_hat", g, h, b, e)


def _close_rows(got, ref, tol, what, g):
    scale = np.maximum(np.abs(ref).max(axis=1, keepdims=True), 1e-30)
    err = float((np.abs(got - ref) / scale).max())
    assert err <= tol, (what, g, err)
