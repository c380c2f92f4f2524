"""fp64 oracles in worker processes, stepped in parallel (test infrastructure).

A full-size parity run compares sampled groups of a launch with one oracle
each; the oracle is plain numpy, about 4 K group-steps per second on one
core, and a 32K-token prompt takes seconds just to draw.  To compare many
groups at full size, the oracles live in spawned worker processes, each
owning a slice of the sample.  A worker draws its groups' inputs from the
same seeded per-group streams the test uses, optionally hands the prompts
(and the token streams, positioned after them) to the parent for the GPU,
seals its oracles, and then, per decode token, steps them and returns their
outputs and the rows that sit on a discontinuity of the method (checked
finite only).
State comparisons run in the worker too, on the device regions the test
sends it.  Workers are started with the spawn method (a forked child of a
process that has initialised CUDA can hang); every wait on a worker is
bounded.
"""
import os

for _var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, "1")

import multiprocessing as mp  # noqa: E402
import traceback  # noqa: E402

import numpy as np  # noqa: E402

REPLY_TIMEOUT_S = 900.0


def _worker(conn, wl, groups, guard_band, underflow_gap, send_prompts):
    try:
        from oracle import NystromOracle
        from parity_util import compare_group_state
        from streaming_nystr_landmark_gb300.workloads import (host_prompt_batch,
                                                              host_token_batch)
        prompts = [host_prompt_batch(wl, [g]) for g in groups]
        if send_prompts:  # all of them first: the parent waits on them
            for g, (qh, kh, vh, gi) in zip(groups, prompts):
                conn.send(("prompt", (g, qh[0], kh[0], vh[0], gi[0])))
        oracles, gens = [], []
        for i in range(len(groups)):
            qh, kh, vh, gi = prompts[i]
            o = NystromOracle(wl.m, wl.w, wl.sink, wl.heads_per_kv, wl.rect)
            o.prefill(qh[0], kh[0], vh[0])
            oracles.append(o)
            gens += gi
            prompts[i] = None
        conn.send(("ok", None))
        while True:
            cmd, arg = conn.recv()
            if cmd == "close":
                return
            if cmd == "step":
                tq, tk, tv = host_token_batch(gens, arg)
                outs = np.stack([o.step(tq[i], tk[i], tv[i]) for i, o in enumerate(oracles)])
                flags = np.array([[abs(dg.margin) < guard_band or dg.near_gap > underflow_gap
                                   for dg in o.diags[-1]] for o in oracles])
                diag = np.array([[(dg.kappa, dg.margin, dg.near_gap) for dg in o.diags[-1]]
                                 for o in oracles])
                conn.send(("ok", (outs, flags, diag)))
            elif cmd == "state":
                regs, far_tol = arg
                for i, o in enumerate(oracles):
                    compare_group_state(regs, i, o, far_tol)
                conn.send(("ok", None))
    except Exception:  # report, never leave the parent waiting
        try:
            conn.send(("error", traceback.format_exc()))
        except Exception:
            pass


class OraclePool:
    """Oracles for `groups` (global group indices) split over `workers`
    spawned processes, in the order given."""

    def __init__(self, wl, groups, workers, guard_band, underflow_gap, send_prompts=False):
        ctx = mp.get_context("spawn")
        groups = list(groups)
        workers = max(1, min(workers, len(groups)))
        self.parts = [list(p) for p in np.array_split(np.array(groups), workers)]
        self.conns, self.procs = [], []
        for part in self.parts:
            a, b = ctx.Pipe()
            p = ctx.Process(target=_worker, args=(b, wl, [int(g) for g in part], guard_band,
                                                  underflow_gap, send_prompts), daemon=True)
            p.start()
            b.close()
            self.conns.append(a)
            self.procs.append(p)

    def prompts(self):
        """With send_prompts: (group, q, k, v, token stream) of every group,
        in the order the groups were given."""
        for c, part in zip(self.conns, self.parts):
            for _ in part:
                if not c.poll(REPLY_TIMEOUT_S):
                    raise TimeoutError("an oracle worker did not answer")
                status, val = c.recv()
                if status != "prompt":
                    raise AssertionError(val)
                yield val

    def ready(self):
        """Wait (bounded) until every worker has sealed its oracles."""
        for c in self.conns:
            self._reply(c)

    def _reply(self, conn):
        if not conn.poll(REPLY_TIMEOUT_S):
            raise TimeoutError("an oracle worker did not answer")
        status, val = conn.recv()
        if status != "ok":
            raise AssertionError(val)
        return val

    def start_step(self, n):
        """Every worker steps its oracles to decode token n (asynchronously)."""
        for c in self.conns:
            c.send(("step", n))

    def finish_step(self):
        """(outputs [n][H][dv], discontinuity flags [n][H], the rows'
        (kappa, margin, near_gap) [n][H][3]) in group order."""
        res = [self._reply(c) for c in self.conns]
        return tuple(np.concatenate([r[i] for r in res]) for i in range(3))

    def compare_state(self, regs, far_tol):
        """Each worker compares its groups' rows of `regs` (read_state of the
        whole launch) with its oracles."""
        for c, part in zip(self.conns, self.parts):
            idx = np.array(part)
            c.send(("state", ({name: arr[idx] for name, arr in regs.items()}, far_tol)))
        for c in self.conns:
            self._reply(c)

    def close(self):
        for c in self.conns:
            try:
                c.send(("close", None))
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
