"""Row-error tail of a full-size decode against the fp64 oracle (not a test).

    python tests/parity_tail.py WORKLOAD GROUPS [STEPS] [OUT.json]

Runs the whole launch of WORKLOAD on cuda:0, with GROUPS of its groups
(evenly spaced) fed from the seeded host streams and checked against one
oracle each (stepped in worker processes, tests/oracle_pool.py), and reports
the distribution of every checked row's error (max |o - o_ref| / max |o_ref|)
without asserting anything: quantiles, counts above 5e-5 and 1e-4, and the
worst rows with their mixing cancellation, guard margin and near gap.  Rows
on a discontinuity of the method (guard band, near-weight underflow) are
left out, as in the parity tests.
"""
import json
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import numpy as np  # noqa: E402

import parity_util as pu  # noqa: E402
from streaming_nystr_landmark_gb300.workloads import WORKLOADS, host_token_batch  # noqa: E402


def main():
    import torch
    wl = WORKLOADS[sys.argv[1]]
    ngr = int(sys.argv[2])
    steps = int(sys.argv[3]) if len(sys.argv) > 3 else wl.steps
    out_path = sys.argv[4] if len(sys.argv) > 4 else None
    n = wl.n_groups
    sample = sorted(set(int(g) for g in np.linspace(0, n - 1, ngr)))
    dev = torch.device("cuda:0")
    run = pu.ParityRun(wl, sample, dev, workers=pu.oracle_workers())
    rows = []  # (error, group, token, head, kappa, margin, near_gap)
    t0 = time.time()
    try:
        run.seal()
        idx = torch.tensor(run.sample, device=dev)
        for step in range(steps):
            qh, kh, vh = host_token_batch(run.gens, step)
            q = torch.empty((1, run.G, wl.heads_per_kv, wl.d), device=dev)
            k = torch.empty((1, run.G, wl.d), device=dev)
            v = torch.empty((1, run.G, wl.dv), device=dev)
            run.fill.tokens_into(q, k, v)
            q, k, v = q[0], k[0], v[0]
            q[idx] = torch.from_numpy(qh).to(dev)
            k[idx] = torch.from_numpy(kh).to(dev)
            v[idx] = torch.from_numpy(vh).to(dev)
            run.pool.start_step(step)
            out = torch.empty((run.G, wl.heads_per_kv, wl.dv), device=dev)
            run.st.step(q, k, v, out)
            got = out[idx].cpu().numpy().astype(np.float64)
            refs, flags, diag = run.pool.finish_step()
            for i in range(len(sample)):
                for h in range(wl.heads_per_kv):
                    if not flags[i, h]:
                        rows.append((pu.row_err(got[i, h], refs[i, h]), sample[i], step, h,
                                     *map(float, diag[i, h])))
    finally:
        run.close()
    rows.sort(reverse=True)
    e = np.array([r[0] for r in rows])
    res = {"workload": wl.name, "rows": len(rows), "groups": len(sample), "steps": steps,
           "seconds": round(time.time() - t0, 1),
           "quantiles": {str(p): float(np.quantile(e, p)) for p in (0.5, 0.9, 0.99, 0.999, 0.9999)},
           "over_5e-5": int((e > 5e-5).sum()), "over_1e-4": int((e > 1e-4).sum()),
           "worst": [{"error": r[0], "group": r[1], "token": r[2], "head": r[3],
                      "mixing_cancellation": r[4], "guard_margin": r[5], "near_gap": r[6]}
                     for r in rows[:10]]}
    if out_path:
        with open(out_path, "w") as f:
            json.dump(res, f, indent=1)
    print(json.dumps(res, indent=1))


if __name__ == "__main__":
    main()
