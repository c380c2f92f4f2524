"""Named decode workloads and their seeded synthetic inputs.

This module holds no arithmetic of the attention method: only geometry and
random numbers.  It is the one piece of Python that both the CUDA path's
tests/benchmark and the CPU oracle receive inputs from.

Workloads (all fp32; shapes follow a Qwen3-0.6B attention layer: 16 query
heads over 8 KV heads, head dim 128, and the page's validated operator setting
m=32, W=128, sink=4 from nystrom.rs, ``O1_DEFAULT_*``):

=========  ===========================================================  =====
name       geometry                                                     k mean
=========  ===========================================================  =====
single     1 group, H=1, d=dv=64, m=8, w=16, s=4, t=64, 64 steps       2*u
layer      8 groups (one layer), H=2, d=128, m=32, w=128, s=4, t=256,  3*u_g
           256 steps
batch64    64 seq x 28 layers x 8 groups = 14336 groups, H=2, d=128,   2*u_g
           m=32, w=128, s=4, t=256, 1024 steps (one launch per token)
sweep      256 seq x 8 groups = 2048 groups, H=2, d=128, w=128, s=4,   2*u_g
           t=512, 512 steps, m in {8,16,32,64} x {aggregate, fm}
long       128 seq x 4 groups = 512 groups, H=8, d=128, m=64, w=128,   walk
           s=4, t=32768, 2048 steps
=========  ===========================================================  =====

Draw recipe.  q, k and v entries are i.i.d. N(0, 1) float32.  k then gets a
per-group mean: ``2*u`` / ``3*u`` with u a random unit vector of that group,
or ``walk``: a mean that starts at 0 and moves by 0.01 * xi/|xi| (xi ~ N(0, I))
at every position, prompt and decode alike.

Keying.  Every (workload seed, sequence, layer, KV group) owns independent
numpy ``Philox`` streams derived through ``SeedSequence`` from that tuple plus
a tensor tag and, for decode tokens, the step index.  Any group's inputs can
therefore be drawn on its own, which is how the full-size parity tests feed
the oracle a sample of groups while the device holds all of them.  The device
fill (``fill_device_*``) draws the same distributions with torch on the GPU
for groups no oracle looks at, and for the benchmark.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

AGGREGATE, FM = 0, 1

_TAG_Q, _TAG_K, _TAG_V, _TAG_DIR, _TAG_WALK = 1, 2, 3, 4, 5
_PROMPT = 0xFFFFFFFF  # step index used for prompt streams


@dataclass(frozen=True)
class Workload:
    name: str
    heads_per_kv: int
    d: int
    dv: int
    m: int
    w: int
    sink: int
    rect: int
    t: int            # prompt length sealed into every group
    steps: int        # decode tokens after the seal
    seqs: int
    layers: int
    kv_groups: int
    k_mean: str       # "unit2" | "unit3" | "walk"
    seed: int = 0

    @property
    def n_groups(self) -> int:
        return self.seqs * self.layers * self.kv_groups

    def group_coords(self, g: int):
        """(sequence, layer, kv group) of flat group index g; groups are
        ordered sequence-major, then layer, then KV group."""
        kvg = g % self.kv_groups
        rest = g // self.kv_groups
        return rest // self.layers, rest % self.layers, kvg

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "single": Workload("single", 1, 64, 64, 8, 16, 4, AGGREGATE, 64, 64,
                       1, 1, 1, "unit2", seed=0),
    "layer": Workload("layer", 2, 128, 128, 32, 128, 4, AGGREGATE, 256, 256,
                      1, 1, 8, "unit3", seed=1),
    "batch64": Workload("batch64", 2, 128, 128, 32, 128, 4, AGGREGATE, 256,
                        1024, 64, 28, 8, "unit2", seed=2),
    "long": Workload("long", 8, 128, 128, 64, 128, 4, AGGREGATE, 32768, 2048,
                     128, 1, 4, "walk", seed=4),
}
for _m in (8, 16, 32, 64):
    for _r, _rn in ((AGGREGATE, "agg"), (FM, "fm")):
        WORKLOADS[f"sweep_m{_m}_{_rn}"] = Workload(
            f"sweep_m{_m}_{_rn}", 2, 128, 128, _m, 128, 4, _r, 512, 512,
            256, 1, 8, "unit2", seed=3)


def _rng(wl: Workload, g: int, tag: int, step: int) -> np.random.Generator:
    s, layer, kvg = wl.group_coords(g)
    ss = np.random.SeedSequence([wl.seed, s, layer, kvg, tag, step])
    return np.random.Generator(np.random.Philox(ss))


def _direction(wl: Workload, g: int) -> np.ndarray:
    u = _rng(wl, g, _TAG_DIR, _PROMPT).standard_normal(wl.d)
    return u / np.linalg.norm(u)


def _mean_scale(wl: Workload) -> float:
    return {"unit2": 2.0, "unit3": 3.0}[wl.k_mean]


def _walk_increments(wl: Workload, g: int, step: int, n: int) -> np.ndarray:
    xi = _rng(wl, g, _TAG_WALK, step).standard_normal((n, wl.d))
    return 0.01 * xi / np.linalg.norm(xi, axis=1, keepdims=True)


class GroupInputs:
    """Host-side inputs of one group: its prompt and its decode tokens.

    Decode tokens are produced in order (the ``walk`` mean carries state from
    one token to the next); ``token(n)`` for n = 0, 1, ... must be called in
    sequence or through ``tokens(n0, count)``."""

    def __init__(self, wl: Workload, g: int):
        self.wl, self.g = wl, g
        self._walk_pos = None
        self._next = 0

    def prompt(self):
        """(q [H][t][d], k [t][d], v [t][dv]) float32."""
        wl, g = self.wl, self.g
        q = _rng(wl, g, _TAG_Q, _PROMPT).standard_normal(
            (wl.heads_per_kv, wl.t, wl.d), dtype=np.float32)
        k = _rng(wl, g, _TAG_K, _PROMPT).standard_normal(
            (wl.t, wl.d), dtype=np.float32)
        v = _rng(wl, g, _TAG_V, _PROMPT).standard_normal(
            (wl.t, wl.dv), dtype=np.float32)
        if wl.k_mean == "walk":
            means = np.cumsum(_walk_increments(wl, g, _PROMPT, wl.t), axis=0)
            self._walk_pos = means[-1].copy()
            k = (k.astype(np.float64) + means).astype(np.float32)
        else:
            k = (k.astype(np.float64)
                 + _mean_scale(wl) * _direction(wl, g)).astype(np.float32)
        self._next = 0
        return q, k, v

    def token(self, n: int):
        """Decode token n (0-based): (q [H][d], k [d], v [dv]) float32."""
        wl, g = self.wl, self.g
        if n != self._next:
            raise ValueError("decode tokens must be drawn in order")
        q = _rng(wl, g, _TAG_Q, n).standard_normal(
            (wl.heads_per_kv, wl.d), dtype=np.float32)
        k = _rng(wl, g, _TAG_K, n).standard_normal(wl.d, dtype=np.float32)
        v = _rng(wl, g, _TAG_V, n).standard_normal(wl.dv, dtype=np.float32)
        if wl.k_mean == "walk":
            if self._walk_pos is None:
                raise ValueError("draw the prompt first")
            self._walk_pos = self._walk_pos + _walk_increments(wl, g, n, 1)[0]
            k = (k.astype(np.float64) + self._walk_pos).astype(np.float32)
        else:
            k = (k.astype(np.float64)
                 + _mean_scale(wl) * _direction(wl, g)).astype(np.float32)
        self._next = n + 1
        return q, k, v


def host_prompt_batch(wl: Workload, groups):
    """Stacked prompts of the given groups: q [n][H][t][d], k [n][t][d],
    v [n][t][dv], plus the per-group generators (positioned for token 0)."""
    gens = [GroupInputs(wl, g) for g in groups]
    parts = [gi.prompt() for gi in gens]
    q = np.stack([p[0] for p in parts])
    k = np.stack([p[1] for p in parts])
    v = np.stack([p[2] for p in parts])
    return q, k, v, gens


def host_token_batch(gens, n: int):
    """Decode token n of every generator: q [n][H][d], k [n][d], v [n][dv]."""
    parts = [gi.token(n) for gi in gens]
    return (np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
            np.stack([p[2] for p in parts]))


# ---------------------------------------------------------------- device fill
class DeviceFill:
    """Same distributions drawn with torch on a CUDA device, for groups no
    oracle reads and for the benchmark's bulk inputs.  Not bit-identical to
    the host streams (a different generator), only identically distributed.
    """

    def __init__(self, wl: Workload, device, seed: int = 12345):
        import torch
        self.torch = torch
        self.wl = wl
        self.dev = device
        self.gen = torch.Generator(device=device)
        self.gen.manual_seed(seed)
        self.n = wl.n_groups
        if wl.k_mean == "walk":
            self.mean = torch.zeros(self.n, wl.d, device=device)
        else:
            u = torch.randn(self.n, wl.d, device=device, generator=self.gen)
            self.mean = _mean_scale(wl) * u / u.norm(dim=1, keepdim=True)

    def _walk(self, rows: int):
        torch = self.torch
        xi = torch.randn(self.n, rows, self.wl.d, device=self.dev,
                         generator=self.gen)
        inc = 0.01 * xi / xi.norm(dim=2, keepdim=True)
        path = self.mean[:, None, :] + torch.cumsum(inc, dim=1)
        self.mean = path[:, -1, :].contiguous()
        return path

    def prompt_into(self, q, k, v, g0: int = 0):
        """Fill device tensors q [n][H][t][d], k [n][t][d], v [n][t][dv] for
        groups g0..g0+n in place (chunked to bound temporaries)."""
        torch = self.torch
        n = k.shape[0]
        q.normal_(generator=self.gen)
        v.normal_(generator=self.gen)
        k.normal_(generator=self.gen)
        if self.wl.k_mean == "walk":
            if g0 != 0 or n != self.n:
                raise ValueError("walk fill covers all groups at once")
            chunk = 1024
            for c0 in range(0, self.wl.t, chunk):
                rows = min(chunk, self.wl.t - c0)
                k[:, c0:c0 + rows] += self._walk(rows)
        else:
            k += self.mean[g0:g0 + n, None, :]
        torch.cuda.synchronize(self.dev)

    def tokens_into(self, q, k, v):
        """Fill decode inputs for S tokens: q [S][n][H][d], k [S][n][d],
        v [S][n][dv] (all groups)."""
        q.normal_(generator=self.gen)
        v.normal_(generator=self.gen)
        k.normal_(generator=self.gen)
        if self.wl.k_mean == "walk":
            path = self._walk(k.shape[0])          # [n][S][d]
            k += path.transpose(0, 1)
        else:
            k += self.mean[None, :, :]
