"""ctypes binding of libnys (include/nys.h): same names, argument marshalling only.

Every operation runs in the CUDA kernels of libnys.so.  Importing this module
raises ImportError if the library has not been built, and every call raises
NysError on a non-zero status: there is no fallback.

``NystromStates`` is a convenience wrapper that keeps the state buffer in a
torch tensor and passes torch tensors' device pointers and the current torch
stream to the C calls.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnys.so")

NYS_OK = 0
NYS_E_INVAL = -1
NYS_E_RANGE = -2
NYS_E_NOT_SEALED = -3
NYS_E_EXACT_ONLY = -4
NYS_E_BUF = -5
NYS_E_ALIGN = -6
NYS_E_CUDA = -7
NYS_E_UNSUPPORTED = -8
NYS_E_SCRATCH = -9
NYS_E_CAPACITY = -10
NYS_RECT_AGGREGATE = 0
NYS_RECT_FM = 1

# Every entry point include/nys.h declares.
EXPORTED = ("nys_memory_bytes", "nys_alloc_states", "nys_free_states",
            "nys_seal", "nys_step_batch", "nys_query", "nys_layout_of",
            "nys_mark_sealed", "nys_config_of", "nys_strerror",
            "nys_seal_static", "nys_seal_ragged", "nys_o1_begin", "nys_o1_push_q",
            "nys_o1_seal", "nys_o1_sealed", "nys_o1_step", "nys_o1_memory_bytes",
            "nys_o1_states", "nys_o1_free", "nys_debug_stall_once",
            "nys_debug_stall_replay_once")


class NysConfig(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("w", ctypes.c_int32),
                ("sink", ctypes.c_int32), ("heads_per_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("rect", ctypes.c_int32), ("exact_cap", ctypes.c_int32)]


class NysLayout(ctypes.Structure):
    _fields_ = [("total_bytes", ctypes.c_size_t),
                ("off_win_k", ctypes.c_size_t), ("off_win_v", ctypes.c_size_t),
                ("off_sink_k", ctypes.c_size_t), ("off_sink_v", ctypes.c_size_t),
                ("off_k_tilde", ctypes.c_size_t), ("off_q_tilde", ctypes.c_size_t),
                ("off_mu", ctypes.c_size_t), ("off_t_hat", ctypes.c_size_t),
                ("off_z_hat", ctypes.c_size_t), ("off_m_max", ctypes.c_size_t),
                ("off_t_lo", ctypes.c_size_t), ("off_z_lo", ctypes.c_size_t),
                ("off_far_len", ctypes.c_size_t), ("off_ints", ctypes.c_size_t),
                ("off_exact_k", ctypes.c_size_t), ("off_exact_v", ctypes.c_size_t),
                ("n_groups", ctypes.c_int64), ("ints_per_group", ctypes.c_int32)]


class NysGroupInfo(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("m_eff", ctypes.c_int32),
                ("t", ctypes.c_int32), ("win_len", ctypes.c_int32),
                ("win_head", ctypes.c_int32), ("status", ctypes.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with "
            "`python -m streaming_nystr_landmark_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I64, I32, VP = ctypes.POINTER, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    sig = {
        "nys_memory_bytes": [P(NysConfig), I64, P(ctypes.c_size_t)],
        "nys_alloc_states": [P(NysConfig), I64, VP, ctypes.c_size_t, P(VP)],
        "nys_free_states": [VP],
        "nys_seal": [VP, I64, I64, I32, VP, VP, VP, VP],
        "nys_step_batch": [VP, I64, I64, VP, VP, VP, VP, VP],
        "nys_query": [VP, I64, P(NysGroupInfo), P(I32), VP],
        "nys_layout_of": [VP, P(VP), P(NysLayout)],
        "nys_mark_sealed": [VP, I64, I64],
        "nys_config_of": [VP, P(NysConfig), P(I64)],
        "nys_strerror": [ctypes.c_int],
        "nys_seal_static": [VP, I64, I64, I32, VP, VP, VP, VP],
        "nys_seal_ragged": [VP, I64, I64, P(I32), VP, VP, VP, VP],
        "nys_o1_begin": [P(NysConfig), I32, I32, I32, I32, P(VP)],
        "nys_o1_push_q": [VP, VP, VP],
        "nys_o1_seal": [VP, VP, VP, I32, I32, VP, P(I32)],
        "nys_o1_sealed": [VP, P(I32)],
        "nys_o1_step": [VP, VP, VP, VP, VP, VP],
        "nys_o1_memory_bytes": [VP, P(ctypes.c_size_t)],
        "nys_o1_states": [VP, P(VP)],
        "nys_o1_free": [VP],
        "nys_debug_stall_once": [VP, I32],
        "nys_debug_stall_replay_once": [VP],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "nys_strerror" else ctypes.c_int
    return lib


_lib = _load()


class NysError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {nys_strerror(code)} (status {code})")


def _check(code: int, where: str):
    if code != NYS_OK:
        raise NysError(code, where)


def nys_strerror(code: int) -> str:
    return _lib.nys_strerror(code).decode()


def make_config(m, w, sink, heads_per_kv, d, dv, rect=NYS_RECT_AGGREGATE,
                exact_cap=0) -> NysConfig:
    return NysConfig(m, w, sink, heads_per_kv, d, dv, rect, exact_cap)


def nys_memory_bytes(cfg: NysConfig, n_groups: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.nys_memory_bytes(ctypes.byref(cfg), n_groups, ctypes.byref(out)),
           "nys_memory_bytes")
    return out.value


def nys_alloc_states(cfg: NysConfig, n_groups: int, dev_buf: int = 0,
                     buf_bytes: int = 0) -> int:
    h = ctypes.c_void_p(0)
    _check(_lib.nys_alloc_states(ctypes.byref(cfg), n_groups, dev_buf or None,
                                 buf_bytes, ctypes.byref(h)), "nys_alloc_states")
    return h.value


def nys_free_states(handle: int):
    _check(_lib.nys_free_states(handle), "nys_free_states")


def nys_seal(handle, g0, n, t, q, k, v, stream=0):
    _check(_lib.nys_seal(handle, g0, n, t, q, k, v, stream or None), "nys_seal")


def nys_seal_static(handle, g0, n, t, q, k, v, stream=0):
    """nys_seal with the library's static workspace instead of an allocation
    (for callers that cannot allocate device memory while they run)."""
    _check(_lib.nys_seal_static(handle, g0, n, t, q, k, v, stream or None),
           "nys_seal_static")


def nys_seal_ragged(handle, g0, t_list, q, k, v, stream=0):
    """Seal len(t_list) groups from g0 on prompts of the given lengths,
    packed back to back (see include/nys.h)."""
    n = len(t_list)
    arr = (ctypes.c_int32 * max(n, 1))(*t_list)
    _check(_lib.nys_seal_ragged(handle, g0, n, arr, q, k, v, stream or None),
           "nys_seal_ragged")


def nys_step_batch(handle, g0, n, q, k, v, out, stream=0):
    _check(_lib.nys_step_batch(handle, g0, n, q, k, v, out, stream or None),
           "nys_step_batch")


def nys_query(handle, g, heads, stream=0):
    info = NysGroupInfo()
    far = (ctypes.c_int32 * heads)()
    _check(_lib.nys_query(handle, g, ctypes.byref(info), far, stream or None),
           "nys_query")
    return ({"mode": info.mode, "m_eff": info.m_eff, "t": info.t,
             "win_len": info.win_len, "win_head": info.win_head,
             "status": info.status}, list(far))


def nys_debug_stall_once(handle, stage):
    _check(_lib.nys_debug_stall_once(handle, stage), "nys_debug_stall_once")


def nys_debug_stall_replay_once(handle):
    _check(_lib.nys_debug_stall_replay_once(handle), "nys_debug_stall_replay_once")


def nys_layout_of(handle):
    base = ctypes.c_void_p(0)
    lay = NysLayout()
    _check(_lib.nys_layout_of(handle, ctypes.byref(base), ctypes.byref(lay)),
           "nys_layout_of")
    return base.value, lay


def nys_mark_sealed(handle, g0, n):
    _check(_lib.nys_mark_sealed(handle, g0, n), "nys_mark_sealed")


def nys_config_of(handle):
    cfg = NysConfig()
    n = ctypes.c_int64(0)
    _check(_lib.nys_config_of(handle, ctypes.byref(cfg), ctypes.byref(n)),
           "nys_config_of")
    return cfg, n.value


# ---------------------------------------------------------------- torch wrapper
def _ptr(t, dtype, shape, where):
    import torch
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{where}: need a contiguous CUDA {dtype} tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{where}: shape {tuple(t.shape)} != {tuple(shape)}")
    return t.data_ptr()


class NystromStates:
    """A batch of group states in one torch-owned device buffer."""

    def __init__(self, m, w, sink, heads_per_kv, d, dv, n_groups,
                 rect=NYS_RECT_AGGREGATE, device="cuda", exact_cap=0):
        import torch
        self.torch = torch
        self.cfg = make_config(m, w, sink, heads_per_kv, d, dv, rect, exact_cap)
        self.n_groups = n_groups
        self.device = torch.device(device)
        nbytes = nys_memory_bytes(self.cfg, n_groups)
        self.buf = torch.empty(max(nbytes, 1) + 256, dtype=torch.uint8,
                               device=self.device)
        base = self.buf.data_ptr()
        self._off = (-base) % 256
        self.handle = nys_alloc_states(self.cfg, n_groups, base + self._off, nbytes)
        self.base, self.layout = nys_layout_of(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            nys_free_states(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def seal(self, q, k, v, g0=0, n=None):
        c = self.cfg
        n = k.shape[0] if n is None else n
        t = k.shape[1]
        torch = self.torch
        nys_seal(self.handle, g0, n, t,
                 _ptr(q, torch.float32, (n, c.heads_per_kv, t, c.d), "q"),
                 _ptr(k, torch.float32, (n, t, c.d), "k"),
                 _ptr(v, torch.float32, (n, t, c.dv), "v"), self._stream())

    def seal_ragged(self, t_list, q, k, v, g0=0):
        """Seal groups g0.. on prompts of lengths t_list packed back to back:
        k [sum t][d], v [sum t][dv], q [H * sum t][d] (per group [H][t][d])."""
        c = self.cfg
        torch = self.torch
        total = int(sum(t_list))
        nys_seal_ragged(self.handle, g0, list(t_list),
                        _ptr(q, torch.float32, (c.heads_per_kv * total, c.d), "q"),
                        _ptr(k, torch.float32, (total, c.d), "k"),
                        _ptr(v, torch.float32, (total, c.dv), "v"), self._stream())

    def step(self, q, k, v, out, g0=0, n=None):
        c = self.cfg
        n = k.shape[0] if n is None else n
        torch = self.torch
        nys_step_batch(self.handle, g0, n,
                       _ptr(q, torch.float32, (n, c.heads_per_kv, c.d), "q"),
                       _ptr(k, torch.float32, (n, c.d), "k"),
                       _ptr(v, torch.float32, (n, c.dv), "v"),
                       _ptr(out, torch.float32, (n, c.heads_per_kv, c.dv), "out"),
                       self._stream())
        return out

    def step_host(self, hq, hk, hv, hout, dq, dk, dv, dout):
        """One token from pinned host buffers: copy q/k/v to the device
        staging tensors, launch nys_step_batch, copy the outputs back to
        ``hout``; everything is enqueued on the current stream."""
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        self.step(dq, dk, dv, dout)
        hout.copy_(dout, non_blocking=True)
        return hout

    def host_pipeline(self, n=None, depth=2):
        """A pipelined host-buffer driver for this handle (see HostPipeline)."""
        return HostPipeline(self, self.n_groups if n is None else n, depth)

    def query(self, g):
        return nys_query(self.handle, g, self.cfg.heads_per_kv, self._stream())

    def debug_stall_once(self, stage):
        """Test hook: the next step's first CTA withholds ring stage `stage`,
        so its bounded waits run out and its groups report status 1."""
        nys_debug_stall_once(self.handle, stage)

    def debug_stall_replay_once(self):
        """Test hook: the next seal's tensor-core replay withholds its first
        CTA's first MMAs; that group reports status 3."""
        nys_debug_stall_replay_once(self.handle)

    def region(self, name):
        """A torch view of one state region, shaped as nys_layout documents."""
        torch = self.torch
        c, G = self.cfg, self.n_groups
        H, m = c.heads_per_kv, c.m
        shapes = {
            "win_k": (torch.float32, (G, c.w, c.d)),
            "win_v": (torch.float32, (G, c.w, c.dv)),
            "sink_k": (torch.float32, (G, c.sink, c.d)),
            "sink_v": (torch.float32, (G, c.sink, c.dv)),
            "k_tilde": (torch.float32, (G, m, c.d)),
            "q_tilde": (torch.float32, (G, H, m, c.d)),
            "mu": (torch.float32, (G, H, m, m)),
            "t_hat": (torch.float32, (G, H, m, c.dv)),
            "z_hat": (torch.float32, (G, H, m)),
            "m_max": (torch.float32, (G, H, m)),
            "t_lo": (torch.bfloat16, (G, H, m, c.dv)),
            "z_lo": (torch.float32, (G, H, m)),
            "far_len": (torch.int32, (G, H)),
            "ints": (torch.int32, (G, self.layout.ints_per_group)),
            "exact_k": (torch.float32, (G, c.exact_cap, c.d)),
            "exact_v": (torch.float32, (G, c.exact_cap, c.dv)),
        }
        dtype, shape = shapes[name]
        off = getattr(self.layout, "off_" + name) + self._off
        count = 1
        for s in shape:
            count *= s
        size = 2 if dtype == torch.bfloat16 else 4
        raw = self.buf[off: off + size * count]
        return raw.view(dtype).view(shape)

    def far_numerator(self):
        """T^ = t_hat + t_lo as float64 on the host (test helper)."""
        return (self.region("t_hat").double() + self.region("t_lo").double()).cpu().numpy()

    def far_denominator(self):
        """Z^ = z_hat + z_lo as float64 on the host (test helper)."""
        return (self.region("z_hat").double() + self.region("z_lo").double()).cpu().numpy()

    def mark_sealed(self, g0=0, n=None):
        nys_mark_sealed(self.handle, g0, self.n_groups if n is None else n)


class HostPipeline:
    """Decode tokens from pinned host buffers with copies overlapped.

    Each ``submit`` enqueues, for one token: the host->device copy of q, k, v
    on an upload stream into one of ``depth`` device staging slots, the
    decode launch on the compute stream once that copy has landed, and the
    device->host copy of the outputs on a separate download stream once the
    launch is done.  Token n+1's inputs therefore travel while token n
    computes (uploads never queue behind downloads), and a staging slot is
    reused only after the launch that read it has finished.
    ``synchronize`` waits for everything submitted.  All ordering is by CUDA
    events; the decode itself is nys_step_batch.
    """

    def __init__(self, states, n, depth=2):
        import torch
        self.torch = torch
        self.st = states
        self.n = n
        c = states.cfg
        dev = states.device
        self.compute = torch.cuda.current_stream(dev)
        self.copy = torch.cuda.Stream(dev)      # uploads
        self.down = torch.cuda.Stream(dev)      # downloads
        mk = lambda *shape: torch.empty(shape, device=dev)
        self.slots = [dict(q=mk(n, c.heads_per_kv, c.d), k=mk(n, c.d), v=mk(n, c.dv),
                           out=mk(n, c.heads_per_kv, c.dv),
                           loaded=torch.cuda.Event(), done=torch.cuda.Event(),
                           drained=torch.cuda.Event())
                      for _ in range(depth)]
        for sl in self.slots:
            sl["done"].record(self.compute)
            sl["drained"].record(self.down)
        self.i = 0

    def submit(self, hq, hk, hv, hout):
        sl = self.slots[self.i % len(self.slots)]
        self.i += 1
        with self.torch.cuda.stream(self.copy):
            self.copy.wait_event(sl["done"])       # the last launch read this slot
            sl["q"].copy_(hq, non_blocking=True)
            sl["k"].copy_(hk, non_blocking=True)
            sl["v"].copy_(hv, non_blocking=True)
            sl["loaded"].record(self.copy)
        self.compute.wait_event(sl["loaded"])
        self.compute.wait_event(sl["drained"])      # its previous outputs left
        self.st.step(sl["q"], sl["k"], sl["v"], sl["out"])
        sl["done"].record(self.compute)
        with self.torch.cuda.stream(self.down):
            self.down.wait_event(sl["done"])
            hout.copy_(sl["out"], non_blocking=True)
            sl["drained"].record(self.down)

    def synchronize(self):
        self.torch.cuda.synchronize(self.st.device)


class O1Layer:
    """One attention layer's O(1) override for a batch of sequences (the
    LayerKvCache o1 lifecycle: begin -> push_q per prompt position -> seal ->
    step per decode token), over the nys_o1_* calls."""

    def __init__(self, m, w, sink, d, dv, batch, num_heads, num_kv_heads, max_prompt,
                 rect=NYS_RECT_AGGREGATE, exact_cap=0, device="cuda"):
        import torch
        self.torch = torch
        self.device = torch.device(device)
        self.cfg = make_config(m, w, sink, 1, d, dv, rect, exact_cap)
        self.batch, self.num_heads, self.num_kv = batch, num_heads, num_kv_heads
        h = ctypes.c_void_p(0)
        _check(_lib.nys_o1_begin(ctypes.byref(self.cfg), batch, num_heads, num_kv_heads,
                                 max_prompt, ctypes.byref(h)), "nys_o1_begin")
        self.handle = h.value

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def push_q(self, q_all):
        c = self.cfg
        _check(_lib.nys_o1_push_q(self.handle, _ptr(q_all, self.torch.float32,
                                                    (self.batch, self.num_heads, c.d), "q_all"),
                                  self._stream()), "nys_o1_push_q")

    def seal(self, k, v, kv_dense=True):
        """k [batch][num_kv][t][d], v [..][dv]; True when sealed."""
        c = self.cfg
        t = k.shape[2]
        flag = ctypes.c_int32(0)
        _check(_lib.nys_o1_seal(
            self.handle,
            _ptr(k, self.torch.float32, (self.batch, self.num_kv, t, c.d), "k"),
            _ptr(v, self.torch.float32, (self.batch, self.num_kv, t, c.dv), "v"),
            t, int(bool(kv_dense)), self._stream(), ctypes.byref(flag)), "nys_o1_seal")
        return bool(flag.value)

    def sealed(self):
        flag = ctypes.c_int32(0)
        _check(_lib.nys_o1_sealed(self.handle, ctypes.byref(flag)), "nys_o1_sealed")
        return bool(flag.value)

    def step(self, q_all, k_new, v_new, out):
        c, f = self.cfg, self.torch.float32
        _check(_lib.nys_o1_step(
            self.handle, _ptr(q_all, f, (self.batch, self.num_heads, c.d), "q_all"),
            _ptr(k_new, f, (self.batch, self.num_kv, c.d), "k_new"),
            _ptr(v_new, f, (self.batch, self.num_kv, c.dv), "v_new"),
            _ptr(out, f, (self.batch, self.num_heads, c.dv), "out"), self._stream()),
            "nys_o1_step")
        return out

    def memory_bytes(self):
        out = ctypes.c_size_t(0)
        _check(_lib.nys_o1_memory_bytes(self.handle, ctypes.byref(out)), "nys_o1_memory_bytes")
        return out.value

    def close(self):
        if getattr(self, "handle", None):
            _check(_lib.nys_o1_free(self.handle), "nys_o1_free")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
