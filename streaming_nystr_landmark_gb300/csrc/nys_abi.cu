// Host side of the libnys C ABI (declared in include/nys.h): argument
// checks, the state-buffer layout, handle bookkeeping and kernel launches.
// Every check runs before anything is enqueued; nothing here aborts.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <cmath>
#include <new>
#include <vector>

#include "nys_internal.h"

struct nys_states {
  nys_config cfg;
  int64_t n_groups;
  void* base;
  bool owned;
  nys_layout lay;
  std::vector<uint8_t> sealed;  // host record of groups with a sealed state
  std::vector<int32_t> exact_len;  // keys held by exact-only groups, -1 otherwise
  int64_t n_exact;                 // how many groups are exact-only
  int debug_skip;                  // test hook for the next decode launch
  int debug_replay;                // test hook for the next seal's replay
  int device;
  nys::SealFork fork;              // the seal's second stream, made at the first seal
};

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kWorkspaceBudget = size_t(512) << 20;  // per seal chunk

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// The seal's side stream and its two events, made once per handle; if any
// of them cannot be made the seal stays on the caller's stream.
const nys::SealFork& seal_fork(nys_states* st) {
  nys::SealFork& f = st->fork;
  bool failed = false;
  if (!f.side && cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking) != cudaSuccess) {
    f.side = nullptr;
    failed = true;
  }
  if (!f.forked && cudaEventCreateWithFlags(&f.forked, cudaEventDisableTiming) != cudaSuccess) {
    f.forked = nullptr;
    failed = true;
  }
  if (!f.joined && cudaEventCreateWithFlags(&f.joined, cudaEventDisableTiming) != cudaSuccess) {
    f.joined = nullptr;
    failed = true;
  }
  if (failed) cudaGetLastError();  // only this call's failure: no second stream
  return f;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_config(const nys_config* c) {
  if (!c) return NYS_E_INVAL;
  if (c->m < 4 || c->w < 1 || c->sink < 0 || c->heads_per_kv < 1) return NYS_E_INVAL;
  if (c->d <= 0 || c->dv <= 0 || (c->d & 3) || (c->dv & 3)) return NYS_E_INVAL;
  if (c->rect != NYS_RECT_AGGREGATE && c->rect != NYS_RECT_FM) return NYS_E_INVAL;
  if (c->exact_cap < 0) return NYS_E_INVAL;
  if (c->exact_cap > nys::kMaxExactCap) return NYS_E_UNSUPPORTED;
  if (c->m > nys::kMaxM || c->d > nys::kMaxDim || c->dv > nys::kMaxDim ||
      c->heads_per_kv > nys::kMaxHeads || (int64_t)c->sink + c->w > nys::kMaxNear)
    return NYS_E_UNSUPPORTED;
  return NYS_OK;
}

// Lay the regions out one after another, each on a 256-byte boundary.
bool make_layout(const nys_config& c, int64_t G, nys_layout* L) {
  if (G < 0) return false;
  const double approx = (double)G * ((double)c.w * (c.d + c.dv) + (double)c.sink * (c.d + c.dv) +
                                     (double)c.m * c.d +
                                     (double)c.heads_per_kv * c.m * (c.d + c.m + c.dv + 2) +
                                     c.heads_per_kv + 8) * 4.0;
  if (approx > 9.0e18) return false;
  const size_t g = (size_t)G, H = (size_t)c.heads_per_kv, m = (size_t)c.m;
  size_t o = 0;
  auto region = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  std::memset(L, 0, sizeof(*L));
  L->off_win_k = region(g * c.w * c.d * 4);
  L->off_win_v = region(g * c.w * c.dv * 4);
  L->off_sink_k = region(g * c.sink * c.d * 4);
  L->off_sink_v = region(g * c.sink * c.dv * 4);
  L->off_k_tilde = region(g * m * c.d * 4);
  L->off_q_tilde = region(g * H * m * c.d * 4);
  L->off_mu = region(g * H * m * m * 4);
  L->off_t_hat = region(g * H * m * c.dv * 4);
  L->off_z_hat = region(g * H * m * 4);
  L->off_m_max = region(g * H * m * 4);
  L->off_t_lo = region(g * H * m * c.dv * 2);
  L->off_z_lo = region(g * H * m * 4);
  L->off_far_len = region(g * H * 4);
  L->off_ints = region(g * nys::kIntsPerGroup * 4);
  L->off_exact_k = region(g * (size_t)c.exact_cap * c.d * 4);
  L->off_exact_v = region(g * (size_t)c.exact_cap * c.dv * 4);
  L->total_bytes = o;
  L->n_groups = G;
  L->ints_per_group = nys::kIntsPerGroup;
  return true;
}

nys::DevState dev_state(const nys_states* st) {
  nys::DevState s;
  char* b = static_cast<char*>(st->base);
  const nys_layout& L = st->lay;
  s.win_k = reinterpret_cast<float*>(b + L.off_win_k);
  s.win_v = reinterpret_cast<float*>(b + L.off_win_v);
  s.sink_k = reinterpret_cast<float*>(b + L.off_sink_k);
  s.sink_v = reinterpret_cast<float*>(b + L.off_sink_v);
  s.k_tilde = reinterpret_cast<float*>(b + L.off_k_tilde);
  s.q_tilde = reinterpret_cast<float*>(b + L.off_q_tilde);
  s.mu = reinterpret_cast<float*>(b + L.off_mu);
  s.t_hat = reinterpret_cast<float*>(b + L.off_t_hat);
  s.z_hat = reinterpret_cast<float*>(b + L.off_z_hat);
  s.m_max = reinterpret_cast<float*>(b + L.off_m_max);
  s.t_lo = reinterpret_cast<uint16_t*>(b + L.off_t_lo);
  s.z_lo = reinterpret_cast<float*>(b + L.off_z_lo);
  s.far_len = reinterpret_cast<int32_t*>(b + L.off_far_len);
  s.ints = reinterpret_cast<int32_t*>(b + L.off_ints);
  s.exact_k = reinterpret_cast<float*>(b + L.off_exact_k);
  s.exact_v = reinterpret_cast<float*>(b + L.off_exact_v);
  s.exact_cap = st->cfg.exact_cap;
  s.m = st->cfg.m;
  s.w = st->cfg.w;
  s.sink = st->cfg.sink;
  s.heads = st->cfg.heads_per_kv;
  s.d = st->cfg.d;
  s.dv = st->cfg.dv;
  s.rect = st->cfg.rect;
  // 1/sqrt(d) in f32, as nystrom.rs prefill_shared computes it.
  s.scale = 1.0f / std::sqrt((float)st->cfg.d);
  return s;
}

int check_range(const nys_states* st, int64_t g0, int64_t n) {
  if (g0 < 0 || n < 0 || g0 > st->n_groups || n > st->n_groups - g0) return NYS_E_RANGE;
  if (n > (int64_t)INT32_MAX / 64) return NYS_E_RANGE;  // grid limit with head blocks
  return NYS_OK;
}

std::atomic<bool> g_clamp_said{false};

// Host record: groups [g0, g0+n) now hold landmark-path states.
void forget_exact(nys_states* st, int64_t g0, int64_t n) {
  if (!st->n_exact) return;
  for (int64_t g = g0; g < g0 + n; ++g) {
    if (st->exact_len[(size_t)g] >= 0) {
      st->exact_len[(size_t)g] = -1;
      --st->n_exact;
    }
  }
}

}  // namespace

namespace nys {

int plan_seal(nys_states* st, int64_t g0, int64_t n, int32_t t, const float* q,
              const float* k, const float* v, SealPlan* plan) {
  if (!st || !plan) return NYS_E_INVAL;
  int rc = check_range(st, g0, n);
  if (rc) return rc;
  const nys_config& c = st->cfg;
  if (t < 1) return NYS_E_RANGE;
  plan->ds = dev_state(st);
  // nystrom.rs, prefill_shared: short prompts skip the skeleton entirely and
  // keep every key exact (exact-only mode), which needs the exact region.
  if ((int64_t)t <= (int64_t)c.w + c.sink + 8) {
    if (c.exact_cap == 0) return NYS_E_EXACT_ONLY;
    if (t > c.exact_cap) return NYS_E_RANGE;
    if (n > 0) {
      if (!k || !v) return NYS_E_INVAL;
      if (!aligned16(k) || !aligned16(v)) return NYS_E_ALIGN;
    }
    plan->exact = true;
    plan->m_eff = 0;
    return NYS_OK;
  }
  if (n > 0) {
    if (!q || !k || !v) return NYS_E_INVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return NYS_E_ALIGN;
  }
  plan->exact = false;
  plan->m_eff = std::min(std::max(t / 8, 4), c.m);
  if (n > 0 && plan->m_eff < c.m && !g_clamp_said.exchange(true)) {
    std::fprintf(stderr,
                 "nys: landmark budget m=%d clamped to m_eff=%d: the prompt is %d tokens and "
                 "the landmarks take t/8; seal at least %d tokens to use the whole budget\n",
                 c.m, plan->m_eff, t, c.m * 8);
  }
  return NYS_OK;
}

int run_exact_seal(nys_states* st, int64_t g0, int64_t n, int32_t t, const float* k,
                   const float* v, cudaStream_t stream) {
  if (n == 0) return NYS_OK;
  if (launch_exact_seal(dev_state(st), g0, n, t, k, v, stream) != cudaSuccess) return NYS_E_CUDA;
  std::memset(st->sealed.data() + g0, 1, (size_t)n);
  for (int64_t g = g0; g < g0 + n; ++g) {
    if (st->exact_len[(size_t)g] < 0) ++st->n_exact;
    st->exact_len[(size_t)g] = t;
  }
  return NYS_OK;
}

void record_sealed(nys_states* st, int64_t g0, int64_t n) {
  if (n > 0) std::memset(st->sealed.data() + g0, 1, (size_t)n);
  forget_exact(st, g0, n);
}

}  // namespace nys

extern "C" {

const char* nys_strerror(int status) {
  switch (status) {
    case NYS_OK: return "ok";
    case NYS_E_INVAL: return "invalid argument or geometry";
    case NYS_E_RANGE: return "group range or prompt length out of range";
    case NYS_E_NOT_SEALED: return "group not sealed: run nys_seal before nys_step_batch";
    case NYS_E_EXACT_ONLY:
      return "prompt too short (t <= w + sink + 8): exact-only mode is not carried on the GPU";
    case NYS_E_BUF: return "device buffer smaller than nys_memory_bytes";
    case NYS_E_ALIGN: return "pointer not aligned (inputs 16 bytes, state buffer 256 bytes)";
    case NYS_E_CUDA: return "CUDA error";
    case NYS_E_UNSUPPORTED:
      return "geometry beyond kernel limits (m <= 64, d, dv <= 256, heads <= 64, sink + w <= 2048)";
    case NYS_E_CAPACITY:
      return "an exact-only group would hold more than exact_cap keys";
    case NYS_E_SCRATCH:
      return "one group's seal workspace, (1 + heads_per_kv) * m * d * 8 bytes, exceeds the "
             "4 MiB static scratch of nys_seal_static; use nys_seal";
    default: return "unknown status";
  }
}

int nys_memory_bytes(const nys_config* cfg, int64_t n_groups, size_t* device_bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!device_bytes || n_groups < 0) return NYS_E_INVAL;
  nys_layout L;
  if (!make_layout(*cfg, n_groups, &L)) return NYS_E_INVAL;
  *device_bytes = L.total_bytes;
  return NYS_OK;
}

int nys_alloc_states(const nys_config* cfg, int64_t n_groups, void* dev_buf,
                     size_t buf_bytes, nys_states** out) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!out || n_groups < 0) return NYS_E_INVAL;
  *out = nullptr;
  nys_layout L;
  if (!make_layout(*cfg, n_groups, &L)) return NYS_E_INVAL;
  if (dev_buf) {
    if (buf_bytes < L.total_bytes) return NYS_E_BUF;
    if (reinterpret_cast<uintptr_t>(dev_buf) % kAlign) return NYS_E_ALIGN;
  }
  nys_states* st = new (std::nothrow) nys_states();
  if (!st) return NYS_E_INVAL;
  st->cfg = *cfg;
  st->n_groups = n_groups;
  st->lay = L;
  st->owned = (dev_buf == nullptr);
  st->base = dev_buf;
  if (cudaGetDevice(&st->device) != cudaSuccess) {
    delete st;
    return NYS_E_CUDA;
  }
  if (st->owned && L.total_bytes) {
    if (cudaMalloc(&st->base, L.total_bytes) != cudaSuccess) {
      delete st;
      return NYS_E_CUDA;
    }
  }
  if (L.total_bytes && cudaMemset(st->base, 0, L.total_bytes) != cudaSuccess) {
    if (st->owned) cudaFree(st->base);
    delete st;
    return NYS_E_CUDA;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    if (st->owned) cudaFree(st->base);
    delete st;
    return NYS_E_CUDA;
  }
  st->sealed.assign((size_t)n_groups, 0);
  st->exact_len.assign((size_t)n_groups, -1);
  st->n_exact = 0;
  st->debug_skip = -1;
  st->debug_replay = 0;
  *out = st;
  return NYS_OK;
}

int nys_free_states(nys_states* st) {
  if (!st) return NYS_OK;
  int rc = NYS_OK;
  if (st->owned && st->base && cudaFree(st->base) != cudaSuccess) rc = NYS_E_CUDA;
  if (st->fork.side && cudaStreamDestroy(st->fork.side) != cudaSuccess) rc = NYS_E_CUDA;
  if (st->fork.forked && cudaEventDestroy(st->fork.forked) != cudaSuccess) rc = NYS_E_CUDA;
  if (st->fork.joined && cudaEventDestroy(st->fork.joined) != cudaSuccess) rc = NYS_E_CUDA;
  delete st;
  return rc;
}

int nys_seal(nys_states* st, int64_t g0, int64_t n, int32_t t, const float* q,
             const float* k, const float* v, void* stream) {
  nys::SealPlan plan;
  int rc = nys::plan_seal(st, g0, n, t, q, k, v, &plan);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan.exact) return nys::run_exact_seal(st, g0, n, t, k, v, s);
  if (n == 0) return NYS_OK;
  const nys_config& c = st->cfg;
  const int m_eff = plan.m_eff;
  const nys::DevState& ds = plan.ds;
  const size_t per = nys::seal_workspace_bytes_per_group(ds);
  int64_t chunk = (int64_t)(kWorkspaceBudget / per);
  if (chunk < 1) chunk = 1;
  if (chunk > n) chunk = n;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, per * (size_t)chunk, s) != cudaSuccess) return NYS_E_CUDA;
  cudaError_t e = cudaSuccess;
  const int64_t H = c.heads_per_kv;
  const int stall = st->debug_replay;
  st->debug_replay = 0;
  for (int64_t a = 0; a < n && e == cudaSuccess; a += chunk) {
    const int64_t nb = std::min(chunk, n - a);
    e = nys::launch_seal(ds, g0 + a, nb, t, m_eff, q + a * H * (int64_t)t * c.d,
                         k + a * (int64_t)t * c.d, v + a * (int64_t)t * c.dv,
                         static_cast<double*>(ws), s, a == 0 ? stall : 0, seal_fork(st));
  }
  const cudaError_t ef = cudaFreeAsync(ws, s);
  if (e != cudaSuccess || ef != cudaSuccess) return NYS_E_CUDA;
  std::memset(st->sealed.data() + g0, 1, (size_t)n);
  forget_exact(st, g0, n);
  return NYS_OK;
}

int nys_seal_ragged(nys_states* st, int64_t g0, int64_t n, const int32_t* t_host,
                    const float* q, const float* k, const float* v, void* stream) {
  if (!st) return NYS_E_INVAL;
  int rc = check_range(st, g0, n);
  if (rc) return rc;
  if (n == 0) return NYS_OK;
  if (!t_host || !q || !k || !v) return NYS_E_INVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return NYS_E_ALIGN;
  const nys_config& c = st->cfg;
  // Per-group geometry, packed for one upload: t, m_eff (int32 each), then
  // the first row of every group's prompt (int64).
  std::vector<int32_t> ti((size_t)n), mi((size_t)n);
  std::vector<int64_t> off((size_t)n);
  int64_t rows = 0;
  int max_me = 0, min_me = c.m, clamp_t = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t t = t_host[i];
    if (t < 1) return NYS_E_RANGE;
    if ((int64_t)t <= (int64_t)c.w + c.sink + 8) return NYS_E_EXACT_ONLY;
    const int me = std::min(std::max(t / 8, 4), c.m);
    ti[(size_t)i] = t;
    mi[(size_t)i] = me;
    off[(size_t)i] = rows;
    rows += t;
    max_me = std::max(max_me, me);
    if (me < min_me) {
      min_me = me;
      clamp_t = t;
    }
  }
  if (min_me < c.m && !g_clamp_said.exchange(true)) {
    std::fprintf(stderr,
                 "nys: landmark budget m=%d clamped to m_eff=%d: the prompt is %d tokens and "
                 "the landmarks take t/8; seal at least %d tokens to use the whole budget\n",
                 c.m, min_me, clamp_t, c.m * 8);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const nys::DevState ds = dev_state(st);
  const size_t per = nys::seal_workspace_bytes_per_group(ds);
  int64_t chunk = (int64_t)(kWorkspaceBudget / per);
  if (chunk < 1) chunk = 1;
  if (chunk > n) chunk = n;
  const size_t meta_bytes = (size_t)n * 16;
  void* ws = nullptr;
  void* meta = nullptr;
  if (cudaMallocAsync(&ws, per * (size_t)chunk, s) != cudaSuccess) return NYS_E_CUDA;
  if (cudaMallocAsync(&meta, meta_bytes, s) != cudaSuccess) {
    cudaFreeAsync(ws, s);
    return NYS_E_CUDA;
  }
  int64_t* off_dev = static_cast<int64_t*>(meta);
  int32_t* t_dev = reinterpret_cast<int32_t*>(off_dev + n);
  int32_t* me_dev = t_dev + n;
  cudaError_t e = cudaMemcpyAsync(off_dev, off.data(), (size_t)n * 8, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(t_dev, ti.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(me_dev, mi.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s);
  for (int64_t a = 0; a < n && e == cudaSuccess; a += chunk) {
    const int64_t nb = std::min(chunk, n - a);
    const nys::SealGeom sg{0, 0, t_dev + a, me_dev + a, off_dev + a};
    e = nys::launch_seal_geom(ds, g0 + a, nb, sg, max_me, q, k, v, static_cast<double*>(ws), s,
                              0, seal_fork(st));
  }
  const cudaError_t f1 = cudaFreeAsync(ws, s), f2 = cudaFreeAsync(meta, s);
  // The host arrays above were staged by the copies before they returned.
  if (e != cudaSuccess || f1 != cudaSuccess || f2 != cudaSuccess) return NYS_E_CUDA;
  std::memset(st->sealed.data() + g0, 1, (size_t)n);
  forget_exact(st, g0, n);
  return NYS_OK;
}

int nys_step_batch(nys_states* st, int64_t g0, int64_t n, const float* q,
                   const float* k, const float* v, float* out, void* stream) {
  if (!st) return NYS_E_INVAL;
  int rc = check_range(st, g0, n);
  if (rc) return rc;
  if (n == 0) return NYS_OK;
  if (!q || !k || !v || !out) return NYS_E_INVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return NYS_E_ALIGN;
  if (std::memchr(st->sealed.data() + g0, 0, (size_t)n)) return NYS_E_NOT_SEALED;
  int64_t exact_here = 0;
  if (st->n_exact) {
    for (int64_t g = g0; g < g0 + n; ++g) {
      const int32_t len = st->exact_len[(size_t)g];
      if (len < 0) continue;
      if (len >= st->cfg.exact_cap) return NYS_E_CAPACITY;
      ++exact_here;
    }
  }
  const nys::DevState ds = dev_state(st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int skip = st->debug_skip;
  st->debug_skip = -1;
  if (exact_here < n && nys::launch_step(ds, g0, n, q, k, v, out, s, skip) != cudaSuccess)
    return NYS_E_CUDA;
  if (exact_here) {
    if (nys::launch_exact_step(ds, g0, n, q, k, v, out, s) != cudaSuccess) return NYS_E_CUDA;
    for (int64_t g = g0; g < g0 + n; ++g)
      if (st->exact_len[(size_t)g] >= 0) ++st->exact_len[(size_t)g];
  }
  return NYS_OK;
}

int nys_query(const nys_states* st, int64_t g, nys_group_info* info, int32_t* far_len,
              void* stream) {
  if (!st || !info) return NYS_E_INVAL;
  if (g < 0 || g >= st->n_groups) return NYS_E_RANGE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* b = static_cast<const char*>(st->base);
  int32_t ints[nys::kIntsPerGroup];
  if (cudaMemcpyAsync(ints, b + st->lay.off_ints + (size_t)g * sizeof(ints), sizeof(ints),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return NYS_E_CUDA;
  if (far_len &&
      cudaMemcpyAsync(far_len, b + st->lay.off_far_len + (size_t)g * st->cfg.heads_per_kv * 4,
                      (size_t)st->cfg.heads_per_kv * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return NYS_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NYS_E_CUDA;
  info->win_head = ints[nys::kIntWinHead];
  info->win_len = ints[nys::kIntWinLen];
  info->m_eff = ints[nys::kIntMEff];
  info->t = ints[nys::kIntT];
  info->mode = ints[nys::kIntMode];
  info->status = ints[nys::kIntStatus];
  return NYS_OK;
}

int nys_layout_of(const nys_states* st, void** base, nys_layout* layout) {
  if (!st || !base || !layout) return NYS_E_INVAL;
  *base = st->base;
  *layout = st->lay;
  return NYS_OK;
}

int nys_mark_sealed(nys_states* st, int64_t g0, int64_t n) {
  if (!st) return NYS_E_INVAL;
  int rc = check_range(st, g0, n);
  if (rc) return rc;
  if (n) std::memset(st->sealed.data() + g0, 1, (size_t)n);
  forget_exact(st, g0, n);
  return NYS_OK;
}

int nys_debug_stall_once(nys_states* st, int32_t stage) {
  if (!st || stage < 0) return NYS_E_INVAL;
  st->debug_skip = stage;
  return NYS_OK;
}

int nys_debug_stall_replay_once(nys_states* st) {
  if (!st) return NYS_E_INVAL;
  st->debug_replay = 1;
  return NYS_OK;
}

int nys_config_of(const nys_states* st, nys_config* cfg, int64_t* n_groups) {
  if (!st || !cfg) return NYS_E_INVAL;
  *cfg = st->cfg;
  if (n_groups) *n_groups = st->n_groups;
  return NYS_OK;
}

}  // extern "C"
