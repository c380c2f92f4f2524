// Persistent, TMA-fed decode step (the fast path of nys_step_batch).
//
// Same arithmetic as nys_step.cu -- nystrom.rs (docs.rs source view,
// cortiq-engine 0.5.71), NystromState::advance, NystromHead::far_insert and
// NystromHead::step -- reorganised for GB300's memory system.  The step is a
// stream of ~300 KB per group with little arithmetic, so the kernel is built
// around keeping HBM busy:
//
//  * one CTA per SM loops over groups; warp 8 is a producer whose lane 0
//    streams every byte a group needs into a ring of 16 KB shared-memory
//    stages with cp.async.bulk (the TMA bulk-copy engine), signalling each
//    stage's arrival on an mbarrier with a transaction count;
//  * warps 0..7 consume the stages in order and hand each one back through a
//    second mbarrier, so the producer is always several stages -- and across
//    group boundaries, the next group -- ahead;
//  * per group the stages are: one "misc" stage (counters, queries, the new
//    and the evicted key/value, running maxima, Z^), the K side (sink keys,
//    window keys, key landmarks, each head's query landmarks, as one
//    sequence of d-float rows), M, the V side (sink and window values), and
//    T^ (hi and lo rows together).  Dot products of four rows x all heads are finished with one
//    multi-value butterfly (4*HT values across 32 lanes in 4*HT - 1 shuffles).
//
// Every wait is bounded.  A wait that runs out sets a status word in the
// group's ints slot kIntStatus and makes every warp leave; the producer then
// waits (bounded) for its copies still in flight before the CTA exits.
#include <cfloat>
#include <cmath>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kCWarps = 8;
constexpr int kCThreads = kCWarps * 32;
constexpr int kThreadsTma = kCThreads + 32;
constexpr int kMaxRing = 12;
constexpr int kRowsPerRound = 4;
constexpr int kQRows = 8;  // Q~ rows a warp reduces at once (generic path)
constexpr uint64_t kWaitNs = 2000000000ull;  // every wait gives up after 2 s
constexpr uint32_t kSuspendNs = 1000000;      // a waiting thread sleeps up to 1 ms per try
constexpr int kSmemBudget = 227 * 1024;    // one CTA per SM
constexpr int kSmemBudget2 = 113 * 1024;   // each of two CTAs per SM
constexpr int kMinRing = 3;

__host__ __device__ inline int r4(int x) { return (x + 3) & ~3; }

// Where everything lives; computed once on the host, passed by value.
struct TmaPlan {
  int rows_k, rows_m, rows_v, rows_t;  // rows per stage of each stream
  int tot_k;                           // w + m + H*m rows of d floats
  int n_k, n_m, n_v, n_t, per_group;   // stages per group of each stream
  // misc stage (bytes)
  int mo_ints, mo_q, mo_knew, mo_vnew, mo_kev, mo_vev, mo_mmax, mo_zhi, mo_zlo;
  int misc_bytes;
  // consumer scratch (floats, after the ring)
  int x_q, x_knew, x_vnew, x_kev, x_vev, x_mmax, x_zhi, x_zlo;
  int x_sig, x_fh, x_lg, x_rc, x_ms, x_den, x_fl, x_ints, x_part;
  int nrp, mp, scratch_floats;
  int ring;
  int debug_skip;   // test hook: ring stage CTA 0 withholds (-1: none)
  int stage_bytes;  // 32 KB when the ring still fits, else 16 KB
  int ctas_per_sm;
  int ring_off;  // bytes from the smem base to the ring
  size_t smem_bytes;
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t sptr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sptr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sptr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sptr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sptr(b)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(sptr(dst)),
      "l"(src), "r"(bytes), "r"(sptr(bar))
      : "memory");
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
// Three (two) independent butterfly reductions over the warp, interleaved so
// that they share one latency chain.
__device__ __forceinline__ void warp_max3(float& a, float& b, float& c) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, a, o);
    const float y = __shfl_xor_sync(0xffffffffu, b, o);
    const float z = __shfl_xor_sync(0xffffffffu, c, o);
    a = fmaxf(a, x);
    b = fmaxf(b, y);
    c = fmaxf(c, z);
  }
}
__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, a, o);
    const float y = __shfl_xor_sync(0xffffffffu, b, o);
    a += x;
    b += y;
  }
}

// Sum each of V per-lane partials over the 32 lanes.  Returns, in every lane,
// the total of value index reduce_index<V>(lane); lanes that share an index
// hold the same total.
template <int V>
__device__ __forceinline__ float reduce_multi(float (&x)[V], int lane) {
  constexpr int kSteps = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int half = V >> (st + 1);
    const int off = 16 >> st;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? x[i] : x[i + half];
      const float keep = upper ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = x[0];
#pragma unroll
  for (int off = 16 >> kSteps; off >= 1; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}
template <int V>
__device__ __forceinline__ int reduce_index(int lane) {
  constexpr int kSteps = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  int v = 0;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) v |= ((lane >> (4 - st)) & 1) << (kSteps - 1 - st);
  return v;
}
template <int V>
__device__ __forceinline__ bool reduce_writer(int lane) {
  constexpr int kSteps = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  return (lane & ((1 << (5 - kSteps)) - 1)) == 0;
}

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: false when 2 s passed or another warp gave up.
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, volatile int* abort) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test(b, parity)) return true;
    if ((i & 15u) == 0u) {
      if (abort && *abort) return false;
      if (gtime() - t0 > kWaitNs) return false;
    }
  }
}

// -------------------------------------------------------------- kernel
template <int HT, int KD>
__global__ void __launch_bounds__(kThreadsTma, 2)
step_tma_kernel(DevState s, TmaPlan P, int64_t g0, int64_t n, const float* __restrict__ q,
                const float* __restrict__ k, const float* __restrict__ v,
                float* __restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxRing;
  uint64_t* cbar = empty + kMaxRing;
  int* abort = reinterpret_cast<int*>(cbar + 1);
  unsigned char* ring = smem + P.ring_off;
  float* X = reinterpret_cast<float*>(ring + (size_t)P.ring * P.stage_bytes);

  const int d = s.d, dv = s.dv, w = s.w, ns = s.sink, H = s.heads, m = s.m;
  const int d4 = d >> 2, S = P.ring;

  for (int i = tid; i < P.scratch_floats; i += blockDim.x) X[i] = 0.f;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCWarps);
    }
    mbar_init(cbar, kCWarps);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Launched as a programmatic dependent of the previous kernel on the
  // stream (launch_tma_ht): everything above touches only this CTA's shared
  // memory, so it may overlap that kernel's tail; nothing global is read
  // before the previous kernel has completed and its writes are visible.
  // (Without that launch attribute this returns at once.)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ============================================================ producer
  if (warp == kCWarps) {
    if (lane != 0) return;
    uint32_t c = 0;        // stages issued so far
    int idx = 0;           // c % S
    uint32_t phase = 0;    // (c / S) & 1
    bool ok = true;
    int64_t gfail = n;     // first group left unstepped, when a wait gave up
    // The ring slot of the next group is read one group ahead so that the
    // load's latency overlaps the current group's copies.
    int3 nxt = make_int3(0, 0, 0);
    if (blockIdx.x < n) {
      const int32_t* ints0 = s.ints + (g0 + blockIdx.x) * kIntsPerGroup;
      nxt = make_int3(ints0[kIntWinHead], ints0[kIntWinLen], ints0[kIntMode]);
    }
    for (int64_t gi = blockIdx.x; gi < n && ok; gi += gridDim.x) {
      const int64_t g = g0 + gi;
      const int32_t* ints = s.ints + g * kIntsPerGroup;
      int slot = (nxt.y == w) ? nxt.x : nxt.y;
      slot = min(max(slot, 0), w - 1);
      // Exact-only groups (a separate kernel steps them) take only the misc
      // stage, from which the consumers learn to skip them.
      const int stages = (nxt.z == kModeExact) ? 1 : P.per_group;
      if (gi + gridDim.x < n) {
        const int32_t* in2 = s.ints + (g + gridDim.x) * kIntsPerGroup;
        nxt = make_int3(in2[kIntWinHead], in2[kIntWinLen], in2[kIntMode]);
      }
      for (int st = 0; st < stages && ok;
           ++st, ++c, idx = (idx + 1 == S) ? 0 : idx + 1, phase ^= (idx == 0) ? 1u : 0u) {
        if (!wait_bar(&empty[idx], phase ^ 1u, abort)) {
          ok = false;
          gfail = gi;
          break;
        }
        unsigned char* dst = ring + (size_t)idx * P.stage_bytes;
        uint64_t* bar = &full[idx];
        if ((int)c == P.debug_skip && blockIdx.x == 0) continue;  // test hook
        if (st == 0) {
          mbar_expect_tx(bar, (uint32_t)P.misc_bytes);
          bulk_load(dst + P.mo_ints, ints, kIntsPerGroup * 4, bar);
          bulk_load(dst + P.mo_q, q + gi * H * (int64_t)d, H * d * 4, bar);
          bulk_load(dst + P.mo_knew, k + gi * (int64_t)d, d * 4, bar);
          bulk_load(dst + P.mo_vnew, v + gi * (int64_t)dv, dv * 4, bar);
          bulk_load(dst + P.mo_kev, s.win_k + (g * w + slot) * (int64_t)d, d * 4, bar);
          bulk_load(dst + P.mo_vev, s.win_v + (g * w + slot) * (int64_t)dv, dv * 4, bar);
          bulk_load(dst + P.mo_mmax, s.m_max + g * H * (int64_t)m, H * m * 4, bar);
          bulk_load(dst + P.mo_zhi, s.z_hat + g * H * (int64_t)m, H * m * 4, bar);
          bulk_load(dst + P.mo_zlo, s.z_lo + g * H * (int64_t)m, H * m * 4, bar);
        } else if (st <= P.n_k) {
          // K side: rows [r0, r1) of sink keys | window keys | key landmarks |
          // Q~ (all heads), one row = d floats.
          const int r0 = (st - 1) * P.rows_k;
          const int r1 = min(r0 + P.rows_k, P.tot_k);
          mbar_expect_tx(bar, (uint32_t)((r1 - r0) * d * 4));
          const int seg[5] = {0, ns, ns + w, ns + w + m, P.tot_k};
          const float* base[4] = {s.sink_k + g * ns * (int64_t)d, s.win_k + g * w * (int64_t)d,
                                  s.k_tilde + g * m * (int64_t)d,
                                  s.q_tilde + g * H * m * (int64_t)d};
          for (int a = 0; a < 4; ++a) {
            const int lo = max(r0, seg[a]), hi = min(r1, seg[a + 1]);
            if (lo < hi)
              bulk_load(dst + (size_t)(lo - r0) * d * 4, base[a] + (int64_t)(lo - seg[a]) * d,
                        (uint32_t)((hi - lo) * d * 4), bar);
          }
        } else if (st <= P.n_k + P.n_m) {
          const int r0 = (st - 1 - P.n_k) * P.rows_m;
          const int r1 = min(r0 + P.rows_m, H * m);
          mbar_expect_tx(bar, (uint32_t)((r1 - r0) * m * 4));
          bulk_load(dst, s.mu + (g * H * m + r0) * (int64_t)m, (uint32_t)((r1 - r0) * m * 4), bar);
        } else if (st <= P.n_k + P.n_m + P.n_v) {
          // V side: rows [r0, r1) of sink values | window values.
          const int r0 = (st - 1 - P.n_k - P.n_m) * P.rows_v;
          const int r1 = min(r0 + P.rows_v, ns + w);
          mbar_expect_tx(bar, (uint32_t)((r1 - r0) * dv * 4));
          const int seg[3] = {0, ns, ns + w};
          const float* base[2] = {s.sink_v + g * ns * (int64_t)dv, s.win_v + g * w * (int64_t)dv};
          for (int a = 0; a < 2; ++a) {
            const int lo = max(r0, seg[a]), hi = min(r1, seg[a + 1]);
            if (lo < hi)
              bulk_load(dst + (size_t)(lo - r0) * dv * 4, base[a] + (int64_t)(lo - seg[a]) * dv,
                        (uint32_t)((hi - lo) * dv * 4), bar);
          }
        } else {
          const int r0 = (st - 1 - P.n_k - P.n_m - P.n_v) * P.rows_t;
          const int r1 = min(r0 + P.rows_t, H * m);
          const uint32_t hb = (uint32_t)((r1 - r0) * dv * 4), lb = (uint32_t)((r1 - r0) * dv * 2);
          mbar_expect_tx(bar, hb + lb);
          bulk_load(dst, s.t_hat + (g * H * m + r0) * (int64_t)dv, hb, bar);
          bulk_load(dst + (size_t)P.rows_t * dv * 4, s.t_lo + (g * H * m + r0) * (int64_t)dv, lb,
                    bar);
        }
      }
    }
    if (!ok) {
      atomicExch(abort, 1);
      for (int64_t g2 = g0 + gfail; g2 < g0 + n; g2 += gridDim.x)
        s.ints[g2 * kIntsPerGroup + kIntStatus] = 1;
    }
    // Whatever happened, no copy may still be landing in shared memory when
    // the CTA exits: wait (bounded) for the last S stages issued.
    const uint32_t first = c > (uint32_t)S ? c - (uint32_t)S : 0u;
    for (uint32_t cc = first; cc < c; ++cc)
      if (!((int)cc == P.debug_skip && blockIdx.x == 0))
        wait_bar(&full[cc % S], (cc / S) & 1u, nullptr);
    return;  // (the division above runs once, at exit)
  }

  // ============================================================ consumers
  float* xq = X + P.x_q;
  float* pT = xq;  // near weights [sink + window row][HT], written by the per-head phase
  // The new key and value alternate between two buffers from group to
  // group: the ring-slot write at the end of a group reads them while a
  // faster warp may already copy the next group's in, so no barrier is
  // needed between the two.
  float* const xknew2 = X + P.x_knew;
  float* const xvnew2 = X + P.x_vnew;
  int nbuf = 0;
  float* xkev = X + P.x_kev;
  float* xvev = X + P.x_vev;
  float* xmmax = X + P.x_mmax;
  float* xzhi = X + P.x_zhi;
  float* xzlo = X + P.x_zlo;
  float* sig = X + P.x_sig;
  float* fh = X + P.x_fh;
  float* lg = X + P.x_lg;
  // Per (head, landmark): {rescale r, weight e of the evicted key, gain g,
  // updated Z^ (hi + lo)}, one 16-byte load per T^ row.
  float4* rc = reinterpret_cast<float4*>(X + P.x_rc);
  float* ms = X + P.x_ms;
  float* den = X + P.x_den;
  int* xints = reinterpret_cast<int*>(X + P.x_ints);
  float* part = X + P.x_part;
  const float scale = s.scale;
  // Ring cursor of the next stage to consume: slot index and phase parity,
  // advanced incrementally (no division by the ring length).
  int ci = 0;
  uint32_t cpar = 0;
  uint32_t cphase = 0;   // consumer barrier phase
  volatile int* vabort = abort;
  auto advance = [&]() {
    if (++ci == S) {
      ci = 0;
      cpar ^= 1u;
    }
  };
  auto stage_ptr = [&](int i) { return ring + (size_t)i * P.stage_bytes; };
  auto release_slot = [&](int i) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[i]);
  };
  auto acquire_slot = [&](int i, uint32_t par) -> bool {
    return wait_bar(&full[i], par, vabort);
  };
  auto csync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar);
    const bool r = wait_bar(cbar, cphase, vabort);
    cphase ^= 1u;
    return r;
  };
  auto fail = [&](int64_t g) {
    atomicExch(abort, 1);
    // this group and every later one of this CTA are left unstepped
    if (lane == 0)
      for (int64_t g2 = g; g2 < g0 + n; g2 += gridDim.x)
        s.ints[g2 * kIntsPerGroup + kIntStatus] = 1;
  };

  for (int64_t gi = blockIdx.x; gi < n; gi += gridDim.x, nbuf ^= 1) {
    const int64_t g = g0 + gi;
    // This CTA's last group: the next kernel on the stream may be scheduled
    // once every CTA has got here (it still waits for this grid to finish
    // before it reads anything).
    if (gi + gridDim.x >= n && tid == 0) asm volatile("griddepcontrol.launch_dependents;");
    float* const xknew = xknew2 + nbuf * d;
    float* const xvnew = xvnew2 + nbuf * dv;
    // far_len of the head this warp owns in the per-head phase; loaded now so
    // that its latency hides behind the K side.
    const int fl_old = (warp < H && lane == 0) ? s.far_len[g * H + warp] : 0;
    // ---- misc stage: copy to scratch, hand the stage back at once.
    if (!acquire_slot(ci, cpar)) { fail(g); return; }
    {
      const unsigned char* st = stage_ptr(ci);
      auto cp = [&](float* dst, int off, int nfl) {
        const float* src = reinterpret_cast<const float*>(st + off);
        for (int i = tid; i < (nfl >> 2); i += kCThreads) st4(dst + 4 * i, ld4(src + 4 * i));
      };
      cp(xq, P.mo_q, H * d);
      cp(xknew, P.mo_knew, d);
      cp(xvnew, P.mo_vnew, dv);
      cp(xkev, P.mo_kev, d);
      cp(xvev, P.mo_vev, dv);
      cp(xmmax, P.mo_mmax, H * m);
      cp(xzhi, P.mo_zhi, H * m);
      cp(xzlo, P.mo_zlo, H * m);
      if (tid < kIntsPerGroup) xints[tid] = reinterpret_cast<const int*>(st + P.mo_ints)[tid];
    }
    release_slot(ci);
    advance();
    if (!csync()) { fail(g); return; }
    if (xints[kIntMode] == kModeExact) {
      // every thread has read the mode before the next group's misc copy
      if (!csync()) { fail(g); return; }
      continue;
    }
    const int win_head = xints[kIntWinHead];
    const int win_len = xints[kIntWinLen];
    const int m_eff = min(max(xints[kIntMEff], 0), m);
    const bool full = (win_len == w);
    const int slot = full ? win_head : win_len;
    const int nwin = full ? w : win_len + 1;
    const int nnear = ns + nwin;
    const bool ck = lane < d4;  // this lane's float4 column of a d-row
    float4 qr[HT];
#pragma unroll
    for (int hh = 0; hh < HT; ++hh)
      qr[hh] = ck ? ld4(xq + hh * d + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 kev4 = ck ? ld4(xkev + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    // d = 128 path: this lane's four float4 columns (kgl, kgl+8, kgl+16, kgl+24)
    // of every head's query and of the evicted key.
    const int kgrp = lane >> 3, kgl = lane & 7;
    float4 qk[KD == 128 ? HT : 1][4];
    float4 kvr[4];
    if constexpr (KD == 128) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kvr[i] = ld4(xkev + 4 * (kgl + 8 * i));
#pragma unroll
        for (int hh = 0; hh < HT; ++hh) qk[hh][i] = ld4(xq + hh * 128 + 4 * (kgl + 8 * i));
      }
    }

    // ---- A: the K-side stages (sinks, window, key landmarks, Q~).
    for (int st = 0; st < P.n_k; ++st, advance()) {
      if (!acquire_slot(ci, cpar)) { fail(g); return; }
      const float* stage = reinterpret_cast<const float*>(stage_ptr(ci));
      const int r0 = st * P.rows_k;
      const int nrow = min(P.rows_k, P.tot_k - r0);
      if constexpr (KD == 128) {
        // d = 128: a row is 32 float4; 8 lanes share a row (4 float4 each,
        // query chunks in registers), a warp takes 4 rows at once.
        for (int base = 0; base < nrow; base += kCWarps * 4) {
          const int lr = base + warp * 4 + kgrp;
          float x[HT];
#pragma unroll
          for (int hh = 0; hh < HT; ++hh) x[hh] = 0.f;
          const bool valid = lr < nrow;
          const int vr = r0 + lr;
          if (valid) {
            const float* row = stage + lr * 128;
            if (vr - ns == slot && vr >= ns) row = xknew;
            const float4 a0 = ld4(row + 4 * kgl), a1 = ld4(row + 4 * (kgl + 8));
            const float4 a2 = ld4(row + 4 * (kgl + 16)), a3 = ld4(row + 4 * (kgl + 24));
            if (vr < ns + w + m) {
#pragma unroll
              for (int hh = 0; hh < HT; ++hh)
                x[hh] = (dot4(a0, qk[hh][0]) + dot4(a1, qk[hh][1])) +
                        (dot4(a2, qk[hh][2]) + dot4(a3, qk[hh][3]));
            } else {
              x[0] = (dot4(a0, kvr[0]) + dot4(a1, kvr[1])) + (dot4(a2, kvr[2]) + dot4(a3, kvr[3]));
            }
          }
#pragma unroll
          for (int hh = 0; hh < HT; ++hh) {
            x[hh] += __shfl_xor_sync(0xffffffffu, x[hh], 1);
            x[hh] += __shfl_xor_sync(0xffffffffu, x[hh], 2);
            x[hh] += __shfl_xor_sync(0xffffffffu, x[hh], 4);
          }
          if (valid && kgl == 0) {
            if (vr < ns + w) {
#pragma unroll
              for (int hh = 0; hh < HT; ++hh)
                if (hh < H) sig[hh * P.nrp + vr] = x[hh] * scale;
            } else if (vr < ns + w + m) {
#pragma unroll
              for (int hh = 0; hh < HT; ++hh)
                if (hh < H) fh[hh * P.mp + (vr - ns - w)] = x[hh] * scale;
            } else {
              int qr = vr - ns - w - m;
              int h = 0;
              while (qr >= m) {
                qr -= m;
                ++h;
              }
              lg[h * P.mp + qr] = x[0] * scale;
            }
          }
        }
      } else {
      // Rows before kend are keys (dotted with every head's query); the rest
      // are Q~ rows, each dotted with the evicted key only.
      const int kend = min(nrow, max(0, ns + w + m - r0));
      // Eight heads: two rows per round (16 partial sums) keep the loop within
      // the 96 registers of two CTAs per SM; four rows spilled.
      constexpr int kRR = HT > 4 ? 2 : kRowsPerRound;
      for (int base = 0; base < kend; base += kCWarps * kRR) {
        float x[kRR * HT];
#pragma unroll
        for (int i = 0; i < kRR * HT; ++i) x[i] = 0.f;
#pragma unroll
        for (int u = 0; u < kRR; ++u) {
          const int lr = base + warp * kRR + u;
          if (lr < kend && ck) {
            const int vr = r0 + lr;
            const float* row = (vr - ns == slot && vr >= ns) ? xknew : stage + lr * d;
            const float4 a = ld4(row + 4 * lane);
#pragma unroll
            for (int hh = 0; hh < HT; ++hh) x[u * HT + hh] = dot4(a, qr[hh]);
          }
        }
        const float tot = reduce_multi<kRR * HT>(x, lane);
        if (reduce_writer<kRR * HT>(lane)) {
          const int vi = reduce_index<kRR * HT>(lane);
          const int u = vi / HT, hh = vi - u * HT;
          const int lr = base + warp * kRR + u;
          if (lr < kend && hh < H) {
            const int vr = r0 + lr;
            const float l = tot * scale;
            if (vr < ns + w) sig[hh * P.nrp + vr] = l;
            else fh[hh * P.mp + (vr - ns - w)] = l;
          }
        }
      }
      // Q~ rows, kQRows per warp: one value per row, reduced all at once.
      for (int base = kend + warp * kQRows; base < nrow; base += kCWarps * kQRows) {
        float x[kQRows];
#pragma unroll
        for (int u = 0; u < kQRows; ++u) {
          const int lr = base + u;
          x[u] = (lr < nrow && ck) ? dot4(ld4(stage + (lr * d + 4 * lane)), kev4) : 0.f;
        }
        const float tot = reduce_multi<kQRows>(x, lane);
        if (reduce_writer<kQRows>(lane)) {
          const int lr = base + reduce_index<kQRows>(lane);
          if (lr < nrow) {
            int qr = r0 + lr - (ns + w + m);
            int h = 0;
            while (qr >= m) {  // at most H - 1 steps
              qr -= m;
              ++h;
            }
            lg[h * P.mp + qr] = tot * scale;
          }
        }
      }
      }
      release_slot(ci);
    }
    if (!csync()) { fail(g); return; }

    // ---- B: per-head scalars, one warp per head (H <= kCWarps, so a warp
    // has at most one).  Steps (1)-(3) need no M and run first, while M is
    // still on its way; then M streams through the ring a stage at a time
    // (each stage holds the blocks of heads_per_stage consecutive heads), a
    // head's warp takes step (4) as soon as its block has landed, and every
    // stage is handed back right after, so the ring never holds all of M.
    const int hh = warp;
    float c_all = 0.f, f = 0.f, psum = 0.f;
    bool has_far = false;
    if (hh < H) {
      const int64_t hb = g * H + hh;
      float* hfh = fh + hh * P.mp;
      float4* hrc = rc + hh * P.mp;
      float* hms = ms + hh * P.mp;
      float* hsig = sig + hh * P.nrp;
      // (1) Landmark updates: delayed insertion of the evicted key with the
      //     running-maximum rescale.  mx_m collects the maximum of the new
      //     running maxima.
      float mx_m = -INFINITY;
      for (int i = lane; i < m_eff; i += 32) {
        const float mo = xmmax[hh * m + i], zo = xzhi[hh * m + i], zlo = xzlo[hh * m + i];
        float r = 1.f, e = 0.f, mn = mo, zn = zo, zln = zlo;
        if (full) {
          const float l = lg[hh * P.mp + i];
          if (l > mo) {
            r = expf(mo - l);
            mn = l;
          }
          e = expf(l - mn);
          comp_axpy(zo, zlo, r, e, 1.f, zn, zln);
          s.m_max[hb * m + i] = mn;
          s.z_hat[hb * m + i] = zn;
          s.z_lo[hb * m + i] = zln;
        }
        // Z^ stays a pair for the far denominator (step (4)): hi in the
        // rescale record, lo in place of the old lo (no one reads it again).
        hrc[i] = make_float4(r, e, 0.f, zn);
        xzlo[hh * m + i] = zln;
        hms[i] = mn;
        mx_m = fmaxf(mx_m, mn);
      }
      const int fl_new = __shfl_sync(0xffffffffu, fl_old, 0) + (full ? 1 : 0);
      if (full && lane == 0) s.far_len[hb] = fl_new;
      has_far = fl_new > 0;
      // (2) The maxima: near logits, landmark logits f, and the running
      //     maxima, reduced together.  max_b (f + m_b) = f + max_b m_b
      //     exactly, since rounding is monotonic.
      float cmax = -INFINITY;
      f = -INFINITY;
      for (int j = lane; j < nnear; j += 32) cmax = fmaxf(cmax, hsig[j]);
      if (has_far)
        for (int a = lane; a < m_eff; a += 32) f = fmaxf(f, hfh[a]);
      warp_max3(cmax, f, mx_m);
      c_all = has_far ? fmaxf(cmax, f + mx_m) : cmax;
      if (has_far)
        for (int a = lane; a < m_eff; a += 32) hfh[a] = expf(hfh[a] - f);
      // (3) Near weights on the joint scale (positive terms: f32 suffices).
      for (int j = lane; j < nnear; j += 32) {
        const float p = expf(hsig[j] - c_all);
        pT[j * HT + hh] = p;
        psum += p;
      }
    }
    const int heads_per_stage = P.rows_m / m;
    for (int mst = 0; mst < P.n_m; ++mst, advance()) {
      if (!acquire_slot(ci, cpar)) { fail(g); return; }
      const int h_lo = mst * heads_per_stage;
      const int h_hi = min(H, h_lo + heads_per_stage);
      if (hh < H && hh >= h_lo && hh < h_hi) {
        float4* hrc = rc + hh * P.mp;
        float* hfh = fh + hh * P.mp;
        float* hms = ms + hh * P.mp;
        // (4) Far mix u = F^ M (rectified), weights g_b on the joint scale,
        //     far denominator.  The far denominator sum_b g_b Z^_b cancels:
        //     where u has mixed signs its terms can be thousands of times
        //     the result, so it is carried in double-float: u as its Dot2
        //     pair, g_b with its exponent f + m_b - c_all unrounded, Z^ as
        //     the stored pair, the sum compensated across the warp.  The far
        //     numerator takes g_b rounded to f32.
        float dh = 0.f, dl = 0.f;
        if (has_far) {
          __syncwarp();
          // This head's m x m block of M, inside the current M stage.
          const float* Mh = reinterpret_cast<const float*>(stage_ptr(ci)) +
                            (size_t)(hh - h_lo) * m * m;
          for (int b = lane; b < m_eff; b += 32) {
            float uh, ul, eh, el, gh, gl, th, tl;
            dot2_x4_pair(hfh, Mh + b, m, m_eff, uh, ul);
            if (s.rect == NYS_RECT_FM && uh < 0.f) uh = ul = 0.f;
            exp_sum_pair(f, hms[b], c_all, eh, el);
            df_mul(uh, ul, eh, el, gh, gl);
            hrc[b].z = gh;
            df_mul(gh, gl, hrc[b].w, xzlo[hh * m + b], th, tl);
            df_add(dh, dl, th, tl, dh, dl);
          }
        } else {
          for (int b = lane; b < m_eff; b += 32) hrc[b].z = 0.f;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, dh, o);
          const float ol = __shfl_xor_sync(0xffffffffu, dl, o);
          psum += __shfl_xor_sync(0xffffffffu, psum, o);
          df_add(dh, dl, oh, ol, dh, dl);
        }
        float far_den = has_far ? dh + dl : 0.f;
        // Guard: a negative (or NaN) far denominator drops the far field.
        if (has_far && !(far_den >= 0.f)) {
          far_den = 0.f;
          for (int b = lane; b < m_eff; b += 32) hrc[b].z = 0.f;
        }
        if (lane == 0) den[hh] = fmaxf(far_den + psum, 1e-30f);
      }
      release_slot(ci);
    }
    if (!csync()) { fail(g); return; }

    // ---- C: values and the far numerators.  With one or two heads the V
    // and T^ row loops are unrolled (more loads in flight per warp); with
    // more heads the registers are better spent on the head accumulators.
    const bool cv = lane < (dv >> 2);
    float4 acc[HT];
#pragma unroll
    for (int hh = 0; hh < HT; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int st = 0; st < P.n_v; ++st, advance()) {
      if (!acquire_slot(ci, cpar)) { fail(g); return; }
      const float* stage = reinterpret_cast<const float*>(stage_ptr(ci));
      const int r0 = st * P.rows_v;
      const int nrow = min(P.rows_v, ns + w - r0);
#pragma unroll (HT <= 2 ? 4 : 2)
      for (int lr = warp; lr < nrow; lr += kCWarps) {
        const int j = r0 + lr;  // near row: sinks first, then window slots
        if (j < nnear && cv) {
          const float* row = (j - ns == slot) ? xvnew : stage + lr * dv;
          const float4 a = ld4(row + 4 * lane);
          // This row's weight for every head (slots past H hold stale values
          // and feed accumulators that are never written out).
          float pw[HT];
          if constexpr (HT % 4 == 0) {
#pragma unroll
            for (int q4 = 0; q4 < HT / 4; ++q4) {
              const float4 t = ld4(pT + j * HT + 4 * q4);
              pw[4 * q4] = t.x;
              pw[4 * q4 + 1] = t.y;
              pw[4 * q4 + 2] = t.z;
              pw[4 * q4 + 3] = t.w;
            }
          } else if constexpr (HT == 2) {
            const float2 t = *reinterpret_cast<const float2*>(pT + j * 2);
            pw[0] = t.x;
            pw[1] = t.y;
          } else {
            pw[0] = pT[j];
          }
#pragma unroll
          for (int hh = 0; hh < HT; ++hh) {
            const float p = pw[hh];
            acc[hh].x = fmaf(p, a.x, acc[hh].x);
            acc[hh].y = fmaf(p, a.y, acc[hh].y);
            acc[hh].z = fmaf(p, a.z, acc[hh].z);
            acc[hh].w = fmaf(p, a.w, acc[hh].w);
          }
        }
      }
      release_slot(ci);
    }
    const float4 ve = cv ? ld4(xvev + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    // (head, landmark) of T^ rows, stepped without dividing by m: (sh, sb) is
    // the current stage's first row, (th, tb) this warp's next row.
    int sh = 0, sb = 0;
    // Many heads: a warp's rows come head by head, so their far numerator
    // collects in one accumulator that is added to its head's once the head
    // changes (with one or two heads a predicated add per row is cheaper).
    float4 tacc = make_float4(0.f, 0.f, 0.f, 0.f);
    int hcur = 0;
    auto flush_far = [&]() {
#pragma unroll
      for (int hh = 0; hh < HT; ++hh) {
        if (hh == hcur) {
          acc[hh].x += tacc.x;
          acc[hh].y += tacc.y;
          acc[hh].z += tacc.z;
          acc[hh].w += tacc.w;
        }
      }
      tacc = make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float* const t_hi_g = s.t_hat + (g * H * (int64_t)m) * dv + 4 * lane;
    uint16_t* const t_lo_g = s.t_lo + (g * H * (int64_t)m) * dv + 4 * lane;
    for (int st = 0; st < P.n_t; ++st, advance()) {
      if (!acquire_slot(ci, cpar)) { fail(g); return; }
      const unsigned char* stage = stage_ptr(ci);
      int th = sh, tb = sb + warp;
      while (tb >= m) {
        tb -= m;
        ++th;
      }
      sb += P.rows_t;
      while (sb >= m) {
        sb -= m;
        ++sh;
      }
      const float* hi_rows = reinterpret_cast<const float*>(stage);
      const uint16_t* lo_rows =
          reinterpret_cast<const uint16_t*>(stage + (size_t)P.rows_t * dv * 4);
      const int r0 = st * P.rows_t;
      const int nrow = min(P.rows_t, H * m - r0);
#pragma unroll (HT <= 2 ? 2 : 1)
      for (int lr = warp; lr < nrow; lr += kCWarps) {
        const int h = th, b = tb;
        tb += kCWarps;
        while (tb >= m) {
          tb -= m;
          ++th;
        }
        if constexpr (HT > 2) {
          if (h != hcur) {  // warp-uniform
            flush_far();
            hcur = h;
          }
        }
        if (b < m_eff && cv) {
          float4 x = ld4(hi_rows + (lr * dv + 4 * lane));
          const uint2 lr2 = *reinterpret_cast<const uint2*>(lo_rows + (lr * dv + 4 * lane));
          float4 lo = make_float4(bf16_lo(lr2.x), bf16_hi(lr2.x), bf16_lo(lr2.y), bf16_hi(lr2.y));
          const float4 cf = rc[h * P.mp + b];  // {r, e, g, Z^}
          if (full) {
            // Compensated far update (Kahan form), written back in place:
            // the group's T^ rows are h * m + b = r0 + lr.
            kahan_axpy4(x, lo, cf.x, cf.y, ve);
            const int ro = (r0 + lr) * dv;  // < H m dv <= 2^16
            st4(t_hi_g + ro, x);
            uint2 lw;
            lw.x = pack_bf16x2(lo.x, lo.y);
            lw.y = pack_bf16x2(lo.z, lo.w);
            *reinterpret_cast<uint2*>(t_lo_g + ro) = lw;
          }
          // The far numerator enters the output through its high part: the
          // low part is under half an ulp of it, as small as the contraction's
          // own rounding; it matters only for the state it carries forward.
          if constexpr (HT > 2) {
            tacc.x = fmaf(cf.z, x.x, tacc.x);
            tacc.y = fmaf(cf.z, x.y, tacc.y);
            tacc.z = fmaf(cf.z, x.z, tacc.z);
            tacc.w = fmaf(cf.z, x.w, tacc.w);
          } else {
#pragma unroll
            for (int hh = 0; hh < HT; ++hh) {
              if (hh == h) {
                acc[hh].x = fmaf(cf.z, x.x, acc[hh].x);
                acc[hh].y = fmaf(cf.z, x.y, acc[hh].y);
                acc[hh].z = fmaf(cf.z, x.z, acc[hh].z);
                acc[hh].w = fmaf(cf.z, x.w, acc[hh].w);
              }
            }
          }
        }
      }
      release_slot(ci);
    }
    if constexpr (HT > 2) flush_far();
    // Cross-warp sum of the output numerators.  With up to two heads every
    // warp's partials fit the buffer: one barrier, then each output sums
    // kCWarps partials.  With more heads, two rounds through kCWarps/2 slots.
    constexpr int kSlots = HT <= 2 ? kCWarps : kCWarps / 2;
    if constexpr (HT <= 2) {
      if (cv) {
#pragma unroll
        for (int hh = 0; hh < HT; ++hh) st4(part + (warp * HT + hh) * 128 + 4 * lane, acc[hh]);
      }
      if (!csync()) { fail(g); return; }
    } else {
      if (warp >= kSlots && cv) {
#pragma unroll
        for (int hh = 0; hh < HT; ++hh)
          st4(part + ((warp - kSlots) * HT + hh) * 128 + 4 * lane, acc[hh]);
      }
      if (!csync()) { fail(g); return; }
      if (warp < kSlots && cv) {
#pragma unroll
        for (int hh = 0; hh < HT; ++hh) {
          float* p = part + (warp * HT + hh) * 128 + 4 * lane;
          const float4 o = ld4(p);
          st4(p, make_float4(o.x + acc[hh].x, o.y + acc[hh].y, o.z + acc[hh].z, o.w + acc[hh].w));
        }
      }
      if (!csync()) { fail(g); return; }
    }
    for (int idx = tid; idx < H * dv; idx += kCThreads) {
      const int hh = idx / dv, col = idx - hh * dv;
      float sum = 0.f;
#pragma unroll
      for (int wp = 0; wp < kSlots; ++wp) sum += part[(wp * HT + hh) * 128 + col];
      out[(gi * H + hh) * (int64_t)dv + col] = sum / den[hh];
    }
    // The ring slot takes the new key/value; the counters move on.
    for (int i = tid; i < d4; i += kCThreads)
      st4(s.win_k + (g * w + slot) * (int64_t)d + 4 * i, ld4(xknew + 4 * i));
    for (int i = tid; i < (dv >> 2); i += kCThreads)
      st4(s.win_v + (g * w + slot) * (int64_t)dv + 4 * i, ld4(xvnew + 4 * i));
    if (tid == 0) {
      int32_t* ints = s.ints + g * kIntsPerGroup;
      if (full) ints[kIntWinHead] = (win_head + 1) % w;
      else ints[kIntWinLen] = win_len + 1;
    }
    // No barrier here: the next group's misc copy writes the other new
    // key/value buffer, and every other scratch value read above (the
    // partials, den) is next written after that group's first barriers.
  }
}

template <int HT>
cudaError_t launch_tma_ht(const DevState& s, const TmaPlan& P, int64_t g0, int64_t n,
                          const float* q, const float* k, const float* v, float* out,
                          cudaStream_t stream) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      sms = 1;
  }
  // With a few groups per CTA, the last group is a large share of the
  // launch: size the grid so that every CTA takes the same count (512 groups
  // on 304 slots: 256 CTAs of two rather than 208 of two and 96 of one;
  // measured 0.911 -> 0.878 ms per 28 per-layer launches).  With many, keep
  // every slot busy: fewer CTAs mean fewer copies in flight (14,336 groups on
  // 299 CTAs of 48 measured 1.5% slower than on 304).
  const int64_t slots = (int64_t)sms * P.ctas_per_sm;
  const int64_t per = (n + slots - 1) / slots;  // groups per CTA
  const int64_t grid = per <= 4 ? (n + per - 1) / per : slots;
  // Programmatic dependent launch: this grid's CTAs may be scheduled while
  // the previous kernel on the stream drains (their prologue then overlaps
  // its tail); the kernel waits for that kernel's completion before its
  // first global read (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsTma);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (HT <= 2) {
    if (s.d == 128) {
      cudaError_t e = ensure_smem<step_tma_kernel<HT, 128>>(P.smem_bytes);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, step_tma_kernel<HT, 128>, s, P, g0, n, q, k, v, out);
    }
  }
  cudaError_t e = ensure_smem<step_tma_kernel<HT, 0>>(P.smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, step_tma_kernel<HT, 0>, s, P, g0, n, q, k, v, out);
}

}  // namespace

// Plan the stage layout; false when the geometry is outside this kernel
// (every bulk copy must start and end on 16 bytes, dv <= 128, H <= 8, and the
// misc stage and the scratch must fit).
// Plan one stage size and CTA count; false if it does not fit.
static bool plan_with(const DevState& s, int stage_bytes, int per_sm, TmaPlan& P) {
  const int d = s.d, dv = s.dv, m = s.m, H = s.heads, w = s.w, ns = s.sink;
  const int ht = H <= 1 ? 1 : H <= 2 ? 2 : H <= 4 ? 4 : 8;
  P.stage_bytes = stage_bytes;
  P.rows_k = stage_bytes / (d * 4);
  P.rows_m = stage_bytes / (m * 4);
  if (P.rows_m % m) return false;  // a head's M block must not straddle stages
  P.rows_v = stage_bytes / (dv * 4);
  P.rows_t = stage_bytes / (dv * 6);
  P.rows_t &= ~1;  // keeps the bf16 block 16-byte aligned for any dv % 8 == 0
  // A whole number of rows per consumer warp in every full stage (measured:
  // batch64 0.6449 -> 0.6415 ms, the eight-head decode 0.1346 -> 0.1339).
  if (P.rows_t >= kCWarps) P.rows_t -= P.rows_t % kCWarps;
  if (P.rows_k < 1 || P.rows_m < 1 || P.rows_v < 1 || P.rows_t < 1) return false;
  P.tot_k = ns + w + m + H * m;
  P.n_k = (P.tot_k + P.rows_k - 1) / P.rows_k;
  P.n_m = (H * m + P.rows_m - 1) / P.rows_m;
  P.n_v = (ns + w + P.rows_v - 1) / P.rows_v;
  P.n_t = (H * m + P.rows_t - 1) / P.rows_t;
  P.per_group = 1 + P.n_k + P.n_m + P.n_v + P.n_t;
  int o = 0;
  P.mo_ints = o; o += kIntsPerGroup * 4;
  P.mo_q = o;    o += H * d * 4;
  P.mo_knew = o; o += d * 4;
  P.mo_vnew = o; o += dv * 4;
  P.mo_kev = o;  o += d * 4;
  P.mo_vev = o;  o += dv * 4;
  P.mo_mmax = o; o += H * m * 4;
  P.mo_zhi = o;  o += H * m * 4;
  P.mo_zlo = o;  o += H * m * 4;
  P.misc_bytes = o;
  if (o > stage_bytes) return false;
  P.nrp = r4(ns + w);
  P.mp = r4(m);
  int x = 0;
  // The queries are read once, into registers, at the start of the K side;
  // afterwards the region holds the near weights transposed, [row][head].
  P.x_q = x;    x += (ht * d > P.nrp * ht) ? ht * d : P.nrp * ht;
  P.x_knew = x; x += 2 * d;   // two buffers, used by alternate groups
  P.x_vnew = x; x += 2 * dv;
  P.x_kev = x;  x += d;
  P.x_vev = x;  x += dv;
  P.x_mmax = x; x += H * m;
  P.x_zhi = x;  x += H * m;
  P.x_zlo = x;  x += H * m;
  P.x_sig = x;  x += ht * P.nrp;
  P.x_fh = x;   x += ht * P.mp;
  P.x_lg = x;   x += ht * P.mp;
  P.x_rc = x;   x += 4 * ht * P.mp;  // float4 per (head, landmark); x stays a multiple of 4
  P.x_ms = x;   x += ht * P.mp;
  P.x_den = x;  x += r4(ht);
  P.x_fl = x;   x += r4(ht);
  P.x_ints = x; x += kIntsPerGroup;
  P.x_part = x; x += (ht <= 2 ? kCWarps : kCWarps / 2) * ht * 128;
  P.scratch_floats = x;
  P.ring_off = 1024;  // barriers and the abort flag live below
  const long budget = per_sm == 2 ? kSmemBudget2 : kSmemBudget;
  const long avail = budget - P.ring_off - (long)x * 4;
  int ring = (int)(avail / stage_bytes);
  if (ring > kMaxRing) ring = kMaxRing;
  if (ring < kMinRing) return false;
  P.ring = ring;
  P.debug_skip = -1;
  P.ctas_per_sm = per_sm;
  P.smem_bytes = (size_t)P.ring_off + (size_t)ring * stage_bytes + (size_t)x * 4;
  return true;
}

// Plan the stage layout; false when the geometry is outside this kernel
// (every bulk copy must start and end on 16 bytes, d and dv <= 128, H <= 8,
// and the misc stage and the scratch must fit).  Preference, measured on the
// 14336-group workload: two CTAs per SM (two groups in flight per SM) matter
// most, then large stages (fewer hand-offs per group): 32 KB stages 0.707 ms,
// 16 KB 0.774 ms; one CTA per SM 1.1-1.2 ms.
bool plan_step_tma(const DevState& s, void* plan_out) {
  TmaPlan& P = *static_cast<TmaPlan*>(plan_out);
  const int d = s.d, dv = s.dv, m = s.m, H = s.heads;
  if (H > 8 || d > 128 || dv > 128 || (dv & 7) || (d & 3) || ((H * m) & 3) || (m & 3))
    return false;
  const int tries[4][2] = {{32768, 2}, {16384, 2}, {32768, 1}, {16384, 1}};
  for (const auto& t : tries)
    if (plan_with(s, t[0], t[1], P)) return true;
  return false;
}

size_t step_tma_plan_bytes() { return sizeof(TmaPlan); }

cudaError_t launch_step_tma(const DevState& s, const void* plan, int64_t g0, int64_t n,
                            const float* q, const float* k, const float* v, float* out,
                            cudaStream_t stream, int debug_skip) {
  TmaPlan P = *static_cast<const TmaPlan*>(plan);
  P.debug_skip = debug_skip;
  if (n <= 0) return cudaSuccess;
  if (s.heads == 1) return launch_tma_ht<1>(s, P, g0, n, q, k, v, out, stream);
  if (s.heads == 2) return launch_tma_ht<2>(s, P, g0, n, q, k, v, out, stream);
  if (s.heads <= 4) return launch_tma_ht<4>(s, P, g0, n, q, k, v, out, stream);
  return launch_tma_ht<8>(s, P, g0, n, q, k, v, out, stream);
}

}  // namespace nys
