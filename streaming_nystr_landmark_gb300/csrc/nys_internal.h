// Internal declarations shared by the libnys translation units: the device
// view of a state buffer and the kernel launchers.  Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "nys.h"

namespace nys {

// Raise a kernel's dynamic shared-memory limit only when a launch needs more
// than any earlier one (one driver call per kernel and size, none during
// later launches -- e.g. inside CUDA graph capture after a warm-up launch).
template <auto Kernel>
inline cudaError_t ensure_smem(size_t bytes) {
  static size_t set_bytes = 48 * 1024;  // one record per kernel
  if (bytes <= set_bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) set_bytes = bytes;
  return e;
}

// Limits the kernels are written for (the ABI reports NYS_E_UNSUPPORTED
// beyond them).  They bound the on-chip buffers: the seal keeps A, A^T A and
// its Cholesky factor (3 m^2 doubles) in shared memory, and the step keeps a
// tile of heads' near logits (heads x (sink + w) floats) on chip.
constexpr int kMaxM = 64;
constexpr int kMaxDim = 256;
constexpr int kMaxHeads = 64;
constexpr int kMaxNear = 2048;  // sink + w

// Per-group integer slots in the `ints` region.
enum : int {
  kIntWinHead = 0,
  kIntWinLen = 1,
  kIntMEff = 2,
  kIntT = 3,
  kIntMode = 4,
  kIntStatus = 5,  // nonzero: a bounded wait in the step kernel gave up
  kIntsPerGroup = 8
};
enum : int { kModeEmpty = 0, kModeSealed = 1, kModeExact = 2 };
constexpr int kMaxExactCap = 4096;

// Device pointers of every state region plus the geometry, passed by value
// to the kernels.  Region layout: see nys_layout in nys.h.
struct DevState {
  float* win_k;
  float* win_v;
  float* sink_k;
  float* sink_v;
  float* k_tilde;
  float* q_tilde;
  float* mu;
  float* t_hat;
  float* z_hat;
  float* m_max;
  uint16_t* t_lo;  // bf16 bits: low part of t_hat
  float* z_lo;     // low part of z_hat
  int32_t* far_len;
  int32_t* ints;
  float* exact_k;  // [G][exact_cap][d], exact-only groups
  float* exact_v;  // [G][exact_cap][dv]
  int32_t m, w, sink, heads, d, dv, rect, exact_cap;
  float scale;  // 1/sqrt(d) evaluated in f32
};

#ifdef __CUDACC__
// Compensated update of an unevaluated sum hi + lo:
//   (hi + lo) * r + x * y  ->  (nhi, nlo),  nhi = fl(value), nlo = remainder.
// The product errors come exactly from FMA (a*b - fl(a*b)), the sum error from
// Knuth's two-sum, so the pair tracks the update to ~2^-48 relative instead of
// rounding it to 2^-24 each time.  Used for the far accumulators T^ and Z^.
// r == 1 (no new running maximum, the common case) skips the rescale terms.
__device__ __forceinline__ void comp_axpy(float hi, float lo, float r, float x, float y,
                                          float& nhi, float& nlo) {
  const float b = x * y;
  const float pb = fmaf(x, y, -b);
  float a = hi, t0 = pb;
  if (r != 1.f) {
    a = hi * r;
    t0 += fmaf(hi, r, -a);
    lo *= r;
  }
  const float s = a + b;
  const float sb = s - a;
  const float es = (a - (s - sb)) + (b - sb);
  const float t = lo + (t0 + es);
  nhi = s + t;
  nlo = t - (nhi - s);
}

// ---- double-float arithmetic (unevaluated pairs hi + lo of f32) for the
// sums that need more than f32: GB300's f32 pipe is tens of times faster
// than its f64 pipe.  df_two_sum is Knuth's exact sum, df_fast_two_sum
// Dekker's (|a| >= |b|), df_mul the product of two pairs by FMA.
__device__ __forceinline__ void df_two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float z = s - a;
  e = (a - (s - z)) + (b - z);
}
__device__ __forceinline__ void df_fast_two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  e = b - (s - a);
}
__device__ __forceinline__ void df_mul(float ah, float al, float bh, float bl, float& ph,
                                       float& pl) {
  const float p = ah * bh;
  float e = fmaf(ah, bh, -p);
  e = fmaf(ah, bl, e);
  e = fmaf(al, bh, e);
  df_fast_two_sum(p, e, ph, pl);
}
__device__ __forceinline__ void df_add(float ah, float al, float bh, float bl, float& sh,
                                       float& sl) {
  float s, e;
  df_two_sum(ah, bh, s, e);
  e += al + bl;
  df_fast_two_sum(s, e, sh, sl);
}
// e^{a + b - c} for f32 a, b, c, without rounding the exponent: the
// exponent is formed exactly as a pair (xh, xl) and e^{xh + xl} taken as
// expf(xh) (1 + xl), |xl| <= ulp(xh) / 2 (the second-order term is below
// 2^-48).  Returns the value as a pair (hi, lo); only expf's own error
// remains.  a + b may be -INF (no key absorbed yet): then the result is 0.
__device__ __forceinline__ void exp_sum_pair(float a, float b, float c, float& hi, float& lo) {
  float s1, e1, s2, e2, xh, xl;
  df_two_sum(a, b, s1, e1);
  df_two_sum(s1, -c, s2, e2);
  if (!isfinite(s2)) {  // -INF: nothing absorbed (the error terms are NaN)
    hi = expf(s2);
    lo = 0.f;
    return;
  }
  df_fast_two_sum(s2, e1 + e2, xh, xl);
  hi = expf(xh);
  lo = hi * xl;
}

// Kahan's compensated update of the running sum hi + lo by one term x * y,
// after an optional rescale by r: lo carries the rounding error of the
// running sum (recovered by Fast2Sum), so many steps drift no more than a
// rounding or two.  Five operations when r == 1 against comp_axpy's twelve;
// the rescale's own rounding error is recovered exactly by FMA.
__device__ __forceinline__ void kahan_axpy(float& hi, float& lo, float r, float x, float y) {
  if (r != 1.f) {
    const float a = hi * r;
    lo = fmaf(lo, r, fmaf(hi, r, -a));
    hi = a;
  }
  const float yv = fmaf(x, y, lo);
  const float t = hi + yv;
  lo = yv - (t - hi);
  hi = t;
}

// kahan_axpy on four elements sharing r and e (one T^ row chunk): the rescale
// test is taken once for the four, then each element gets the same
// operations in the same order as kahan_axpy.
__device__ __forceinline__ void kahan_axpy4(float4& hi, float4& lo, float r, float e, float4 v) {
  if (r != 1.f) {
    float a = hi.x * r;
    lo.x = fmaf(lo.x, r, fmaf(hi.x, r, -a));
    hi.x = a;
    a = hi.y * r;
    lo.y = fmaf(lo.y, r, fmaf(hi.y, r, -a));
    hi.y = a;
    a = hi.z * r;
    lo.z = fmaf(lo.z, r, fmaf(hi.z, r, -a));
    hi.z = a;
    a = hi.w * r;
    lo.w = fmaf(lo.w, r, fmaf(hi.w, r, -a));
    hi.w = a;
  }
  float yv = fmaf(e, v.x, lo.x), t = hi.x + yv;
  lo.x = yv - (t - hi.x);
  hi.x = t;
  yv = fmaf(e, v.y, lo.y);
  t = hi.y + yv;
  lo.y = yv - (t - hi.y);
  hi.y = t;
  yv = fmaf(e, v.z, lo.z);
  t = hi.z + yv;
  lo.z = yv - (t - hi.z);
  hi.z = t;
  yv = fmaf(e, v.w, lo.w);
  t = hi.w + yv;
  lo.w = yv - (t - hi.w);
  hi.w = t;
}

// comp_axpy with r == 1, for callers that branch on r once for many elements.
__device__ __forceinline__ void comp_add(float hi, float lo, float x, float y, float& nhi,
                                         float& nlo) {
  const float b = x * y;
  const float pb = fmaf(x, y, -b);
  const float s = hi + b;
  const float sb = s - hi;
  const float es = (hi - (s - sb)) + (b - sb);
  const float t = lo + (pb + es);
  nhi = s + t;
  nlo = t - (nhi - s);
}

// Compensated dot product (Ogita, Rump and Oishi's Dot2): sum_a x[a] * y[a*ys]
// with each product's rounding error recovered by FMA and each addition's by
// two-sum, so the result is as accurate as if accumulated in twice the
// precision.  The mixing row u = F^ M is a sum with heavy cancellation (M is
// the ridge pseudo-inverse of an ill-conditioned kernel matrix), and plain
// f32 accumulation there costs up to ~1e-4 of output accuracy at m = 64.
// Two interleaved chains shorten the dependency chain.
__device__ __forceinline__ float dot2(const float* x, const float* y, int ys, int n) {
  float s0 = 0.f, c0 = 0.f, s1 = 0.f, c1 = 0.f;
  int a = 0;
  for (; a + 2 <= n; a += 2) {
    {
      const float h = x[a] * y[a * ys];
      const float r = fmaf(x[a], y[a * ys], -h);
      const float t = s0 + h;
      const float z = t - s0;
      c0 += ((s0 - (t - z)) + (h - z)) + r;
      s0 = t;
    }
    {
      const float h = x[a + 1] * y[(a + 1) * ys];
      const float r = fmaf(x[a + 1], y[(a + 1) * ys], -h);
      const float t = s1 + h;
      const float z = t - s1;
      c1 += ((s1 - (t - z)) + (h - z)) + r;
      s1 = t;
    }
  }
  if (a < n) {
    const float h = x[a] * y[a * ys];
    const float r = fmaf(x[a], y[a * ys], -h);
    const float t = s0 + h;
    const float z = t - s0;
    c0 += ((s0 - (t - z)) + (h - z)) + r;
    s0 = t;
  }
  const float t = s0 + s1;
  const float z = t - s0;
  const float e = (s0 - (t - z)) + (s1 - z);
  return t + ((c0 + c1) + e);
}

// dot2 with x read four at a time (x 16-byte aligned): the same operations
// in the same order -- even terms on the first chain, odd on the second --
// so the result is bit-identical to dot2's.
__device__ __forceinline__ float dot2_x4(const float* x, const float* y, int ys, int n) {
  float s0 = 0.f, c0 = 0.f, s1 = 0.f, c1 = 0.f;
  auto term = [](float& sv, float& cv, float xa, float ya) {
    const float h = xa * ya;
    const float r = fmaf(xa, ya, -h);
    const float t = sv + h;
    const float z = t - sv;
    cv += ((sv - (t - z)) + (h - z)) + r;
    sv = t;
  };
  int a = 0;
  for (; a + 4 <= n; a += 4) {
    const float4 xv = *reinterpret_cast<const float4*>(x + a);
    term(s0, c0, xv.x, y[a * ys]);
    term(s1, c1, xv.y, y[(a + 1) * ys]);
    term(s0, c0, xv.z, y[(a + 2) * ys]);
    term(s1, c1, xv.w, y[(a + 3) * ys]);
  }
  if (a + 2 <= n) {
    term(s0, c0, x[a], y[a * ys]);
    term(s1, c1, x[a + 1], y[(a + 1) * ys]);
    a += 2;
  }
  if (a < n) term(s0, c0, x[a], y[a * ys]);
  const float t = s0 + s1;
  const float z = t - s0;
  const float e = (s0 - (t - z)) + (s1 - z);
  return t + ((c0 + c1) + e);
}
// dot2_x4 with the result kept as a normalised pair (hi is dot2_x4's value).
__device__ __forceinline__ void dot2_x4_pair(const float* x, const float* y, int ys, int n,
                                             float& hi, float& lo) {
  float s0 = 0.f, c0 = 0.f, s1 = 0.f, c1 = 0.f;
  auto term = [](float& sv, float& cv, float xa, float ya) {
    const float h = xa * ya;
    const float r = fmaf(xa, ya, -h);
    const float t = sv + h;
    const float z = t - sv;
    cv += ((sv - (t - z)) + (h - z)) + r;
    sv = t;
  };
  int a = 0;
  for (; a + 4 <= n; a += 4) {
    const float4 xv = *reinterpret_cast<const float4*>(x + a);
    term(s0, c0, xv.x, y[a * ys]);
    term(s1, c1, xv.y, y[(a + 1) * ys]);
    term(s0, c0, xv.z, y[(a + 2) * ys]);
    term(s1, c1, xv.w, y[(a + 3) * ys]);
  }
  if (a + 2 <= n) {
    term(s0, c0, x[a], y[a * ys]);
    term(s1, c1, x[a + 1], y[(a + 1) * ys]);
    a += 2;
  }
  if (a < n) term(s0, c0, x[a], y[a * ys]);
  const float t = s0 + s1;
  const float z = t - s0;
  const float e = (s0 - (t - z)) + (s1 - z);
  df_fast_two_sum(t, (c0 + c1) + e, hi, lo);
}

// bf16 storage of low parts: two values per 32-bit word, round to nearest
// even (hardware conversion).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
#endif

// One decode token for groups [g0, g0+n): one kernel launch on `stream`.
// debug_skip >= 0 (test hook) makes the fast kernel's first CTA withhold that
// ring stage, so its bounded waits run out.
cudaError_t launch_step(const DevState& s, int64_t g0, int64_t n,
                        const float* q, const float* k, const float* v,
                        float* out, cudaStream_t stream, int debug_skip = -1);

// Fast path of the step (nys_step_tma.cu): plan_step_tma fills an opaque
// plan of at most kPlanBytes and returns false for geometries it does not
// cover; launch_step_tma runs it.
constexpr size_t kPlanBytes = 512;
bool plan_step_tma(const DevState& s, void* plan_out);
size_t step_tma_plan_bytes();
cudaError_t launch_step_tma(const DevState& s, const void* plan, int64_t g0, int64_t n,
                            const float* q, const float* k, const float* v, float* out,
                            cudaStream_t stream, int debug_skip = -1);

// Prompt geometry of a seal launch.  Uniform batches (every group has prompt
// length t and m_eff landmarks, group i's rows start at i * t) leave the
// arrays null; ragged batches give per-group length, landmark count and
// first row (device arrays indexed by the group's position in the launch).
struct SealGeom {
  int t, m_eff;
  const int32_t* t_arr;
  const int32_t* me_arr;
  const int64_t* off_arr;
};
#ifdef __CUDACC__
__device__ __forceinline__ void seal_geom(const SealGeom& sg, int64_t gi, int& t, int& me,
                                          int64_t& off) {
  if (sg.t_arr) {
    t = sg.t_arr[gi];
    me = sg.me_arr[gi];
    off = sg.off_arr[gi];
  } else {
    t = sg.t;
    me = sg.m_eff;
    off = gi * (int64_t)sg.t;
  }
}
#endif

// Exact-only (short-prompt) groups: copy the prompt into the exact region and
// set the counters (seal), and one decode token of exact softmax attention over
// every key held (step; groups in other modes are left alone).
cudaError_t launch_exact_seal(const DevState& s, int64_t g0, int64_t n, int t, const float* k,
                              const float* v, cudaStream_t stream);
cudaError_t launch_exact_step(const DevState& s, int64_t g0, int64_t n, const float* q,
                              const float* k, const float* v, float* out, cudaStream_t stream);

// Bytes of f64 workspace the seal needs per group (key landmarks and every
// head's query landmarks before rounding).
size_t seal_workspace_bytes_per_group(const DevState& s);

// A second stream for the seal: the pinv (which needs the landmarks) and the
// replay (which needs Q~ but not M) are independent, so the pinv runs on
// `side` next to the replay on the caller's stream (measured: long seal
// 86.8 -> 85.7 ms, a ragged m = 64 batch 5.29 -> 5.08 ms, the rest within
// 1%; with the replay on a high-priority side stream instead, slower).  The
// seal forks `side` from the caller's stream after the landmarks and joins
// it back before it returns; null members keep everything on one stream.
struct SealFork {
  cudaStream_t side = nullptr;
  cudaEvent_t forked = nullptr, joined = nullptr;
  bool on() const { return side && forked && joined; }
};

// Seal groups [g0, g0+n) with prompt length t and m_eff landmarks, using
// `ws` (seal_workspace_bytes_per_group * n bytes) as f64 scratch.  Three
// kernel launches on `stream` (the pinv on fork.side when fork is on; the
// call returns with `stream` ordered after all of them).
// debug_stall (test hook): the tensor-core replay's first CTA withholds its
// first MMA, so its bounded waits run out (status 3 for its group).
cudaError_t launch_seal(const DevState& s, int64_t g0, int64_t n, int t,
                        int m_eff, const float* q, const float* k,
                        const float* v, double* ws, cudaStream_t stream,
                        int debug_stall = 0, const SealFork& fork = SealFork());

// Seal with per-group prompt geometry (sg's arrays on the device, indexed
// from 0 for group g0); max_me bounds every group's m_eff.  q, k, v point at
// the start of the packed batch.
cudaError_t launch_seal_geom(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                             int max_me, const float* q, const float* k, const float* v,
                             double* ws, cudaStream_t stream, int debug_stall = 0,
                             const SealFork& fork = SealFork());

// Tensor-core replay (nys_replay_tc.cu): whether the geometry fits it
// (m >= 32, d and dv <= 128 in multiples of 32), and its launch.  It takes
// the groups whose replay folds at least kReplayTcMinKeys keys; the CUDA-core
// replay takes the others (its per-CTA setup is cheaper for short prompts),
// so a group's result does not depend on the batch it is sealed in.
constexpr int kReplayTcMinKeys = 256;
bool replay_tc_fits(const DevState& s);
cudaError_t launch_replay_tc(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                             const float* k, const float* v, cudaStream_t stream,
                             int debug_stall = 0);

// One uniform-length seal request after the host-side checks that every
// seal entry point shares (nys_seal, nys_seal_static): range, prompt length,
// pointers, alignment, and the page's mode choice (nystrom.rs,
// prefill_shared).  `exact` marks an exact-only prompt (t <= w + sink + 8) on
// a handle that has an exact region; otherwise the landmark path runs with
// m_eff landmarks on the device view `ds`.
struct SealPlan {
  bool exact = false;
  int m_eff = 0;
  DevState ds;
};

// Check a seal request and fill `plan` (printing the one-time clamp notice
// when m_eff < m and n > 0).  Returns a nys_status; nothing is enqueued.
int plan_seal(nys_states* st, int64_t g0, int64_t n, int32_t t, const float* q,
              const float* k, const float* v, SealPlan* plan);

// Seal groups [g0, g0+n) in exact-only mode (no workspace needed) and record
// them as exact-only groups on the host.  Returns a nys_status.
int run_exact_seal(nys_states* st, int64_t g0, int64_t n, int32_t t, const float* k,
                   const float* v, cudaStream_t stream);

// Host record that groups [g0, g0+n) hold a landmark-path sealed state.
void record_sealed(nys_states* st, int64_t g0, int64_t n);

}  // namespace nys
