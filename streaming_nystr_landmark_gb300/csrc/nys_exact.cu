// Exact-only (short-prompt) groups on the GPU.
//
// nystrom.rs (docs.rs source view, cortiq-engine 0.5.71), prefill_shared and
// NystromHead::seal_exact: a prompt of t <= w + sink + 8 keys builds no
// skeleton -- every key stays an exact key in a window that grows by one key
// per decode token (NystromState::advance, exact-only branch), there are no
// sinks and no far field, and each output is plain softmax attention over all
// keys held (NystromHead::step with sink_len = 0 and far_len = 0).  The page's
// own GPU mirror refuses such groups; here they live in a separate region of
// exact_cap rows per group, and the host refuses a token that would overflow
// it before anything is launched.
#include <cmath>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Block-wide max / sum through a 32-float scratch; every thread gets the result.
__device__ float block_max(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_max(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float r = lane < kWarps ? red[lane] : -INFINITY;
  r = warp_max(r);
  __syncthreads();
  return r;
}
__device__ float block_sum(float x, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = warp_sum(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float r = lane < kWarps ? red[lane] : 0.f;
  r = warp_sum(r);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads)
exact_seal_kernel(DevState s, int64_t g0, int t, const float* __restrict__ k,
                  const float* __restrict__ v) {
  const int64_t gi = blockIdx.x, g = g0 + gi;
  const int d = s.d, dv = s.dv, cap = s.exact_cap, H = s.heads;
  float* ek = s.exact_k + g * (int64_t)cap * d;
  float* ev = s.exact_v + g * (int64_t)cap * dv;
  const float* ks = k + gi * (int64_t)t * d;
  const float* vs = v + gi * (int64_t)t * dv;
  for (int64_t i = threadIdx.x; i < (int64_t)t * d; i += kThreads) ek[i] = ks[i];
  for (int64_t i = threadIdx.x; i < (int64_t)t * dv; i += kThreads) ev[i] = vs[i];
  if (threadIdx.x == 0) {
    int32_t* ints = s.ints + g * kIntsPerGroup;
    ints[kIntWinHead] = 0;
    ints[kIntWinLen] = t;
    ints[kIntMEff] = 0;
    ints[kIntT] = t;
    ints[kIntMode] = kModeExact;
    ints[kIntStatus] = 0;
  }
  for (int h = threadIdx.x; h < H; h += kThreads) s.far_len[g * H + h] = 0;
}

__global__ void __launch_bounds__(kThreads)
exact_step_kernel(DevState s, int64_t g0, const float* __restrict__ q,
                  const float* __restrict__ k, const float* __restrict__ v,
                  float* __restrict__ out) {
  extern __shared__ float esm[];
  const int64_t gi = blockIdx.x, g = g0 + gi;
  int32_t* ints = s.ints + g * kIntsPerGroup;
  if (ints[kIntMode] != kModeExact) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = s.d, dv = s.dv, cap = s.exact_cap, H = s.heads;
  const int held = ints[kIntWinLen];  // < cap, checked on the host
  float* ek = s.exact_k + g * (int64_t)cap * d;
  float* ev = s.exact_v + g * (int64_t)cap * dv;
  // Append this token's key and value (the exact window grows by one).
  for (int c = tid; c < d; c += kThreads) ek[(int64_t)held * d + c] = k[gi * d + c];
  for (int c = tid; c < dv; c += kThreads) ev[(int64_t)held * dv + c] = v[gi * dv + c];
  __syncthreads();
  const int n = held + 1;
  float* lg = esm;          // [n] logits, then weights
  float* red = esm + cap + 1;
  for (int h = 0; h < H; ++h) {
    const float* qh = q + (gi * H + h) * (int64_t)d;
    for (int j = warp; j < n; j += kWarps) {
      const float* row = ek + (int64_t)j * d;
      float acc = 0.f;
      for (int c = lane; c < d; c += 32) acc = fmaf(qh[c], row[c], acc);
      acc = warp_sum(acc);
      if (lane == 0) lg[j] = acc * s.scale;
    }
    __syncthreads();
    float mx = -INFINITY;
    for (int j = tid; j < n; j += kThreads) mx = fmaxf(mx, lg[j]);
    mx = block_max(mx, red);
    float ps = 0.f;
    for (int j = tid; j < n; j += kThreads) {
      const float p = expf(lg[j] - mx);
      lg[j] = p;
      ps += p;
    }
    const float den = fmaxf(block_sum(ps, red), 1e-30f);
    for (int c = tid; c < dv; c += kThreads) {
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(lg[j], ev[(int64_t)j * dv + c], acc);
      out[(gi * H + h) * (int64_t)dv + c] = acc / den;
    }
    __syncthreads();
  }
  if (tid == 0) ints[kIntWinLen] = n;
}

}  // namespace

cudaError_t launch_exact_seal(const DevState& s, int64_t g0, int64_t n, int t, const float* k,
                              const float* v, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  exact_seal_kernel<<<(unsigned)n, kThreads, 0, stream>>>(s, g0, t, k, v);
  return cudaGetLastError();
}

cudaError_t launch_exact_step(const DevState& s, int64_t g0, int64_t n, const float* q,
                              const float* k, const float* v, float* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const size_t bytes = ((size_t)s.exact_cap + 1 + 32) * sizeof(float);
  exact_step_kernel<<<(unsigned)n, kThreads, bytes, stream>>>(s, g0, q, k, v, out);
  return cudaGetLastError();
}

}  // namespace nys
