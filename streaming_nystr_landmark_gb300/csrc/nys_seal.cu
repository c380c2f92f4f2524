// Batched seal (prefill) of streaming Nystrom attention states.
//
// Follows nystrom.rs (docs.rs source view, cortiq-engine 0.5.71),
// NystromState::prefill_group, in three launches over all groups at once:
//
//  1. landmarks_kernel, grid (n, 1 + heads): block (g, 0) takes the group's
//     keys -- K~ = seg_means(k) (prefill_shared), sinks, ring fill, counters;
//     block (g, 1 + h) takes head h's queries -- Q~_h = seg_means(q_h)
//     (NystromHead::seal).  Segment i covers rows [i t / m_eff,
//     (i+1) t / m_eff); sums are accumulated in f64 (fn seg_means).  The f64
//     means go to a workspace for step 2, their f32 roundings to the state.
//  2. pinv_kernel, one block per (group, head): A = exp(Q~64 K~64^T * scale)
//     in f64, then M = (A^T A + lambda I)^-1 A^T (fn ridge_pinv):
//     lambda = 1e-6 * max(mean diag(A^T A), DBL_MIN); a failed Cholesky
//     (pivot not > 0 or not finite, fn cholesky) multiplies lambda by ten, at
//     most twelve attempts, then M = I / max(mean diag, DBL_MIN).  The
//     Cholesky and the two triangular solves keep the page's summation order.
//  3. replay_kernel, one block per (group, head): the replay of positions
//     sink..t-1 through the ring leaves keys sink..t-w-1 in the far field
//     (NystromState::advance -> NystromHead::far_insert).  The state that
//     sequential loop produces is m_max_i = max_j l_ij, Z^_i = sum_j
//     exp(l_ij - m_max_i), T^_i = sum_j exp(l_ij - m_max_i) v_j with
//     l_ij = (q~_i . k_j) * scale in f32; this kernel reaches it with a
//     blocked online maximum (flash-style rescale per block of keys), which
//     changes only the rounding order, and folds each block's sums into
//     compensated (hi, lo) accumulators so that tens of thousands of
//     evictions do not accumulate f32 rounding.
#include <cfloat>
#include <cmath>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ void st4(float* p, float4 x) {
  *reinterpret_cast<float4*>(p) = x;
}

// ---------------------------------------------------------------- 1
__global__ void __launch_bounds__(kThreads)
landmarks_kernel(DevState s, int64_t g0, int t, int m_eff,
                 const float* __restrict__ q, const float* __restrict__ k,
                 const float* __restrict__ v, double* __restrict__ ws) {
  __shared__ double red[kWarps][128];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t gi = blockIdx.x, g = g0 + gi;
  const int r = blockIdx.y;  // 0: keys, 1 + h: queries of head h
  const int d = s.d, dv = s.dv, H = s.heads, m = s.m, w = s.w, ns = s.sink;
  const int d4 = d >> 2, dv4 = dv >> 2;

  const float* src;
  float* dst32;
  if (r == 0) {
    src = k + gi * (int64_t)t * d;
    dst32 = s.k_tilde + g * m * (int64_t)d;
  } else {
    src = q + ((gi * H + (r - 1)) * (int64_t)t) * d;
    dst32 = s.q_tilde + ((g * H + (r - 1)) * m) * (int64_t)d;
  }
  double* dst64 = ws + (gi * (1 + H) + r) * (int64_t)m * d;

  for (int i = 0; i < m_eff; ++i) {
    const int lo = (int)(((int64_t)i * t) / m_eff);
    const int hi = (int)(((int64_t)(i + 1) * t) / m_eff);
    const double inv = 1.0 / (double)(hi - lo);
    for (int ct = 0; ct < d; ct += 128) {
      const int c4 = (ct >> 2) + lane;
      const bool cv = c4 < d4;
      double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
      if (cv) {
#pragma unroll 4
        for (int j = lo + warp; j < hi; j += kWarps) {
          const float4 x = ld4(src + (int64_t)j * d + 4 * c4);
          a0 += (double)x.x;
          a1 += (double)x.y;
          a2 += (double)x.z;
          a3 += (double)x.w;
        }
        red[warp][4 * lane + 0] = a0;
        red[warp][4 * lane + 1] = a1;
        red[warp][4 * lane + 2] = a2;
        red[warp][4 * lane + 3] = a3;
      }
      __syncthreads();
      if (tid < 128 && ct + tid < d) {
        double sum = 0.0;
#pragma unroll
        for (int wp = 0; wp < kWarps; ++wp) sum += red[wp][tid];
        const double mean = sum * inv;
        dst64[(int64_t)i * d + ct + tid] = mean;
        dst32[(int64_t)i * d + ct + tid] = (float)mean;
      }
      __syncthreads();
    }
  }

  if (r != 0) return;
  // Sinks: positions 0..sink, permanent (prefill_shared).
  const float* vsrc = v + gi * (int64_t)t * dv;
  for (int idx = tid; idx < ns * d4; idx += kThreads)
    st4(s.sink_k + g * ns * (int64_t)d + 4 * idx, ld4(src + 4 * idx));
  for (int idx = tid; idx < ns * dv4; idx += kThreads)
    st4(s.sink_v + g * ns * (int64_t)dv + 4 * idx, ld4(vsrc + 4 * idx));
  // Ring: post-sink position j sits in slot (j - sink) mod w; the last w
  // positions t-w..t-1 are the ones left after the replay.
  for (int idx = tid; idx < w * d4; idx += kThreads) {
    const int jj = idx / d4, c = idx - jj * d4;
    const int j = t - w + jj;
    const int slot = (j - ns) % w;
    st4(s.win_k + (g * w + slot) * (int64_t)d + 4 * c,
        ld4(src + (int64_t)j * d + 4 * c));
  }
  for (int idx = tid; idx < w * dv4; idx += kThreads) {
    const int jj = idx / dv4, c = idx - jj * dv4;
    const int j = t - w + jj;
    const int slot = (j - ns) % w;
    st4(s.win_v + (g * w + slot) * (int64_t)dv + 4 * c,
        ld4(vsrc + (int64_t)j * dv + 4 * c));
  }
  if (tid == 0) {
    int32_t* ints = s.ints + g * kIntsPerGroup;
    ints[kIntWinHead] = (t - ns) % w;
    ints[kIntWinLen] = w;
    ints[kIntMEff] = m_eff;
    ints[kIntT] = t;
    ints[kIntMode] = kModeSealed;
  }
  for (int h = tid; h < H; h += kThreads) s.far_len[g * H + h] = t - ns - w;
}

// ---------------------------------------------------------------- 2
constexpr int kTile = 32;        // landmark-product column tile
constexpr int kTileStride = 33;  // padded row stride of the tiles (doubles)

__host__ __device__ inline size_t pinv_smem_doubles(int me) {
  return 3 * (size_t)me * me + 2 * (size_t)me * kTileStride;
}

__global__ void __launch_bounds__(kThreads)
pinv_kernel(DevState s, int64_t g0, int m_eff, const double* __restrict__ ws) {
  extern __shared__ __align__(16) double dsm[];
  __shared__ int fail;
  __shared__ double lam_s, mean_diag_s;
  const int tid = threadIdx.x;
  const int H = s.heads, m = s.m, d = s.d, me = m_eff;
  const int64_t gi = blockIdx.x / H, g = g0 + gi;
  const int h = (int)(blockIdx.x - gi * H);
  double* A = dsm;            // [me][me]
  double* G = A + me * me;    // [me][me]  A^T A
  double* Lf = G + me * me;   // [me][me]  Cholesky factor / working copy
  double* Qt = Lf + me * me;  // [me][kTileStride]
  double* Kt = Qt + me * kTileStride;
  const double* K64 = ws + (gi * (1 + H)) * (int64_t)m * d;
  const double* Q64 = ws + (gi * (1 + H) + 1 + h) * (int64_t)m * d;
  const double scale = (double)s.scale;

  // A[i][j] = exp((q~64_i . k~64_j) * scale)
  constexpr int kPer = (kMaxM * kMaxM + kThreads - 1) / kThreads;
  double acc[kPer];
#pragma unroll
  for (int p = 0; p < kPer; ++p) acc[p] = 0.0;
  for (int c0 = 0; c0 < d; c0 += kTile) {
    const int cw = min(kTile, d - c0);
    for (int idx = tid; idx < me * kTile; idx += kThreads) {
      const int i = idx / kTile, cc = idx - i * kTile;
      Qt[i * kTileStride + cc] = cc < cw ? Q64[(int64_t)i * d + c0 + cc] : 0.0;
      Kt[i * kTileStride + cc] = cc < cw ? K64[(int64_t)i * d + c0 + cc] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < kPer; ++p) {
      const int pair = tid + p * kThreads;
      if (pair < me * me) {
        const int i = pair / me, j = pair - i * me;
        double a = acc[p];
        for (int cc = 0; cc < cw; ++cc)
          a = fma(Qt[i * kTileStride + cc], Kt[j * kTileStride + cc], a);
        acc[p] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < kPer; ++p) {
    const int pair = tid + p * kThreads;
    if (pair < me * me) A[pair] = exp(acc[p] * scale);
  }
  __syncthreads();

  // G = A^T A
  for (int pair = tid; pair < me * me; pair += kThreads) {
    const int i = pair / me, j = pair - i * me;
    double a = 0.0;
    for (int kk = 0; kk < me; ++kk) a = fma(A[kk * me + i], A[kk * me + j], a);
    G[pair] = a;
  }
  __syncthreads();
  if (tid == 0) {
    double sd = 0.0;
    for (int i = 0; i < me; ++i) sd += G[i * me + i];
    mean_diag_s = sd / (double)me;
    lam_s = 1e-6 * fmax(mean_diag_s, DBL_MIN);
  }
  __syncthreads();

  bool solved = false;
  for (int attempt = 0; attempt < 12 && !solved; ++attempt) {
    const double lam = lam_s;
    for (int pair = tid; pair < me * me; pair += kThreads) {
      const int i = pair / me, j = pair - i * me;
      Lf[pair] = G[pair] + (i == j ? lam : 0.0);
    }
    if (tid == 0) fail = 0;
    __syncthreads();
    for (int j = 0; j < me; ++j) {
      if (tid == 0) {
        double sp = Lf[j * me + j];
        for (int kk = 0; kk < j; ++kk) sp -= Lf[j * me + kk] * Lf[j * me + kk];
        if (!(sp > 0.0) || !isfinite(sp)) fail = 1;
        else Lf[j * me + j] = sqrt(sp);
      }
      __syncthreads();
      if (fail) break;
      for (int i = j + 1 + tid; i < me; i += kThreads) {
        double a = Lf[i * me + j];
        for (int kk = 0; kk < j; ++kk) a -= Lf[i * me + kk] * Lf[j * me + kk];
        Lf[i * me + j] = a / Lf[j * me + j];
      }
      __syncthreads();
    }
    if (!fail) {
      solved = true;
    } else {
      __syncthreads();
      if (tid == 0) lam_s = lam * 10.0;
      __syncthreads();
    }
  }

  float* M = s.mu + (g * H + h) * (int64_t)m * m;
  if (solved) {
    // G M = A^T, one right-hand side (row j of A) per thread; X reuses G.
    double* X = G;
    __syncthreads();
    for (int j = tid; j < me; j += kThreads) {
      for (int i = 0; i < me; ++i) {
        double a = A[j * me + i];
        for (int kk = 0; kk < i; ++kk) a -= Lf[i * me + kk] * X[kk * me + j];
        X[i * me + j] = a / Lf[i * me + i];
      }
      for (int i = me - 1; i >= 0; --i) {
        double a = X[i * me + j];
        for (int kk = i + 1; kk < me; ++kk) a -= Lf[kk * me + i] * X[kk * me + j];
        X[i * me + j] = a / Lf[i * me + i];
      }
    }
    __syncthreads();
    for (int pair = tid; pair < me * me; pair += kThreads) {
      const int i = pair / me, j = pair - i * me;
      M[i * m + j] = (float)X[pair];
    }
  } else {
    const double diag = 1.0 / fmax(mean_diag_s, DBL_MIN);
    for (int pair = tid; pair < me * me; pair += kThreads) {
      const int i = pair / me, j = pair - i * me;
      M[i * m + j] = (i == j) ? (float)diag : 0.f;
    }
  }
}

// ---------------------------------------------------------------- 3
constexpr int kKeyBlock = 32;
constexpr int kValTile = 128;  // value columns per block (grid.y tiles dv)

struct ReplaySmem {
  int qt, kb, vb, p, hi, lo, rmax, zhi, zlo, alpha, total, dp, pp;
  __host__ __device__ ReplaySmem(int me, int d) {
    dp = d + 4;  // skewed rows: float4 reads across lanes hit all banks
    pp = kKeyBlock + 1;
    const int m4 = (me + 3) & ~3;
    int o = 0;
    qt = o;    o += me * dp;
    kb = o;    o += kKeyBlock * dp;
    vb = o;    o += kKeyBlock * kValTile;
    p = o;     o += ((me * pp + 3) & ~3);
    hi = o;    o += me * kValTile;
    lo = o;    o += me * kValTile;
    rmax = o;  o += m4;
    zhi = o;   o += m4;
    zlo = o;   o += m4;
    alpha = o; o += m4;
    total = o;
  }
};

// One block per (group, head, value tile).  Keys are consumed in blocks of
// kKeyBlock: logits L = Q~ K_blk^T * scale, a per-landmark online maximum,
// block sums of exp(L - max) and of exp(L - max) v, and a compensated fold of
// each block sum into the running (hi, lo) accumulators.  Every value tile
// recomputes the same logits, so the tile with blockIdx.y == 0 alone writes
// m_max and Z^.
__global__ void __launch_bounds__(kThreads)
replay_kernel(DevState s, int64_t g0, int t, int m_eff,
              const float* __restrict__ k, const float* __restrict__ v) {
  extern __shared__ __align__(16) float fsm[];
  const int tid = threadIdx.x;
  const int H = s.heads, m = s.m, d = s.d, dv = s.dv, w = s.w, ns = s.sink;
  const int d4 = d >> 2, me = m_eff;
  const int64_t gi = blockIdx.x / H, g = g0 + gi;
  const int h = (int)(blockIdx.x - gi * H);
  const int64_t hb = g * H + h;
  const int c0 = blockIdx.y * kValTile;
  const int cw = min(kValTile, dv - c0);
  const int cw4 = cw >> 2;
  const float scale = s.scale;
  const ReplaySmem L(me, d);
  float* qt = fsm + L.qt;
  float* kb = fsm + L.kb;
  float* vb = fsm + L.vb;
  float* P = fsm + L.p;
  float* ahi = fsm + L.hi;
  float* alo = fsm + L.lo;
  float* rmax = fsm + L.rmax;
  float* zhi = fsm + L.zhi;
  float* zlo = fsm + L.zlo;
  float* alpha = fsm + L.alpha;

  const float* qsrc = s.q_tilde + hb * m * (int64_t)d;
  for (int idx = tid; idx < me * d4; idx += kThreads) {
    const int i = idx / d4, c = idx - i * d4;
    st4(qt + i * L.dp + 4 * c, ld4(qsrc + (int64_t)i * d + 4 * c));
  }
  for (int i = tid; i < me; i += kThreads) {
    rmax[i] = -INFINITY;
    zhi[i] = 0.f;
    zlo[i] = 0.f;
  }
  for (int idx = tid; idx < me * kValTile; idx += kThreads) {
    ahi[idx] = 0.f;
    alo[idx] = 0.f;
  }

  const float* ksrc = k + gi * (int64_t)t * d;
  const float* vsrc = v + gi * (int64_t)t * dv + c0;
  const int j_end = t - w;  // keys sink .. t-w-1 were evicted by the replay
  for (int j0 = ns; j0 < j_end; j0 += kKeyBlock) {
    const int nb = min(kKeyBlock, j_end - j0);
    for (int idx = tid; idx < nb * d4; idx += kThreads) {
      const int jj = idx / d4, c = idx - jj * d4;
      st4(kb + jj * L.dp + 4 * c, ld4(ksrc + (int64_t)(j0 + jj) * d + 4 * c));
    }
    for (int idx = tid; idx < nb * cw4; idx += kThreads) {
      const int jj = idx / cw4, c = idx - jj * cw4;
      st4(vb + jj * kValTile + 4 * c, ld4(vsrc + (int64_t)(j0 + jj) * dv + 4 * c));
    }
    __syncthreads();
    for (int p = tid; p < me * nb; p += kThreads) {
      const int i = p / nb, jj = p - i * nb;
      const float* a = qt + i * L.dp;
      const float* b = kb + jj * L.dp;
      float x = 0.f;
      for (int c = 0; c < d4; ++c) {
        const float4 qa = ld4(a + 4 * c), kk = ld4(b + 4 * c);
        x += qa.x * kk.x + qa.y * kk.y + qa.z * kk.z + qa.w * kk.w;
      }
      P[i * L.pp + jj] = x * scale;
    }
    __syncthreads();
    for (int i = tid; i < me; i += kThreads) {
      float bm = -INFINITY;
      for (int jj = 0; jj < nb; ++jj) bm = fmaxf(bm, P[i * L.pp + jj]);
      const float old = rmax[i];
      const float nm = fmaxf(old, bm);
      const float a = (old == -INFINITY) ? 0.f : expf(old - nm);
      float zb = 0.f;
      for (int jj = 0; jj < nb; ++jj) {
        const float e = expf(P[i * L.pp + jj] - nm);
        P[i * L.pp + jj] = e;
        zb += e;
      }
      float nh, nl;
      comp_axpy(zhi[i], zlo[i], a, zb, 1.f, nh, nl);
      zhi[i] = nh;
      zlo[i] = nl;
      rmax[i] = nm;
      alpha[i] = a;
    }
    __syncthreads();
    for (int p = tid; p < me * cw; p += kThreads) {
      const int i = p / cw, c = p - i * cw;
      float part = 0.f;
      for (int jj = 0; jj < nb; ++jj) part = fmaf(P[i * L.pp + jj], vb[jj * kValTile + c], part);
      float nh, nl;
      comp_axpy(ahi[i * kValTile + c], alo[i * kValTile + c], alpha[i], part, 1.f, nh, nl);
      ahi[i * kValTile + c] = nh;
      alo[i * kValTile + c] = nl;
    }
    __syncthreads();
  }

  if (blockIdx.y == 0) {
    for (int i = tid; i < me; i += kThreads) {
      s.m_max[hb * m + i] = rmax[i];
      s.z_hat[hb * m + i] = zhi[i];
      s.z_lo[hb * m + i] = zlo[i];
    }
  }
  float* tdst = s.t_hat + hb * m * (int64_t)dv + c0;
  uint16_t* ldst = s.t_lo + hb * m * (int64_t)dv + c0;
  for (int p = tid; p < me * cw; p += kThreads) {
    const int i = p / cw, c = p - i * cw;
    tdst[(int64_t)i * dv + c] = ahi[i * kValTile + c];
    ldst[(int64_t)i * dv + c] = (uint16_t)(pack_bf16x2(alo[i * kValTile + c], 0.f) & 0xffffu);
  }
}

cudaError_t set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

}  // namespace

size_t seal_workspace_bytes_per_group(const DevState& s) {
  return (size_t)(1 + s.heads) * s.m * s.d * sizeof(double);
}

cudaError_t launch_seal(const DevState& s, int64_t g0, int64_t n, int t,
                        int m_eff, const float* q, const float* k,
                        const float* v, double* ws, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e;
  landmarks_kernel<<<dim3((unsigned)n, 1 + s.heads), kThreads, 0, stream>>>(
      s, g0, t, m_eff, q, k, v, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const size_t pbytes = pinv_smem_doubles(m_eff) * sizeof(double);
  if ((e = set_smem((const void*)pinv_kernel, pbytes)) != cudaSuccess) return e;
  pinv_kernel<<<(unsigned)(n * s.heads), kThreads, pbytes, stream>>>(s, g0, m_eff, ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const ReplaySmem R(m_eff, s.d);
  const size_t rbytes = (size_t)R.total * sizeof(float);
  if ((e = set_smem((const void*)replay_kernel, rbytes)) != cudaSuccess) return e;
  const unsigned tiles = (unsigned)((s.dv + kValTile - 1) / kValTile);
  replay_kernel<<<dim3((unsigned)(n * s.heads), tiles), kThreads, rbytes, stream>>>(
      s, g0, t, m_eff, k, v);
  return cudaGetLastError();
}

}  // namespace nys
