// Batched seal (prefill) of streaming Nystrom attention states.
//
// Follows nystrom.rs (docs.rs source view, cortiq-engine 0.5.71),
// NystromState::prefill_group, in three launches over all groups at once:
//
//  1. landmarks_kernel, grid (n, 1 + heads): block (g, 0) takes the group's
//     keys -- K~ = seg_means(k) (prefill_shared), sinks, ring fill, counters;
//     block (g, 1 + h) takes head h's queries -- Q~_h = seg_means(q_h)
//     (NystromHead::seal).  Segment i covers rows [i t / m_eff,
//     (i+1) t / m_eff); sums keep f64 accuracy (fn seg_means accumulates in
//     f64), computed in double-float.  The f64-accurate means go to a
//     workspace for step 2 as (hi, lo) pairs, their f32 roundings to the
//     state.
//  2. pinv_kernel, one block per (group, head): A = exp(Q~64 K~64^T * scale)
//     to f64 accuracy (double-float arithmetic), then
//     M = (A^T A + lambda I)^-1 A^T (fn ridge_pinv):
//     lambda = 1e-6 * max(mean diag(A^T A), DBL_MIN); a failed Cholesky
//     (pivot not > 0 or not finite, fn cholesky) multiplies lambda by ten, at
//     most twelve attempts, then M = I / max(mean diag, DBL_MIN).  The
//     Cholesky keeps the page's summation order.
//  3. replay_kernel (or, for long prompts, replay_tc_kernel in
//     nys_replay_tc.cu), one block per group and value tile for up to 64
//     landmark rows (several heads of a group; more heads take more blocks):
//     the replay of positions sink..t-1 through the ring leaves keys
//     sink..t-w-1 in the far field
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
// Knuth's two-sum: a + b = s + e exactly in f32.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Sum of 8 f32 values as hi + lo with hi = the f32 sum of a balanced tree and
// lo = the exact rounding errors of its seven additions (accumulated in f32,
// whose own rounding is ~2^-48 of the total).
__device__ __forceinline__ void sum8(const float (&x)[8], float& hi, float& lo) {
  float s01, e01, s23, e23, s45, e45, s67, e67, s03, e03, s47, e47;
  two_sum(x[0], x[1], s01, e01);
  two_sum(x[2], x[3], s23, e23);
  two_sum(x[4], x[5], s45, e45);
  two_sum(x[6], x[7], s67, e67);
  two_sum(s01, s23, s03, e03);
  two_sum(s45, s67, s47, e47);
  float e;
  two_sum(s03, s47, hi, e);
  lo = ((e01 + e23) + (e45 + e67)) + ((e03 + e47) + e);
}

// One block per (group, row source): y = 0 reads the group's keys (K~ plus
// sinks, ring and counters), y = 1 + h head h's queries (Q~_h).  One warp per
// landmark segment, lanes over float4 columns: no cross-warp reduction.  Rows
// are summed eight at a time exactly (sum8) and each such partial enters a
// double-float (hi, lo) accumulator; the mean is the pair divided by the
// segment length (exact remainder by FMA).  The segment means keep f64
// accuracy (~1e-14 of a sequential f64 sum) with no f64 operation: GB300's
// f64 rate, not HBM, bounded even one f64 addition per eight rows here.
__global__ void __launch_bounds__(kThreads)
landmarks_kernel(DevState s, int64_t g0, SealGeom sg,
                 const float* __restrict__ q, const float* __restrict__ k,
                 const float* __restrict__ v, double* __restrict__ ws) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t gi = blockIdx.x, g = g0 + gi;
  const int r = blockIdx.y;  // 0: keys, 1 + h: queries of head h
  const int d = s.d, dv = s.dv, H = s.heads, m = s.m, w = s.w, ns = s.sink;
  const int d4 = d >> 2, dv4 = dv >> 2;
  int t, m_eff;
  int64_t off;
  seal_geom(sg, gi, t, m_eff, off);

  const float* src;
  float* dst32;
  if (r == 0) {
    src = k + off * d;
    dst32 = s.k_tilde + g * m * (int64_t)d;
  } else {
    src = q + (off * H + (int64_t)(r - 1) * t) * d;
    dst32 = s.q_tilde + ((g * H + (r - 1)) * m) * (int64_t)d;
  }
  // The f64-accurate means go to the workspace as (hi, lo) pairs.
  float2* dst2 = reinterpret_cast<float2*>(ws) + (gi * (1 + H) + r) * (int64_t)m * d;

  for (int i = warp; i < m_eff; i += kWarps) {
    const int lo = (int)(((int64_t)i * t) / m_eff);
    const int hi = (int)(((int64_t)(i + 1) * t) / m_eff);
    const float nf = (float)(hi - lo);
    for (int c4 = lane; c4 < d4; c4 += 32) {
      const float* col = src + 4 * c4;
      float ah[4] = {0.f, 0.f, 0.f, 0.f}, al[4] = {0.f, 0.f, 0.f, 0.f};
      int j = lo;
      for (; j + 8 <= hi; j += 8) {
        float x[4][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 v4 = ld4(col + (int64_t)(j + u) * d);
          x[0][u] = v4.x;
          x[1][u] = v4.y;
          x[2][u] = v4.z;
          x[3][u] = v4.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float h, e;
          sum8(x[c], h, e);
          df_add(ah[c], al[c], h, e, ah[c], al[c]);
        }
      }
      for (; j < hi; ++j) {
        const float4 v4 = ld4(col + (int64_t)j * d);
        df_add(ah[0], al[0], v4.x, 0.f, ah[0], al[0]);
        df_add(ah[1], al[1], v4.y, 0.f, ah[1], al[1]);
        df_add(ah[2], al[2], v4.z, 0.f, ah[2], al[2]);
        df_add(ah[3], al[3], v4.w, 0.f, ah[3], al[3]);
      }
      // The mean as a pair: q = sum / n, the exact remainder by FMA.
      float2 mp[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float qh = ah[c] / nf;
        const float r = fmaf(-qh, nf, ah[c]) + al[c];
        float h, l;
        df_fast_two_sum(qh, r / nf, h, l);
        mp[c] = make_float2(h, l);
      }
      float2* o2 = dst2 + (int64_t)i * d + 4 * c4;
      o2[0] = mp[0];
      o2[1] = mp[1];
      o2[2] = mp[2];
      o2[3] = mp[3];
      float* o32 = dst32 + (int64_t)i * d + 4 * c4;
      st4(o32, make_float4(mp[0].x + mp[0].y, mp[1].x + mp[1].y, mp[2].x + mp[2].y,
                           mp[3].x + mp[3].y));
    }
  }

  if (r != 0) return;
  // Sinks: positions 0..sink, permanent (prefill_shared).
  const float* vsrc = v + off * dv;
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
    ints[kIntStatus] = 0;
  }
  for (int h = tid; h < H; h += kThreads) s.far_len[g * H + h] = t - ns - w;
}

// ---------------------------------------------------------------- 2
constexpr int kTile = 32;        // landmark-product column tile
constexpr int kTileStride = 36;  // row stride of the tiles (floats): 16-byte rows

// exp(xh + xl) as a double, |x| <= 700, in double-float arithmetic.
// Cody and Waite's range reduction x = k ln2 + r with ln2 split in three
// parts (the first has 12 significant bits, so k * ln2_hi is exact for
// |k| < 2^12; the parts were computed here to 200 bits), r folded back to a
// pair by exact two-sums, then the Taylor series of exp(r), |r| < 0.36, to
// degree 13 (truncation below 1e-17) by Horner's rule, and the factor 2^k
// applied in f64.  Measured against a 200-bit reference over |x| <= 40:
// within 5e-15 relative.
__device__ double df_exp(float xh, float xl) {
  constexpr float kLn2H = 0.693145751953125f;
  constexpr float kLn2L = 1.428606765330187e-06f;
  constexpr float kLn2LL = 5.497923148104107e-14f;
  const float k = rintf(xh * 1.4426950408889634f);
  float rh = xh - k * kLn2H;  // exact (Sterbenz)
  const float q = k * kLn2L;
  const float qe = fmaf(k, kLn2L, -q);
  float e1, e2;
  df_two_sum(rh, -q, rh, e1);
  df_two_sum(rh, xl, rh, e2);
  float rl = ((e1 + e2) - qe) - k * kLn2LL;
  df_fast_two_sum(rh, rl, rh, rl);
  // 1/n!, n = 0..13, as pairs hi + lo (computed here to 200 bits).
  constexpr float kFh[14] = {1.0f, 1.0f, 0.5f, 0.1666666716337204f, 0.0416666679084301f,
                             0.008333333767950535f, 0.0013888889225199819f,
                             0.00019841270113829523f, 2.4801587642286904e-05f,
                             2.7557318844628753e-06f, 2.755731998149713e-07f,
                             2.5052107943679403e-08f, 2.0876755879584152e-09f,
                             1.6059044372074283e-10f};
  constexpr float kFl[14] = {0.0f, 0.0f, 0.0f, -4.967053879312289e-09f, -1.2417634698280722e-09f,
                             -4.34617203337595e-10f, -3.3631094437103215e-11f,
                             -2.725596874933456e-12f, -3.40699609366682e-13f,
                             3.793571224297229e-14f, -7.575112209051195e-15f,
                             4.4176230446483665e-16f, 1.1082839147459852e-16f,
                             -5.352526511562726e-18f};
  float sh = kFh[13], sl = kFl[13];
#pragma unroll
  for (int n = 12; n >= 0; --n) {
    df_mul(sh, sl, rh, rl, sh, sl);
    df_add(sh, sl, kFh[n], kFl[n], sh, sl);
  }
  return ldexp((double)sh + (double)sl, (int)k);
}

// Shared memory of the pinv kernel: A (me x me doubles; later, transposed in
// place, the right-hand sides and the solution) and the lower triangle of the
// Cholesky region, packed row by row (me (me + 1) / 2 doubles); before A
// exists the same bytes hold the four logit tiles.  49 KB at m = 64, so four
// CTAs share an SM.
__host__ __device__ inline size_t pinv_smem_doubles(int me) {
  const size_t a = (size_t)me * me + (size_t)me * (me + 1) / 2;
  const size_t b = 2 * (size_t)me * kTileStride;
  return a > b ? a : b;
}
// Packed index of (i, j), j <= i, in a lower triangle stored row by row.
__device__ __forceinline__ int tri_idx(int i, int j) { return i * (i + 1) / 2 + j; }

template <int NT, int MM>
__global__ void __launch_bounds__(NT, 1024 / NT)
pinv_kernel(DevState s, int64_t g0, SealGeom sg, const double* __restrict__ ws) {
  extern __shared__ __align__(16) double dsm[];
  __shared__ int fail;
  __shared__ double lam_s, mean_diag_s;
  __shared__ double rdiag[MM];  // 1 / L_jj: one f64 division per column
  __shared__ double colj[MM];   // the current Cholesky column, L_ij for i > j
  const int tid = threadIdx.x;
  const int H = s.heads, m = s.m, d = s.d;
  const int64_t gi = blockIdx.x / H, g = g0 + gi;
  const int h = (int)(blockIdx.x - gi * H);
  int t_unused, me;
  int64_t off_unused;
  seal_geom(sg, gi, t_unused, me, off_unused);
  double* A = dsm;                          // [me][me]
  double* Lf = A + me * me;  // packed lower triangle: A^T A + lambda I -> Cholesky factor
  // Landmark tiles as f32 pairs x = hi + lo (exact to ~2^-48 of x), in the
  // bytes of A and Lf before either is written.
  float* Qh = reinterpret_cast<float*>(dsm);  // [me][kTileStride] each
  float* Ql = Qh + me * kTileStride;
  float* Kh = Ql + me * kTileStride;
  float* Kl = Kh + me * kTileStride;
  // The landmark means as (hi, lo) pairs (landmarks_kernel).
  const float2* K2 = reinterpret_cast<const float2*>(ws) + (gi * (1 + H)) * (int64_t)m * d;
  const float2* Q2 = reinterpret_cast<const float2*>(ws) + (gi * (1 + H) + 1 + h) * (int64_t)m * d;
  const double scale = (double)s.scale;

  // A[i][j] = exp((q~64_i . k~64_j) * scale).  The dot product runs in
  // double-float arithmetic on the fp32 pipe (GB300's f64 rate is a small
  // fraction of its f32 rate): hi*hi exactly by FMA two-product, the cross
  // terms hi*lo + lo*hi into its error, Knuth two-sum into an unevaluated
  // (sh, sl) pair.  Relative to sum|q_c k_c| the result is within ~1e-13 of
  // the f64 dot product; exp and everything after run in f64.
  // Thread tid < R*me (R = NT / me rows per pass) owns column
  // j = tid % me and rows i0 + p*R; key and query rows are read as float4
  // pairs (the query row is the same for the whole warp when me divides 256,
  // a broadcast).  Tile columns past d are zero and add exactly nothing.
  constexpr int kPer = (MM * MM + NT - 1) / NT;
  const int R = NT / me;
  const bool lact = tid < R * me;
  const int lj = lact ? tid % me : 0, li0 = lact ? tid / me : me;
  float sh[kPer], sl[kPer];
#pragma unroll
  for (int p = 0; p < kPer; ++p) {
    sh[p] = 0.f;
    sl[p] = 0.f;
  }
  for (int c0 = 0; c0 < d; c0 += kTile) {
    const int cw = min(kTile, d - c0);
    for (int idx = tid; idx < me * kTile; idx += NT) {
      const int i = idx / kTile, cc = idx - i * kTile;
      const float2 qv = cc < cw ? Q2[(int64_t)i * d + c0 + cc] : make_float2(0.f, 0.f);
      const float2 kv = cc < cw ? K2[(int64_t)i * d + c0 + cc] : make_float2(0.f, 0.f);
      Qh[i * kTileStride + cc] = qv.x;
      Ql[i * kTileStride + cc] = qv.y;
      Kh[i * kTileStride + cc] = kv.x;
      Kl[i * kTileStride + cc] = kv.y;
    }
    __syncthreads();
    if (lact) {
      const float4* kh4 = reinterpret_cast<const float4*>(Kh + lj * kTileStride);
      const float4* kl4 = reinterpret_cast<const float4*>(Kl + lj * kTileStride);
#pragma unroll
      for (int p = 0; p < kPer; ++p) {
        const int i = li0 + p * R;
        if (i < me) {
          const float4* qh4 = reinterpret_cast<const float4*>(Qh + i * kTileStride);
          const float4* ql4 = reinterpret_cast<const float4*>(Ql + i * kTileStride);
          float a = sh[p], b = sl[p];
          auto term = [&](float x, float xl, float y, float yl) {
            const float pr = x * y;
            float pe = fmaf(x, y, -pr);
            pe = fmaf(x, yl, fmaf(xl, y, pe));
            const float t = a + pr;
            const float z = t - a;
            b += ((a - (t - z)) + (pr - z)) + pe;
            a = t;
          };
#pragma unroll 2
          for (int c4 = 0; c4 < kTile / 4; ++c4) {
            const float4 qh = qh4[c4], ql = ql4[c4], kh = kh4[c4], kl = kl4[c4];
            term(qh.x, ql.x, kh.x, kl.x);
            term(qh.y, ql.y, kh.y, kl.y);
            term(qh.z, ql.z, kh.z, kl.z);
            term(qh.w, ql.w, kh.w, kl.w);
          }
          sh[p] = a;
          sl[p] = b;
        }
      }
    }
    __syncthreads();
  }
  float xmax = -INFINITY;
#pragma unroll
  for (int p = 0; p < kPer; ++p) {
    const int i = li0 + p * R;
    if (i < me) {
      // logit * scale as a pair (scale is an f32 value), exp in double-float;
      // non-finite or huge logits keep the f64 exp's semantics.
      float xh, xl;
      df_mul(sh[p], sl[p], (float)scale, 0.f, xh, xl);
      A[i * me + lj] = (fabsf(xh) <= 700.f) ? df_exp(xh, xl)
                                             : exp(((double)sh[p] + (double)sl[p]) * scale);
      xmax = (xh == xh) ? fmaxf(xmax, xh) : INFINITY;  // NaN: take the f64 path
    }
  }
  // A^T A in double-float on the fp32 pipe when every entry of A lies in
  // [e^-41, e^41] (about 2^-59 .. 2^59): its products then stay far inside
  // the f32 range and the pairs keep ~2^-48 of each value; A > 0, so no sum
  // cancels and each entry is within ~2^-47 of the f64 sum, the order of
  // that sum's own rounding.  Otherwise A^T A is summed in f64.  The logits
  // of the maximum bound A's maximum; the entries below it need no bound
  // (an entry under 2^-100 adds under 2^-200 m to an A^T A entry, far below
  // the ridge lambda, which is >= 1e-6 * max_i (A^T A)_ii / m).
  const bool below = __syncthreads_and(xmax <= 41.f), above = __syncthreads_or(xmax >= -41.f);
  const bool df_gram = below && above;
  float2* A2 = reinterpret_cast<float2*>(A);  // A as (hi, lo) pairs on that path
  if (df_gram) {
    for (int e = tid; e < me * me; e += NT) {
      const double a = A[e];  // read, then overwritten by its own pair
      A2[e] = make_float2((float)a, (float)(a - (double)(float)a));
    }
    __syncthreads();
  }

  // G = A^T A + lambda I into Lf, lower triangle only (all the Cholesky
  // reads), the triangle enumerated densely so that every lane has a pair.
  // G itself is not kept: a retry rebuilds it from A (same sums, same
  // order, so the same values).
  const int tri = me * (me + 1) / 2;
  auto build_gram = [&](double lam) {
    for (int p = tid; p < tri; p += NT) {
      int i = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);
      while (i * (i + 1) / 2 > p) --i;
      while ((i + 1) * (i + 2) / 2 <= p) ++i;
      const int j = p - i * (i + 1) / 2;
      double a;
      if (df_gram) {
        float gh = 0.f, gl = 0.f;
        for (int kk = 0; kk < me; ++kk) {
          const float2 x = A2[kk * me + i], y = A2[kk * me + j];
          const float pr = x.x * y.x;
          float pe = fmaf(x.x, y.x, -pr);
          pe = fmaf(x.x, y.y, fmaf(x.y, y.x, pe));
          const float t = gh + pr;
          const float z = t - gh;
          gl += ((gh - (t - z)) + (pr - z)) + pe;
          gh = t;
        }
        a = (double)gh + (double)gl;
      } else {
        a = 0.0;
        for (int kk = 0; kk < me; ++kk) a = fma(A[kk * me + i], A[kk * me + j], a);
      }
      Lf[p] = (i == j) ? a + lam : a;  // p = tri_idx(i, j)
    }
  };
  build_gram(0.0);
  __syncthreads();
  if (tid == 0) {
    double sd = 0.0;
    for (int i = 0; i < me; ++i) sd += Lf[tri_idx(i, i)];
    mean_diag_s = sd / (double)me;
    lam_s = 1e-6 * fmax(mean_diag_s, DBL_MIN);
  }
  __syncthreads();

  bool solved = false;
  for (int attempt = 0; attempt < 12 && !solved; ++attempt) {
    const double lam = lam_s;
    if (attempt == 0) {
      for (int i = tid; i < me; i += NT) Lf[tri_idx(i, i)] += lam;
    } else {
      build_gram(lam);
    }
    if (tid == 0) fail = 0;
    __syncthreads();
    // Right-looking form of the page's Cholesky: before column j, the lower
    // triangle right of it holds G - sum_{k<j} L_.k L_.k^T with each product
    // subtracted in the order k = 0, 1, ... -- the same operations in the
    // same order as the page's left-looking loop, so the same values, but
    // each column is one parallel update instead of j-term serial sums.
    // The scaled column is also copied to colj, so the update reads it
    // without bank conflicts.  The lane that updates the next diagonal entry
    // (j+1, j+1) takes its square root and reciprocal right after, so a
    // column costs two barriers.
    const int cwp = tid >> 5, cln = tid & 31;
    auto pivot = [&](int j, double sp) {  // L_jj = sqrt(sp), or fail
      if (!(sp > 0.0) || !isfinite(sp)) {
        fail = 1;
      } else {
        Lf[tri_idx(j, j)] = sqrt(sp);
        rdiag[j] = 1.0 / Lf[tri_idx(j, j)];
      }
    };
    if (tid == 0) pivot(0, Lf[0]);
    __syncthreads();
    for (int j = 0; j < me; ++j) {
      if (fail) break;
      for (int i = j + 1 + tid; i < me; i += NT) {
        const double lij = Lf[tri_idx(i, j)] * rdiag[j];
        Lf[tri_idx(i, j)] = lij;
        colj[i] = lij;
      }
      __syncthreads();
      for (int a = j + 1 + cwp; a < me; a += NT / 32) {
        const double laj = colj[a];
        double* row = Lf + tri_idx(a, 0);
        for (int b = j + 1 + cln; b <= a; b += 32) {
          row[b] -= laj * colj[b];
          if (b == j + 1 && a == j + 1) pivot(j + 1, row[b]);
        }
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
    // G M = A^T by forward (L Y = A^T) then backward (L^T M = Y)
    // substitution, column-oriented over all threads and in double-float
    // arithmetic (the f64 pipe is the bottleneck), in place: at pivot k
    // every thread reads row k, scales it by 1/L_kk itself, and updates its
    // own (i, j) entries; row k keeps its unscaled value until a scaling
    // pass.  Pair arrays: L in place of Lf, the right-hand sides in place of
    // A (transposed there).
    float2* L2 = reinterpret_cast<float2*>(Lf);
    float2* W = reinterpret_cast<float2*>(A);
    __shared__ float2 rd2[MM];
    __syncthreads();
    for (int e = tid; e < tri; e += NT) {
      const double l = Lf[e];  // read, then overwritten by its own pair
      L2[e] = make_float2((float)l, (float)(l - (double)(float)l));
    }
    for (int e = tid; e < me * me; e += NT) {
      const int i = e / me, j = e - i * me;
      if (df_gram) {  // A is already in pairs: W = A^T by swapping them
        if (i < j) {
          const float2 aij = A2[i * me + j], aji = A2[j * me + i];
          W[i * me + j] = aji;
          W[j * me + i] = aij;
        }
      } else if (i <= j) {  // W[i][j] = A^T[i][j] = A[j][i]: swap the pair (i, j), (j, i)
        const double aij = A[i * me + j], aji = A[j * me + i];
        W[i * me + j] = make_float2((float)aji, (float)(aji - (double)(float)aji));
        W[j * me + i] = make_float2((float)aij, (float)(aij - (double)(float)aij));
      }
    }
    for (int k = tid; k < me; k += NT) {
      const double r = rdiag[k];
      rd2[k] = make_float2((float)r, (float)(r - (double)(float)r));
    }
    __syncthreads();
    // Thread (warp, lane) owns rows warp, warp + 8, ... and columns lane,
    // lane + 32 (no divisions in the pivot loops).
    const int wrp = tid >> 5, lan = tid & 31;
    auto scaled = [&](int k, int j, float& h, float& l) {  // W_kj / L_kk
      const float2 w = W[k * me + j];
      df_mul(w.x, w.y, rd2[k].x, rd2[k].y, h, l);
    };
    auto update = [&](int i, int j, float2 lik, float yh, float yl) {  // W_ij -= l * y
      const float2 w = W[i * me + j];
      float ph, pl, nh, nl;
      df_mul(lik.x, lik.y, yh, yl, ph, pl);
      df_add(w.x, w.y, -ph, -pl, nh, nl);
      W[i * me + j] = make_float2(nh, nl);
    };
    // y = W_kj / L_kk once per pivot and column: row k is final at pivot k.
    constexpr int kCols = (MM + 31) / 32;
    float yh[kCols], yl[kCols];
    auto pivot_row = [&](int k) {
#pragma unroll
      for (int c = 0; c < kCols; ++c)
        if (lan + 32 * c < me) scaled(k, lan + 32 * c, yh[c], yl[c]);
    };
    constexpr int kPinvWarps = NT / 32;
    // Two pivots per barrier: every thread also forms, for its own columns,
    // the second pivot row's value after the first pivot's update (t, with
    // the same operations as `update`) and its scaled value; rows past both
    // pivots then take both updates in order, and the second pivot row's
    // owner stores t after the barrier (no one reads that row again before
    // the next pass, which follows a barrier).
    float y2h[kCols], y2l[kCols], t2h[kCols], t2l[kCols];
    auto second_pivot = [&](int k2, float2 l) {  // row k2 after the update by pivot y
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        const int j = lan + 32 * c;
        if (j < me) {
          const float2 w = W[k2 * me + j];
          float ph, pl;
          df_mul(l.x, l.y, yh[c], yl[c], ph, pl);
          df_add(w.x, w.y, -ph, -pl, t2h[c], t2l[c]);
          df_mul(t2h[c], t2l[c], rd2[k2].x, rd2[k2].y, y2h[c], y2l[c]);
        }
      }
    };
    auto store_second = [&](int k2) {
      if (k2 % kPinvWarps == wrp) {
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (lan + 32 * c < me) W[k2 * me + lan + 32 * c] = make_float2(t2h[c], t2l[c]);
      }
    };
    int k = 0;
    for (; k + 1 < me - 1; k += 2) {  // forward: rows below the pivots
      pivot_row(k);
      second_pivot(k + 1, L2[tri_idx(k + 1, k)]);
      const int i0 = wrp > k + 1 ? wrp : wrp + ((k + 1 - wrp) / kPinvWarps + 1) * kPinvWarps;
      for (int i = i0; i < me; i += kPinvWarps) {
        const float2 l0 = L2[tri_idx(i, k)], l1 = L2[tri_idx(i, k + 1)];
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (lan + 32 * c < me) {
            update(i, lan + 32 * c, l0, yh[c], yl[c]);
            update(i, lan + 32 * c, l1, y2h[c], y2l[c]);
          }
      }
      __syncthreads();
      store_second(k + 1);
    }
    for (; k < me - 1; ++k) {  // the last pivot, when the count is odd
      pivot_row(k);
      const int i0 = wrp > k ? wrp : wrp + ((k - wrp) / kPinvWarps + 1) * kPinvWarps;
      for (int i = i0; i < me; i += kPinvWarps) {
        const float2 lik = L2[tri_idx(i, k)];
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (lan + 32 * c < me) update(i, lan + 32 * c, lik, yh[c], yl[c]);
      }
      __syncthreads();
    }
    __syncthreads();
    for (int i = wrp; i < me; i += kPinvWarps)  // Y = W / diag(L)
      for (int j = lan; j < me; j += 32) {
        float h, l;
        scaled(i, j, h, l);
        W[i * me + j] = make_float2(h, l);
      }
    __syncthreads();
    for (k = me - 1; k - 1 > 0; k -= 2) {  // backward: rows above the pivots
      pivot_row(k);
      second_pivot(k - 1, L2[tri_idx(k, k - 1)]);  // (L^T)_{k-1,k} = L_{k,k-1}
      for (int i = wrp; i < k - 1; i += kPinvWarps) {
        const float2 l0 = L2[tri_idx(k, i)], l1 = L2[tri_idx(k - 1, i)];  // (L^T)_ik = L_ki
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (lan + 32 * c < me) {
            update(i, lan + 32 * c, l0, yh[c], yl[c]);
            update(i, lan + 32 * c, l1, y2h[c], y2l[c]);
          }
      }
      __syncthreads();
      store_second(k - 1);
    }
    for (; k > 0; --k) {  // the last pivot, when the count is odd
      pivot_row(k);
      for (int i = wrp; i < k; i += kPinvWarps) {
        const float2 lki = L2[tri_idx(k, i)];  // (L^T)_ik = L_ki
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (lan + 32 * c < me) update(i, lan + 32 * c, lki, yh[c], yl[c]);
      }
      __syncthreads();
    }
    __syncthreads();
    for (int pair = tid; pair < me * me; pair += NT) {  // M = W / diag(L)
      const int i = pair / me, j = pair - i * me;
      float h, l;
      scaled(i, j, h, l);
      M[i * m + j] = h + l;
    }
  } else {
    const double diag = 1.0 / fmax(mean_diag_s, DBL_MIN);
    for (int pair = tid; pair < me * me; pair += NT) {
      const int i = pair / me, j = pair - i * me;
      M[i * m + j] = (i == j) ? (float)diag : 0.f;
    }
  }
}

// ---------------------------------------------------------------- 3
// One block per (group, head, 128-column value tile): 16 x 16 threads, thread
// (ty, tx) owns landmark rows ty*TR .. ty*TR+TR-1.  Keys are consumed in
// blocks of kKeyBlock = 64:
//   logits  L[TR][4] for keys tx*4..tx*4+3 from Q~^T and K^T in shared memory
//           (one float4 of each feeds 4*TR FMAs);
//   online  per-row block maximum over the 16 lanes of the row group, new
//   max     running maximum, rescale alpha = exp(old - new), p = exp(L - max);
//   values  the block's p (row-major in the key tile's shared memory, one
//           float4 store per row) times the value tile: part[TR][8] for
//           columns tx*4..tx*4+3 and 64+tx*4..64+tx*4+3 (both float4 reads of
//           a value row are contiguous over the 16 lanes: no bank conflicts);
//   fold    (hi, lo) <- (hi, lo) * alpha + part, compensated (kahan_axpy), so
//           that tens of thousands of keys do not accumulate f32 rounding.
constexpr int kKeyBlock = 64;
constexpr int kValTile = 128;
constexpr int kKtStride = kKeyBlock + 4;  // 68: conflict-free transposed stores
constexpr int kPtStride = kKeyBlock + 4;  // p rows, 16-byte aligned

// The key tile and, after the logits, the probability tile share one region.
__host__ __device__ inline size_t replay_kt_floats(int rt, int d) {
  const size_t a = (size_t)d * kKtStride, b = (size_t)rt * kPtStride;
  return a > b ? a : b;
}
__host__ __device__ inline size_t replay_smem_floats(int rt, int d) {
  return (size_t)d * (rt + 4) + replay_kt_floats(rt, d) + (size_t)kKeyBlock * kValTile;
}

template <int TR>
__device__ __forceinline__ void load_rows(const float* p, float (&a)[TR]) {
  if constexpr (TR == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
  } else if constexpr (TR == 2) {
    const float2 x = *reinterpret_cast<const float2*>(p);
    a[0] = x.x; a[1] = x.y;
  } else {
    a[0] = p[0];
  }
}

template <int TR>
__global__ void __launch_bounds__(kThreads, 2)
replay_kernel(DevState s, int64_t g0, SealGeom sg,
              const float* __restrict__ k, const float* __restrict__ v, int skip_long,
              int heads_per_cta, int ctas_per_group) {
  constexpr int RT = 16 * TR;
  extern __shared__ __align__(16) float fsm[];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int H = s.heads, m = s.m, d = s.d, dv = s.dv, w = s.w, ns = s.sink;
  const int d4 = d >> 2;
  // Rows of this CTA: landmark r % m of head h0 + r / m (several heads of a
  // group share the key and value blocks).
  const int64_t gi = blockIdx.x / ctas_per_group, g = g0 + gi;
  const int h0 = (int)(blockIdx.x - gi * ctas_per_group) * heads_per_cta;
  int t, me;
  int64_t off;
  seal_geom(sg, gi, t, me, off);
  if (skip_long && t - w - ns >= kReplayTcMinKeys) return;  // the tensor-core replay's
  const int c0 = blockIdx.y * kValTile;
  const int cw = min(kValTile, dv - c0);
  const float scale = s.scale;
  constexpr int QTS = RT + 4;          // row stride of QT: conflict-free transposed stores
  float* QT = fsm;                     // [d][QTS]  Q~ transposed, unused rows zero
  float* KT = QT + (size_t)d * QTS;    // [d][kKtStride]  key block transposed
  float* PT = KT;                      // [RT][kPtStride] p, after the logits
  float* VB = KT + replay_kt_floats(RT, d);  // [kKeyBlock][kValTile]

  // Q~ rows, transposed, moved like the key blocks below: thread
  // (klane, kchunk) takes float4 chunks kchunk, kchunk + 16, ... of rows
  // klane, klane + 16, ...; all of a thread's loads are issued before its
  // stores.
  const int klane = tid & 15, kchunk = tid >> 4;  // 16 rows x 16 chunk lanes
  {
    float4 qx[TR][2];
#pragma unroll
    for (int a = 0; a < TR; ++a) {
      const int i = klane + 16 * a;
      const int hh = h0 + i / m, li = i - (i / m) * m;
      const bool used = i < heads_per_cta * m && hh < H && li < me;
      const float* src = s.q_tilde + ((g * H + hh) * (int64_t)m + li) * d;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int c4 = kchunk + 16 * b;
        qx[a][b] = (used && c4 < d4) ? ld4(src + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int c4 = kchunk + 32; c4 < d4; c4 += 16) {  // d > 128
        const float4 x = used ? ld4(src + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        QT[(4 * c4 + 0) * QTS + i] = x.x;
        QT[(4 * c4 + 1) * QTS + i] = x.y;
        QT[(4 * c4 + 2) * QTS + i] = x.z;
        QT[(4 * c4 + 3) * QTS + i] = x.w;
      }
    }
#pragma unroll
    for (int a = 0; a < TR; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int i = klane + 16 * a, c4 = kchunk + 16 * b;
        if (c4 < d4) {
          QT[(4 * c4 + 0) * QTS + i] = qx[a][b].x;
          QT[(4 * c4 + 1) * QTS + i] = qx[a][b].y;
          QT[(4 * c4 + 2) * QTS + i] = qx[a][b].z;
          QT[(4 * c4 + 3) * QTS + i] = qx[a][b].w;
        }
      }
  }

  float hi[TR][8], lo[TR][8], mrow[TR], zh[TR], zl[TR];
#pragma unroll
  for (int i = 0; i < TR; ++i) {
    mrow[i] = -INFINITY;
    zh[i] = 0.f;
    zl[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      hi[i][c] = 0.f;
      lo[i][c] = 0.f;
    }
  }

  const float* ksrc = k + off * d;
  const float* vsrc = v + off * dv + c0;
  const int j_end = t - w;  // keys sink .. t-w-1 were evicted by the replay
  for (int j0 = ns; j0 < j_end; j0 += kKeyBlock) {
    const int nb = min(kKeyBlock, j_end - j0);
    __syncthreads();  // the previous block is done with KT / PT / VB
    // Keys, transposed: thread (klane, kchunk) moves float4 chunks
    // kchunk, kchunk + 16, ... of keys klane, klane + 16, ...; values of
    // this column tile (rows past the block are zero).  A thread loads its
    // key chunks (the first two of each row), then its value chunks, each
    // set before any of its stores.
    {
      constexpr int kKR = kKeyBlock / 16;                  // key rows per thread
      constexpr int kVR = kKeyBlock * (kValTile / 4) / kThreads;  // value chunks per thread
      const int cw4 = cw >> 2;
#pragma unroll
      for (int a0 = 0; a0 < kKR; a0 += 2) {  // two key rows' chunks in flight
        float4 kx[2][2];
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const int kk = klane + 16 * (a0 + a);
          const float* row = ksrc + (int64_t)(j0 + kk) * d;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int c4 = kchunk + 16 * b;
            kx[a][b] =
                (kk < nb && c4 < d4) ? ld4(row + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          const int kk = klane + 16 * (a0 + a);
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int c4 = kchunk + 16 * b;
            if (c4 < d4) {
              KT[(4 * c4 + 0) * kKtStride + kk] = kx[a][b].x;
              KT[(4 * c4 + 1) * kKtStride + kk] = kx[a][b].y;
              KT[(4 * c4 + 2) * kKtStride + kk] = kx[a][b].z;
              KT[(4 * c4 + 3) * kKtStride + kk] = kx[a][b].w;
            }
          }
          const float* row = ksrc + (int64_t)(j0 + kk) * d;
          for (int c4 = kchunk + 32; c4 < d4; c4 += 16) {  // d > 128
            const float4 x = kk < nb ? ld4(row + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
            KT[(4 * c4 + 0) * kKtStride + kk] = x.x;
            KT[(4 * c4 + 1) * kKtStride + kk] = x.y;
            KT[(4 * c4 + 2) * kKtStride + kk] = x.z;
            KT[(4 * c4 + 3) * kKtStride + kk] = x.w;
          }
        }
      }
#pragma unroll
      for (int e0 = 0; e0 < kVR; e0 += 4) {  // four value chunks in flight
        float4 vx[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int idx = tid + (e0 + e) * kThreads, jj = idx >> 5, c4 = idx & 31;
          vx[e] = (jj < nb && c4 < cw4) ? ld4(vsrc + (int64_t)(j0 + jj) * dv + 4 * c4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int idx = tid + (e0 + e) * kThreads, jj = idx >> 5, c4 = idx & 31;
          *reinterpret_cast<float4*>(VB + jj * kValTile + 4 * c4) = vx[e];
        }
      }
    }
    __syncthreads();

    float L[TR][4];
#pragma unroll
    for (int i = 0; i < TR; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) L[i][j] = 0.f;
#pragma unroll 4
    for (int c = 0; c < d; ++c) {
      float a[TR];
      load_rows<TR>(QT + c * QTS + ty * TR, a);
      const float4 b = *reinterpret_cast<const float4*>(KT + c * kKtStride + tx * 4);
#pragma unroll
      for (int i = 0; i < TR; ++i) {
        L[i][0] = fmaf(a[i], b.x, L[i][0]);
        L[i][1] = fmaf(a[i], b.y, L[i][1]);
        L[i][2] = fmaf(a[i], b.z, L[i][2]);
        L[i][3] = fmaf(a[i], b.w, L[i][3]);
      }
    }
    float alpha[TR];
#pragma unroll
    for (int i = 0; i < TR; ++i) {
      float bm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        L[i][j] = (tx * 4 + j < nb) ? L[i][j] * scale : -INFINITY;
        bm = fmaxf(bm, L[i][j]);
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
      const float nm = fmaxf(mrow[i], bm);
      alpha[i] = (mrow[i] == -INFINITY) ? 0.f : expf(mrow[i] - nm);
      mrow[i] = nm;
      float zb = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        L[i][j] = (tx * 4 + j < nb) ? expf(L[i][j] - nm) : 0.f;
        zb += L[i][j];
      }
#pragma unroll
      for (int o = 8; o; o >>= 1) zb += __shfl_xor_sync(0xffffffffu, zb, o);
      float nh, nl;
      comp_axpy(zh[i], zl[i], alpha[i], zb, 1.f, nh, nl);
      zh[i] = nh;
      zl[i] = nl;
    }
    __syncthreads();  // every thread is done reading KT: p takes its place
#pragma unroll
    for (int i = 0; i < TR; ++i)
      *reinterpret_cast<float4*>(PT + (ty * TR + i) * kPtStride + tx * 4) =
          make_float4(L[i][0], L[i][1], L[i][2], L[i][3]);
    __syncthreads();

    float part[TR][8];
#pragma unroll
    for (int i = 0; i < TR; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) part[i][c] = 0.f;
    // One key of the value contraction: p of this thread's rows times the
    // key's two value chunks.
    auto pv_key = [&](const float (&a)[TR], int jj) {
      const float* vr = VB + jj * kValTile + tx * 4;
      const float4 b0 = *reinterpret_cast<const float4*>(vr);
      const float4 b1 = *reinterpret_cast<const float4*>(vr + kValTile / 2);
#pragma unroll
      for (int i = 0; i < TR; ++i) {
        part[i][0] = fmaf(a[i], b0.x, part[i][0]);
        part[i][1] = fmaf(a[i], b0.y, part[i][1]);
        part[i][2] = fmaf(a[i], b0.z, part[i][2]);
        part[i][3] = fmaf(a[i], b0.w, part[i][3]);
        part[i][4] = fmaf(a[i], b1.x, part[i][4]);
        part[i][5] = fmaf(a[i], b1.y, part[i][5]);
        part[i][6] = fmaf(a[i], b1.z, part[i][6]);
        part[i][7] = fmaf(a[i], b1.w, part[i][7]);
      }
    };
    for (int jj = 0; jj < kKeyBlock; jj += 4) {
      // p of four consecutive keys for each row: one broadcast float4 each.
      float ax[TR], ay[TR], az[TR], aw[TR];
#pragma unroll
      for (int i = 0; i < TR; ++i) {
        const float4 t4 = *reinterpret_cast<const float4*>(PT + (ty * TR + i) * kPtStride + jj);
        ax[i] = t4.x;
        ay[i] = t4.y;
        az[i] = t4.z;
        aw[i] = t4.w;
      }
      pv_key(ax, jj);
      pv_key(ay, jj + 1);
      pv_key(az, jj + 2);
      pv_key(aw, jj + 3);
    }
#pragma unroll
    for (int i = 0; i < TR; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        kahan_axpy(hi[i][c], lo[i][c], alpha[i], part[i][c], 1.f);
      }
  }

#pragma unroll
  for (int i = 0; i < TR; ++i) {
    const int row = ty * TR + i;
    const int hh = h0 + row / m, li = row - (row / m) * m;
    if (row >= heads_per_cta * m || hh >= H || li >= me) continue;
    const int64_t grow = (g * H + hh) * (int64_t)m + li;
    if (blockIdx.y == 0 && tx == 0) {
      s.m_max[grow] = mrow[i];
      s.z_hat[grow] = zh[i];
      s.z_lo[grow] = zl[i];
    }
    float* tdst = s.t_hat + grow * (int64_t)dv + c0;
    uint16_t* ldst = s.t_lo + grow * (int64_t)dv + c0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int col = (c < 4 ? 0 : kValTile / 2 - 4) + tx * 4 + c;
      if (col < cw) {
        tdst[col] = hi[i][c];
        ldst[col] = (uint16_t)(pack_bf16x2(lo[i][c], 0.f) & 0xffffu);
      }
    }
  }
}

// Heads of a group per CUDA-core replay CTA: as many as fit in 64 landmark
// rows (the key and value blocks are loaded once for all of them).
inline int replay_heads_per_cta(const DevState& s) {
  const int fit = 64 / s.m;
  return fit < 1 ? 1 : (fit < s.heads ? fit : s.heads);
}

template <int TR>
cudaError_t launch_replay(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                          const float* k, const float* v, int skip_long, cudaStream_t stream) {
  const size_t bytes = replay_smem_floats(16 * TR, s.d) * sizeof(float);
  cudaError_t e = ensure_smem<replay_kernel<TR>>(bytes);
  if (e != cudaSuccess) return e;
  const unsigned tiles = (unsigned)((s.dv + kValTile - 1) / kValTile);
  const int hpc = replay_heads_per_cta(s);
  const int cpg = (s.heads + hpc - 1) / hpc;
  replay_kernel<TR><<<dim3((unsigned)(n * cpg), tiles), kThreads, bytes, stream>>>(
      s, g0, sg, k, v, skip_long, hpc, cpg);
  return cudaGetLastError();
}

}  // namespace

size_t seal_workspace_bytes_per_group(const DevState& s) {
  return (size_t)(1 + s.heads) * s.m * s.d * sizeof(double);
}

namespace {

cudaError_t launch_pinv(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg, int max_me,
                        double* ws, cudaStream_t stream) {
  // Up to 32 landmarks: 128-thread CTAs, eight per SM, so that the serial
  // steps of one head's Cholesky overlap with more heads' parallel work.
  cudaError_t e;
  const size_t pbytes = pinv_smem_doubles(max_me) * sizeof(double);
  if (max_me <= 32) {
    if ((e = ensure_smem<pinv_kernel<128, 32>>(pbytes)) != cudaSuccess) return e;
    pinv_kernel<128, 32><<<(unsigned)(n * s.heads), 128, pbytes, stream>>>(s, g0, sg, ws);
  } else {
    if ((e = ensure_smem<pinv_kernel<kThreads, kMaxM>>(pbytes)) != cudaSuccess) return e;
    pinv_kernel<kThreads, kMaxM><<<(unsigned)(n * s.heads), kThreads, pbytes, stream>>>(
        s, g0, sg, ws);
  }
  return cudaGetLastError();
}

// Replay: tensor cores for groups with long prompts (where the geometry
// fits), CUDA cores for the rest.  A uniform batch launches only the path
// its prompt length takes; a ragged one launches both, and each skips the
// other's groups.
cudaError_t launch_replays(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                           const float* k, const float* v, cudaStream_t stream,
                           int debug_stall) {
  cudaError_t e;
  const bool tc = replay_tc_fits(s);
  const bool uniform = sg.t_arr == nullptr;
  const bool long_prompt = sg.t - s.w - s.sink >= kReplayTcMinKeys;
  if (tc && (!uniform || long_prompt)) {
    if ((e = launch_replay_tc(s, g0, n, sg, k, v, stream, debug_stall)) != cudaSuccess) return e;
    if (uniform) return cudaSuccess;
  }
  const int skip_long = tc ? 1 : 0;
  const int rows = replay_heads_per_cta(s) * s.m;  // landmark rows per CTA
  if (rows <= 16) return launch_replay<1>(s, g0, n, sg, k, v, skip_long, stream);
  if (rows <= 32) return launch_replay<2>(s, g0, n, sg, k, v, skip_long, stream);
  return launch_replay<4>(s, g0, n, sg, k, v, skip_long, stream);
}

}  // namespace

cudaError_t launch_seal_geom(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                             int max_me, const float* q, const float* k, const float* v,
                             double* ws, cudaStream_t stream, int debug_stall,
                             const SealFork& fork) {
  if (n <= 0) return cudaSuccess;
  cudaError_t e;
  landmarks_kernel<<<dim3((unsigned)n, 1 + s.heads), kThreads, 0, stream>>>(s, g0, sg, q, k, v,
                                                                            ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!fork.on()) {
    if ((e = launch_pinv(s, g0, n, sg, max_me, ws, stream)) != cudaSuccess) return e;
    return launch_replays(s, g0, n, sg, k, v, stream, debug_stall);
  }
  // The pinv on the side stream, the replay on the caller's; both follow
  // the landmarks, and the caller's stream waits for the pinv before the
  // next chunk's landmarks overwrite the workspace it reads.
  if ((e = cudaEventRecord(fork.forked, stream)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(fork.side, fork.forked, 0)) != cudaSuccess) return e;
  const cudaError_t ep = launch_pinv(s, g0, n, sg, max_me, ws, fork.side);
  const cudaError_t ej = cudaEventRecord(fork.joined, fork.side);
  const cudaError_t er = launch_replays(s, g0, n, sg, k, v, stream, debug_stall);
  const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(stream, fork.joined, 0) : ej;
  if (ep != cudaSuccess) return ep;
  if (er != cudaSuccess) return er;
  return ew;
}

cudaError_t launch_seal(const DevState& s, int64_t g0, int64_t n, int t,
                        int m_eff, const float* q, const float* k,
                        const float* v, double* ws, cudaStream_t stream, int debug_stall,
                        const SealFork& fork) {
  const SealGeom sg{t, m_eff, nullptr, nullptr, nullptr};
  return launch_seal_geom(s, g0, n, sg, m_eff, q, k, v, ws, stream, debug_stall, fork);
}

}  // namespace nys
