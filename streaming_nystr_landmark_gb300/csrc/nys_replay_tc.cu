// Seal replay on the tensor cores (tcgen05): the far-field fold of every
// prompt key that the window evicted, from cortiq_engine's nystrom.rs
// (docs.rs source view), `prefill_group`: for each landmark row i of each
// head and every evicted key j (positions sink .. t-w-1, in order)
//   s_ij = (Q~_i . k_j) / sqrt(d),   running max m_i with flash rescale,
//   T^_i = sum_j exp(s_ij - m_i) v_j,  Z^_i = sum_j exp(s_ij - m_i).
// The page does this one key at a time; here a block of 64 keys at once.
//
// Precision: both contractions (Q~ K^T and P V) take fp32 operands split
// into three bf16 pieces, x = x0 + x1 + x2 (each piece the rounded remainder
// of the previous ones, so x is represented to ~2^-24), and sum the six
// products x0y0 + x0y1 + x1y0 + x0y2 + x1y1 + x2y0 in fp32 in tensor memory.
// The dropped products are below 2^-23 of |x y|, about the rounding of an
// fp32 product.  Each 64-key block's P V starts from zero and is folded into
// compensated (hi, lo) accumulators with the block's rescale, as in the
// CUDA-core replay, so the length of the prompt adds no fp32 drift.
//
// One CTA of 256 threads per (group, up to 128 landmark rows = 128 / m
// heads).  Per key block:
//   1. the K block is in three bf16 planes [key][d] (the K-major no-swizzle
//      layout the MMA reads: 8x8 core matrices of 128 B), split by
//      warpgroup 1 from the registers it loaded during the previous block;
//   2. one thread: S = Q~ K^T as 6 * d/16 MMAs (M=128, N=64) into TMEM,
//      while all threads split the V block into three planes of V^T
//      [dv][key];
//   3. warpgroup 0 (thread = row): S row from TMEM, logits, block max, new
//      running max, rescale alpha, p = exp(s - m), Z^ fold, p split into
//      three planes [row][key] in the K block's shared memory;
//   4. one thread: O = P V as 6 * 4 MMAs (M=128, N=dv) into TMEM;
//   5. warpgroup 0 (thread = row): (hi, lo) <- (hi, lo) * alpha + O
//      (Kahan-compensated) on every column, with hi and lo kept in TMEM,
//      while warpgroup 1 splits the next K block into the key planes.
// Every wait on an MMA is bounded (2 s of %globaltimer); a timeout sets the
// group's status word and the CTA stops, frees its tensor memory and
// returns.
#include <cuda_bf16.h>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kTcThreads = 256;
constexpr int kTcRows = 128;     // MMA M: landmark rows per CTA
constexpr int kTcKeys = 64;      // keys per block (S MMA N, P V MMA K)
constexpr int kTcCols = 512;     // tensor memory columns allocated
constexpr int kColS = 0;         // S: kTcKeys columns
constexpr int kColO = 128;       // O: dv columns
constexpr int kColHi = 256;      // hi: dv columns
constexpr int kColLo = 384;      // lo: dv columns
constexpr uint64_t kTcWaitNs = 2000000000ull;
constexpr uint32_t kTcSuspendNs = 100000;  // a waiting thread sleeps up to 0.1 ms per try

__device__ __forceinline__ uint32_t tc_sptr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Byte offset of element (r, k) in an R x K bf16 operand, K-major, no
// swizzle: 8-row x 16-byte core matrices; core matrices adjacent in K are
// 128 B apart (leading byte offset), 8-row groups K*2*8 B apart (stride
// byte offset).
__device__ __forceinline__ uint32_t tc_off(int r, int k, int K) {
  return (uint32_t)((r >> 3) * (K * 16) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
// Shared-memory matrix descriptor: start, leading and stride byte offsets
// (all >> 4), descriptor version 1 (bits 46-47), no swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor, kind::f16: f32 accumulate, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t tc_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          tc_sptr(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_proxy_fence() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&x)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const float (&x)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])), "r"(__float_as_uint(x[2])),
      "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])), "r"(__float_as_uint(x[5])),
      "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7])), "r"(__float_as_uint(x[8])),
      "r"(__float_as_uint(x[9])), "r"(__float_as_uint(x[10])), "r"(__float_as_uint(x[11])),
      "r"(__float_as_uint(x[12])), "r"(__float_as_uint(x[13])), "r"(__float_as_uint(x[14])),
      "r"(__float_as_uint(x[15]))
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bounded wait for phase `parity` of an mbarrier; false after 2 s or when
// another thread of the CTA already gave up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(tc_sptr(bar)), "r"(parity), "r"(kTcSuspendNs)
        : "memory");
    if (ok) return true;
    if ((i & 15u) == 15u) {
      if (*abort) return false;
      uint64_t t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      if (t1 - t0 > kTcWaitNs) return false;
    }
  }
}

// Eight consecutive K elements -> one 16-byte chunk in each of three bf16
// planes: x = x0 + x1 + x2, each piece the round-to-nearest of what the
// previous ones left (the remainders are exact in fp32).  Pairs are rounded
// and packed by one cvt.rn.bf16x2 and unpacked by bit operations.
__device__ __forceinline__ void store_split8(unsigned char* p0, unsigned char* p1,
                                             unsigned char* p2, uint32_t off,
                                             const float (&x)[8]) {
  uint32_t w0[4], w1[4], w2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = x[2 * i], b = x[2 * i + 1];
    w0[i] = pack_bf16x2(a, b);
    const float ra = a - bf16_lo(w0[i]), rb = b - bf16_hi(w0[i]);
    w1[i] = pack_bf16x2(ra, rb);
    w2[i] = pack_bf16x2(ra - bf16_lo(w1[i]), rb - bf16_hi(w1[i]));
  }
  *reinterpret_cast<uint4*>(p0 + off) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  *reinterpret_cast<uint4*>(p1 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *reinterpret_cast<uint4*>(p2 + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
}

// Task t of a row-block split (8 rows x 32 elements per 32-lane warp task):
// a quarter-warp takes eight consecutive rows of one 8-element chunk, so its
// 16-byte stores cover all 32 banks, and each row's global reads are 128
// contiguous bytes.
__device__ __forceinline__ void split_task(int t, int ngc, int& r, int& c8) {
  const int wt = t >> 5, l = t & 31;
  const int rg = wt / ngc, cg = wt - rg * ngc;
  r = rg * 8 + (l & 7);
  c8 = (cg * 4 + (l >> 3)) * 8;
}
__device__ __forceinline__ void load8(const float* src, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  const float4 b = *reinterpret_cast<const float4*>(src + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void zero8(float (&x)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = 0.f;
}

// The six split products, largest first: (piece of the left operand, piece
// of the right operand).
__device__ __constant__ int kPairA[6] = {0, 0, 1, 0, 1, 2};
__device__ __constant__ int kPairB[6] = {0, 1, 0, 2, 1, 0};

__global__ void __launch_bounds__(kTcThreads, 1)
replay_tc_kernel(DevState s, int64_t g0, SealGeom sg, const float* __restrict__ k,
                 const float* __restrict__ v, int heads_per_cta, int ctas_per_group,
                 int debug_stall) {
  extern __shared__ __align__(1024) unsigned char tsm[];
  __shared__ __align__(8) uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float alpha_s[kTcRows];

  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = s.heads, m = s.m, d = s.d, dv = s.dv, w = s.w, ns = s.sink;
  const int64_t gi = blockIdx.x / ctas_per_group, g = g0 + gi;
  const int h0 = (int)(blockIdx.x - gi * ctas_per_group) * heads_per_cta;
  int t, me;
  int64_t off;
  seal_geom(sg, gi, t, me, off);
  if (t - w - ns < kReplayTcMinKeys) return;  // a short prompt: the CUDA-core replay's

  const size_t qplane = (size_t)kTcRows * d * 2;
  const size_t kplane = (size_t)(kTcKeys * d > kTcRows * kTcKeys ? kTcKeys * d
                                                                  : kTcRows * kTcKeys) * 2;
  const size_t vplane = (size_t)dv * kTcKeys * 2;
  unsigned char* Qp[3] = {tsm, tsm + qplane, tsm + 2 * qplane};
  unsigned char* Kp[3] = {tsm + 3 * qplane, tsm + 3 * qplane + kplane,
                          tsm + 3 * qplane + 2 * kplane};
  unsigned char* Vp[3] = {Kp[0] + 3 * kplane, Kp[0] + 3 * kplane + vplane,
                          Kp[0] + 3 * kplane + 2 * vplane};
  unsigned char* const* Pp = Kp;  // p takes the key planes once S is done

  // Landmark row r of this CTA: head h0 + r / m, landmark r % m.
  const float scale = s.scale;
  const int ngc = d >> 5;  // groups of four 8-element chunks per row
  for (int task = tid; task < kTcRows * (d >> 3); task += kTcThreads) {
    int r, c8;
    split_task(task, ngc, r, c8);
    const int hh = h0 + r / m, i = r - (r / m) * m;
    float x[8];
    if (r < heads_per_cta * m && hh < H && i < me)
      load8(s.q_tilde + ((g * H + hh) * (int64_t)m + i) * d + c8, x);
    else
      zero8(x);
    store_split8(Qp[0], Qp[1], Qp[2], tc_off(r, c8, d), x);
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_sptr(&bar_s)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_sptr(&bar_o)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     tc_sptr(&tmem_slot)),
                 "r"(kTcCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // This thread's tensor-memory lane (its landmark row) and column half.
  const int row = tid & (kTcRows - 1);
  const int half = tid >> 7;  // 0: warps 0-3, 1: warps 4-7
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const int cols_half = dv >> 1;  // a multiple of 16; processed 16 at a time
  {
    float z[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] = 0.f;
    for (int c = half * cols_half; c < (half + 1) * cols_half; c += 16) {
      tc_st16(lane_base + kColHi + c, z);
      tc_st16(lane_base + kColLo + c, z);
    }
    tc_wait_st();
  }

  float mrow = -INFINITY, zh = 0.f, zl = 0.f;  // warpgroup 0: this row's max and Z^
  const float* ksrc = k + off * d;
  const float* vsrc = v + off * dv;
  const int j_end = t - w;  // keys sink .. t-w-1 were evicted by the replay
  const uint32_t id_s = tc_idesc(kTcRows, kTcKeys), id_o = tc_idesc(kTcRows, dv);
  volatile int* vabort = &abort_flag;
  uint32_t parity = 0;
  bool ok = true;

  // Warpgroup 1 prefetches the next key block into registers while
  // warpgroup 0 runs the softmax: kKPre tasks of 8 keys' chunks per thread.
  constexpr int kKPre = kTcKeys * 128 / 8 / (kTcThreads / 2);  // d <= 128
  float kpre[kKPre][8];
  const int ktasks = kTcKeys * (d >> 3);
  auto k_load = [&](int jb, int nbb, int t0, int tstep, float (&buf)[kKPre][8], int ntask) {
#pragma unroll
    for (int it = 0; it < kKPre; ++it) {
      const int task = t0 + it * tstep;
      if (it < ntask && task < ktasks) {
        int kk, c8;
        split_task(task, ngc, kk, c8);
        if (kk < nbb) load8(ksrc + (int64_t)(jb + kk) * d + c8, buf[it]);
        else zero8(buf[it]);
      }
    }
  };
  auto k_store = [&](int t0, int tstep, const float (&buf)[kKPre][8], int ntask) {
#pragma unroll
    for (int it = 0; it < kKPre; ++it) {
      const int task = t0 + it * tstep;
      if (it < ntask && task < ktasks) {
        int kk, c8;
        split_task(task, ngc, kk, c8);
        store_split8(Kp[0], Kp[1], Kp[2], tc_off(kk, c8, d), buf[it]);
      }
    }
  };
  // The first key block: every thread loads and splits its share.
  if (ns < j_end) {
    const int nb0 = min(kTcKeys, j_end - ns);
    k_load(ns, nb0, tid, kTcThreads, kpre, kKPre / 2);
    k_store(tid, kTcThreads, kpre, kKPre / 2);
  }

  for (int j0 = ns; j0 < j_end && ok; j0 += kTcKeys, parity ^= 1u) {
    const int nb = min(kTcKeys, j_end - j0);
    const bool more = j0 + kTcKeys < j_end;
    // 1. the key block is in its planes (first block above; later ones from
    //    warpgroup 1's prefetch at the end of the previous block).
    tc_proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // 2. S = Q~ K^T, issued by one thread ...  (test hook: the first CTA
    //    withholds its first block's MMAs, so its waits run out)
    if (tid == 0 && !(debug_stall && blockIdx.x == 0 && j0 == ns)) {
      uint32_t acc = 0;
      for (int ks = 0; ks < (d >> 4); ++ks)
        for (int pr = 0; pr < 6; ++pr) {
          tc_mma(tmem + kColS, tc_desc(tc_sptr(Qp[kPairA[pr]]) + ks * 256, d * 16),
                 tc_desc(tc_sptr(Kp[kPairB[pr]]) + ks * 256, d * 16), id_s, acc);
          acc = 1;
        }
      tc_commit(&bar_s);
    }
    // ... while every thread moves the value block into its planes (the
    // previous block's P V is complete).
    {
      // Task: one value column x eight keys; consecutive lanes take
      // consecutive columns (128-byte loads, conflict-free V^T stores).
      float vx[4][8];
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int task = tid + it * kTcThreads;
        if (task < dv * (kTcKeys >> 3)) {
          const int col = task % dv, k8 = (task / dv) * 8;
#pragma unroll
          for (int jx = 0; jx < 8; ++jx)
            vx[it][jx] = (k8 + jx < nb) ? vsrc[(int64_t)(j0 + k8 + jx) * dv + col] : 0.f;
        }
      }
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int task = tid + it * kTcThreads;
        if (task < dv * (kTcKeys >> 3)) {
          const int col = task % dv, k8 = (task / dv) * 8;
          store_split8(Vp[0], Vp[1], Vp[2], tc_off(col, k8, kTcKeys), vx[it]);
        }
      }
    }
    // (ok is made warp-uniform: the tensor-memory loads below are
    // warp-collective.)
    ok = __all_sync(0xffffffffu, tc_wait(&bar_s, parity, vabort));
    if (!ok) abort_flag = 1;
    tc_fence_after();
    if (half == 1 && ok && more) {
      // 3'. warpgroup 1: next key block -> registers.
      k_load(j0 + kTcKeys, min(kTcKeys, j_end - j0 - kTcKeys), tid - kTcThreads / 2,
             kTcThreads / 2, kpre, kKPre);
    }
    // 3. online softmax of this block, warpgroup 0 (thread = row).
    if (ok && half == 0) {
      float sv[kTcKeys];
#pragma unroll
      for (int c = 0; c < kTcKeys; c += 16) {
        float x[16];
        tc_ld16(lane_base + kColS + c, x);
#pragma unroll
        for (int jx = 0; jx < 16; ++jx) sv[c + jx] = x[jx];
      }
      float bm = -INFINITY;
#pragma unroll
      for (int jx = 0; jx < kTcKeys; ++jx) {
        sv[jx] = (jx < nb) ? sv[jx] * scale : -INFINITY;
        bm = fmaxf(bm, sv[jx]);
      }
      const float nm = fmaxf(mrow, bm);
      // Every exponent is <= 0 and the running sum always holds a term of 1
      // (the key that set the maximum), so the fast exponential (__expf:
      // about 2 ulp near 0, its error growing with |x| only where e^x is far
      // below the sum's rounding) keeps the sums to fp32 accuracy.
      const float alpha = (mrow == -INFINITY) ? 0.f : __expf(mrow - nm);
      mrow = nm;
      float zb = 0.f;
#pragma unroll
      for (int jx = 0; jx < kTcKeys; ++jx) {
        sv[jx] = (jx < nb) ? __expf(sv[jx] - nm) : 0.f;
        zb += sv[jx];
      }
      float nh, nl;
      comp_axpy(zh, zl, alpha, zb, 1.f, nh, nl);
      zh = nh;
      zl = nl;
      alpha_s[row] = alpha;
#pragma unroll
      for (int c = 0; c < kTcKeys; c += 8) {
        float x[8];
#pragma unroll
        for (int jx = 0; jx < 8; ++jx) x[jx] = sv[c + jx];
        store_split8(Pp[0], Pp[1], Pp[2], tc_off(row, c, kTcKeys), x);
      }
    }
    tc_proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*vabort) break;
    // 4. O = P V (fresh each block).
    if (tid == 0) {
      uint32_t acc = 0;
      for (int ks = 0; ks < (kTcKeys >> 4); ++ks)
        for (int pr = 0; pr < 6; ++pr) {
          tc_mma(tmem + kColO, tc_desc(tc_sptr(Pp[kPairA[pr]]) + ks * 256, kTcKeys * 16),
                 tc_desc(tc_sptr(Vp[kPairB[pr]]) + ks * 256, kTcKeys * 16), id_o, acc);
          acc = 1;
        }
      tc_commit(&bar_o);
    }
    ok = __all_sync(0xffffffffu, tc_wait(&bar_o, parity, vabort));
    if (!ok) abort_flag = 1;
    tc_fence_after();
    // 5. warpgroup 0: (hi, lo) <- (hi, lo) * alpha + O on every column of
    //    its row, while
    // 1'. warpgroup 1 splits the prefetched key block into the key planes
    //     (the P V that read them as p is complete).
    if (ok && half == 0) {
      const float alpha = alpha_s[row];
      for (int c = 0; c < dv; c += 16) {
        float o[16], hi[16], lo[16];
        tc_ld16(lane_base + kColO + c, o);
        tc_ld16(lane_base + kColHi + c, hi);
        tc_ld16(lane_base + kColLo + c, lo);
#pragma unroll
        for (int jx = 0; jx < 16; ++jx) kahan_axpy(hi[jx], lo[jx], alpha, o[jx], 1.f);
        tc_st16(lane_base + kColHi + c, hi);
        tc_st16(lane_base + kColLo + c, lo);
      }
      tc_wait_st();
    }
    if (half == 1 && ok && more) k_store(tid - kTcThreads / 2, kTcThreads / 2, kpre, kKPre);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*vabort) break;
  }

  if (*vabort) {
    if (tid == 0) s.ints[g * kIntsPerGroup + kIntStatus] = 3;  // replay gave up
  } else {
    // Write this CTA's rows of T^ (hi f32, lo bf16) and Z^, running maxima.
    const int hh = h0 + row / m, i = row - (row / m) * m;
    const bool valid = row < heads_per_cta * m && hh < H && i < me;
    const int64_t grow = (g * H + hh) * (int64_t)m + i;
    for (int c = half * cols_half; c < (half + 1) * cols_half; c += 16) {
      float hi[16], lo[16];
      tc_ld16(lane_base + kColHi + c, hi);
      tc_ld16(lane_base + kColLo + c, lo);
      if (valid) {
#pragma unroll
        for (int jx = 0; jx < 16; ++jx) {
          s.t_hat[grow * dv + c + jx] = hi[jx];
          s.t_lo[grow * dv + c + jx] = (uint16_t)(pack_bf16x2(lo[jx], 0.f) & 0xffffu);
        }
      }
    }
    if (valid && half == 0) {
      s.m_max[grow] = mrow;
      s.z_hat[grow] = zh;
      s.z_lo[grow] = zl;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTcCols));
}

size_t replay_tc_smem(int d, int dv) {
  const size_t qplane = (size_t)kTcRows * d * 2;
  const size_t kk = (size_t)kTcKeys * d, pp = (size_t)kTcRows * kTcKeys;
  const size_t kplane = (kk > pp ? kk : pp) * 2;
  const size_t vplane = (size_t)dv * kTcKeys * 2;
  return 3 * (qplane + kplane + vplane);
}

}  // namespace

bool replay_tc_fits(const DevState& s) {
  return s.m >= 32 && s.m <= kTcRows && s.d % 32 == 0 && s.dv % 32 == 0 && s.d <= 128 &&
         s.dv <= 128 && replay_tc_smem(s.d, s.dv) <= 200 * 1024;
}

cudaError_t launch_replay_tc(const DevState& s, int64_t g0, int64_t n, const SealGeom& sg,
                             const float* k, const float* v, cudaStream_t stream,
                             int debug_stall) {
  if (n <= 0) return cudaSuccess;
  const int heads_per_cta = kTcRows / s.m < s.heads ? kTcRows / s.m : s.heads;
  const int ctas_per_group = (s.heads + heads_per_cta - 1) / heads_per_cta;
  const size_t bytes = replay_tc_smem(s.d, s.dv);
  cudaError_t e = ensure_smem<replay_tc_kernel>(bytes);
  if (e != cudaSuccess) return e;
  replay_tc_kernel<<<(unsigned)(n * ctas_per_group), kTcThreads, bytes, stream>>>(
      s, g0, sg, k, v, heads_per_cta, ctas_per_group, debug_stall);
  return cudaGetLastError();
}

}  // namespace nys
