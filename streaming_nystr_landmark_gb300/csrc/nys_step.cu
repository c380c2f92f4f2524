// Fused batched decode step of streaming Nystrom attention.
//
// One CTA advances one group (one (sequence, layer, KV head) state) by one
// token and writes all of its query heads' outputs.  The arithmetic follows
// nystrom.rs (docs.rs source view, cortiq-engine 0.5.71):
//   NystromState::advance     -- insert before any output; a full ring first
//                                evicts its oldest slot into every head;
//   NystromHead::far_insert   -- far logits of the evicted key, strict-greater
//                                running max with flash rescale, T^/Z^ update;
//   NystromHead::step         -- exact near logits over sinks + window, the
//                                landmark row with its own shift f, u = F^ M
//                                (Fm clamp), joint shift c_all, Aggregate
//                                guard, one division floored at 1e-30.
// State is fp32 as on the page; the far accumulators also carry a low part.
//
// Work split inside the CTA (8 warps):
//   A  every shared K-side row (sinks, window, key landmarks) is read once and
//      dotted with all heads of the tile; a warp owns a row, lanes own float4
//      columns, the dot is finished with a butterfly reduction.  The evicted
//      key is dotted with each head's query landmarks the same way.
//   B  one warp per head: far-insert scalars, maxima, mixing row u = F^ M,
//      gains, guard, near weights, denominator -- all O(m^2 + sink + w).
//   C  every V-side row (sinks, window) is read once and accumulated into all
//      heads; each head's T^ row is read, updated with the evicted value,
//      written back and accumulated in the same pass, so T^ crosses HBM once
//      each way.  Partial sums are reduced across warps in shared memory.
// T^ and Z^ are carried as hi + lo pairs (fp32 + bf16 / fp32) updated with
// exact FMA product errors and two-sum, so the decode's thousands of
// accumulations do not drift (plain f32 drifts ~1e-6 in T^ per thousand
// tokens, which the ill-conditioned mixing row amplifies into the output).
// The new key/value are written into the ring slot after every read of the
// old slot content (the page's ordering: absorb first, then overwrite).
#include <cfloat>
#include <cmath>

#include "nys_internal.h"

namespace nys {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kColTile = 128;  // value columns per pass: 32 lanes x float4

__host__ __device__ inline int round4(int x) { return (x + 3) & ~3; }

// Shared-memory carve-up in floats, identical on host and device.
struct StepSmem {
  int q, knew, kev, vnew, vev, sig, fh, lg, rs, es, gs, zs, ms, gl, zl, den, part;
  int total;
  int nrp, mp;
  __host__ __device__ StepSmem(int ht, int d, int dv, int near, int m) {
    nrp = round4(near);
    mp = round4(m);
    int o = 0;
    q = o;    o += ht * d;
    knew = o; o += d;
    kev = o;  o += d;
    vnew = o; o += dv;
    vev = o;  o += dv;
    sig = o;  o += ht * nrp;
    fh = o;   o += ht * mp;
    lg = o;   o += ht * mp;
    rs = o;   o += ht * mp;
    es = o;   o += ht * mp;
    gs = o;   o += ht * mp;
    zs = o;   o += ht * mp;
    ms = o;   o += ht * mp;
    gl = o;   o += ht * mp;  // low parts: u, then g (the far denominator's pairs)
    zl = o;   o += ht * mp;  // low part of Z^
    den = o;  o += round4(ht);
    part = o; o += kWarps * ht * kColTile;
    total = o;
  }
};

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

__device__ __forceinline__ float4 ld4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ void st4(float* p, float4 x) {
  *reinterpret_cast<float4*>(p) = x;
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

template <int HT>
__global__ void __launch_bounds__(kThreads)
step_kernel(DevState s, int64_t g0, const float* __restrict__ q,
            const float* __restrict__ k, const float* __restrict__ v,
            float* __restrict__ out) {
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t gi = blockIdx.x;  // row of this launch's inputs/outputs
  const int64_t g = g0 + gi;      // group in the state buffer
  const int d = s.d, dv = s.dv, w = s.w, ns = s.sink, H = s.heads, m = s.m;
  const int d4 = d >> 2, dv4 = dv >> 2;
  const float scale = s.scale;
  const StepSmem L(HT, d, dv, ns + w, m);
  float* sq = sm + L.q;
  float* knew = sm + L.knew;
  float* kev = sm + L.kev;
  float* vnew = sm + L.vnew;
  float* vev = sm + L.vev;
  float* sig = sm + L.sig;
  float* fh = sm + L.fh;
  float* lg = sm + L.lg;
  float* rs = sm + L.rs;
  float* es = sm + L.es;
  float* gs = sm + L.gs;
  float* zs = sm + L.zs;
  float* gls = sm + L.gl;
  float* zls = sm + L.zl;
  float* ms = sm + L.ms;
  float* den = sm + L.den;
  float* part = sm + L.part;

  int32_t* ints = s.ints + g * kIntsPerGroup;
  if (ints[kIntMode] == kModeExact) return;  // exact-only groups: nys_exact.cu
  const int win_head = ints[kIntWinHead];
  const int win_len = ints[kIntWinLen];
  const int m_eff = ints[kIntMEff];
  const bool full = (win_len == w);
  const int slot = full ? win_head : win_len;
  const int nwin = full ? w : win_len + 1;
  const int nnear = ns + nwin;

  const float* win_k = s.win_k + g * w * (int64_t)d;
  const float* win_v = s.win_v + g * w * (int64_t)dv;
  const float* sink_k = s.sink_k + g * ns * (int64_t)d;
  const float* sink_v = s.sink_v + g * ns * (int64_t)dv;
  const float* k_tilde = s.k_tilde + g * m * (int64_t)d;

  // The incoming key/value, and the outgoing ones before they are replaced.
  for (int c = tid; c < d4; c += kThreads) {
    st4(knew + 4 * c, ld4(k + gi * d + 4 * c));
    if (full) st4(kev + 4 * c, ld4(win_k + (int64_t)slot * d + 4 * c));
  }
  for (int c = tid; c < dv4; c += kThreads) {
    st4(vnew + 4 * c, ld4(v + gi * dv + 4 * c));
    if (full) st4(vev + 4 * c, ld4(win_v + (int64_t)slot * dv + 4 * c));
  }

  for (int h0 = 0; h0 < H; h0 += HT) {
    const int nh = min(HT, H - h0);
    for (int idx = tid; idx < HT * d4; idx += kThreads) {
      const int hh = idx / d4, c = idx - hh * d4;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (hh < nh) x = ld4(q + ((gi * H + h0 + hh) * (int64_t)d) + 4 * c);
      st4(sq + hh * d + 4 * c, x);
    }
    __syncthreads();

    // ---- A: shared K-side rows against every head of the tile.
    const int nrows = nnear + m_eff;
    for (int r = warp; r < nrows; r += kWarps) {
      const float* row;
      if (r < ns) {
        row = sink_k + (int64_t)r * d;
      } else if (r < nnear) {
        const int j = r - ns;
        row = (j == slot) ? knew : win_k + (int64_t)j * d;
      } else {
        row = k_tilde + (int64_t)(r - nnear) * d;
      }
      float acc[HT];
#pragma unroll
      for (int hh = 0; hh < HT; ++hh) acc[hh] = 0.f;
      for (int c = lane; c < d4; c += 32) {
        const float4 x = ld4(row + 4 * c);
#pragma unroll
        for (int hh = 0; hh < HT; ++hh) acc[hh] += dot4(x, ld4(sq + hh * d + 4 * c));
      }
#pragma unroll
      for (int hh = 0; hh < HT; ++hh) acc[hh] = warp_sum(acc[hh]);
      if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < HT; ++hh) {
          if (hh < nh) {
            const float l = acc[hh] * scale;
            if (r < nnear) sig[hh * L.nrp + r] = l;
            else fh[hh * L.mp + (r - nnear)] = l;
          }
        }
      }
    }
    // Far logits of the evicted key against each head's query landmarks.
    if (full) {
      for (int r = warp; r < nh * m_eff; r += kWarps) {
        const int hh = r / m_eff, i = r - hh * m_eff;
        const float* row =
            s.q_tilde + (((g * H + h0 + hh) * m + i) * (int64_t)d);
        float acc = 0.f;
        for (int c = lane; c < d4; c += 32) acc += dot4(ld4(row + 4 * c), ld4(kev + 4 * c));
        acc = warp_sum(acc);
        if (lane == 0) lg[hh * L.mp + i] = acc * scale;
      }
    }
    __syncthreads();

    // ---- B: per-head scalars, one warp per head.
    for (int hh = warp; hh < nh; hh += kWarps) {
      const int64_t hb = g * H + h0 + hh;
      float* zh = s.z_hat + hb * m;
      float* mx = s.m_max + hb * m;
      float* hfh = fh + hh * L.mp;
      float* hgs = gs + hh * L.mp;
      float* hzs = zs + hh * L.mp;
      float* hgl = gls + hh * L.mp;
      float* hzl = zls + hh * L.mp;
      float* hms = ms + hh * L.mp;
      float* hsig = sig + hh * L.nrp;
      const int32_t fl = s.far_len[hb];
      float* zl = s.z_lo + hb * m;
      for (int i = lane; i < m_eff; i += 32) {
        const float mo = mx[i], zo = zh[i], zlo = zl[i];
        float r = 1.f, e = 0.f, mn = mo, zn = zo, zln = zlo;
        if (full) {
          const float l = lg[hh * L.mp + i];
          if (l > mo) {
            r = expf(mo - l);
            mn = l;
          }
          e = expf(l - mn);
          comp_axpy(zo, zlo, r, e, 1.f, zn, zln);
          mx[i] = mn;
          zh[i] = zn;
          zl[i] = zln;
        }
        rs[hh * L.mp + i] = r;
        es[hh * L.mp + i] = e;
        hzs[i] = zn;  // Z^ as its pair, for the far denominator
        hzl[i] = zln;
        hms[i] = mn;
      }
      const int32_t fl_new = fl + (full ? 1 : 0);
      if (full && lane == 0) s.far_len[hb] = fl_new;
      __syncwarp();

      float c = -INFINITY;
      for (int j = lane; j < nnear; j += 32) c = fmaxf(c, hsig[j]);
      c = warp_max(c);
      float c_all = c, far_den = 0.f;
      if (fl_new > 0) {
        float f = -INFINITY;
        for (int a = lane; a < m_eff; a += 32) f = fmaxf(f, hfh[a]);
        f = warp_max(f);
        for (int a = lane; a < m_eff; a += 32) hfh[a] = expf(hfh[a] - f);
        __syncwarp();
        const float* M = s.mu + hb * m * (int64_t)m;
        float cm = -INFINITY;
        for (int b = lane; b < m_eff; b += 32) {
          float uh, ul;
          dot2_x4_pair(hfh, M + b, m, m_eff, uh, ul);
          if (s.rect == NYS_RECT_FM && uh < 0.f) uh = ul = 0.f;
          hgs[b] = uh;
          hgl[b] = ul;
          cm = fmaxf(cm, f + hms[b]);
        }
        c_all = fmaxf(c, warp_max(cm));
        // The far denominator in double-float (its terms cancel; see the
        // fast kernel): u as a pair, the exponent unrounded, Z^ as a pair.
        float dh = 0.f, dl = 0.f;
        for (int b = lane; b < m_eff; b += 32) {
          float eh, el, gh, glo, th, tl;
          exp_sum_pair(f, hms[b], c_all, eh, el);
          df_mul(hgs[b], hgl[b], eh, el, gh, glo);
          hgs[b] = gh;
          df_mul(gh, glo, hzs[b], hzl[b], th, tl);
          df_add(dh, dl, th, tl, dh, dl);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, dh, o);
          const float ol = __shfl_xor_sync(0xffffffffu, dl, o);
          df_add(dh, dl, oh, ol, dh, dl);
        }
        far_den = dh + dl;
        if (!(far_den >= 0.f)) {
          far_den = 0.f;
          for (int b = lane; b < m_eff; b += 32) hgs[b] = 0.f;
        }
      } else {
        for (int b = lane; b < m_eff; b += 32) hgs[b] = 0.f;
      }
      float psum = 0.f;
      for (int j = lane; j < nnear; j += 32) {
        const float p = expf(hsig[j] - c_all);
        hsig[j] = p;
        psum += p;
      }
      psum = warp_sum(psum);
      if (lane == 0) den[hh] = fmaxf(far_den + psum, 1e-30f);
    }
    __syncthreads();

    // ---- C: V-side rows and the far numerators, one column tile at a time.
    for (int ct = 0; ct < dv; ct += kColTile) {
      const int c4 = (ct >> 2) + lane;
      const bool cv = c4 < dv4;
      float4 acc[HT];
#pragma unroll
      for (int hh = 0; hh < HT; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = warp; r < nnear; r += kWarps) {
        const float* row;
        if (r < ns) {
          row = sink_v + (int64_t)r * dv;
        } else {
          const int j = r - ns;
          row = (j == slot) ? vnew : win_v + (int64_t)j * dv;
        }
        if (cv) {
          const float4 x = ld4(row + 4 * c4);
#pragma unroll
          for (int hh = 0; hh < HT; ++hh) {
            const float p = sig[hh * L.nrp + r];
            acc[hh].x = fmaf(p, x.x, acc[hh].x);
            acc[hh].y = fmaf(p, x.y, acc[hh].y);
            acc[hh].z = fmaf(p, x.z, acc[hh].z);
            acc[hh].w = fmaf(p, x.w, acc[hh].w);
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < HT; ++hh) {
        if (hh < nh) {
          const int64_t hb = g * H + h0 + hh;
          for (int b = warp; b < m_eff; b += kWarps) {
            float* trow = s.t_hat + (hb * m + b) * (int64_t)dv;
            uint2* lrow = reinterpret_cast<uint2*>(s.t_lo + (hb * m + b) * (int64_t)dv);
            if (cv) {
              float4 x = ld4(trow + 4 * c4);
              const uint2 lr = lrow[c4];
              float4 lo = make_float4(bf16_lo(lr.x), bf16_hi(lr.x), bf16_lo(lr.y), bf16_hi(lr.y));
              if (full) {
                const float r = rs[hh * L.mp + b], e = es[hh * L.mp + b];
                kahan_axpy4(x, lo, r, e, ld4(vev + 4 * c4));
                st4(trow + 4 * c4, x);
                uint2 lw;
                lw.x = pack_bf16x2(lo.x, lo.y);
                lw.y = pack_bf16x2(lo.z, lo.w);
                lrow[c4] = lw;
              }
              // High part only: the low part is under half an ulp of it.
              const float gb = gs[hh * L.mp + b];
              acc[hh].x = fmaf(gb, x.x, acc[hh].x);
              acc[hh].y = fmaf(gb, x.y, acc[hh].y);
              acc[hh].z = fmaf(gb, x.z, acc[hh].z);
              acc[hh].w = fmaf(gb, x.w, acc[hh].w);
            }
          }
        }
      }
      if (cv) {
#pragma unroll
        for (int hh = 0; hh < HT; ++hh)
          st4(part + (warp * HT + hh) * kColTile + 4 * lane, acc[hh]);
      }
      __syncthreads();
      for (int idx = tid; idx < nh * kColTile; idx += kThreads) {
        const int hh = idx / kColTile, col = idx - hh * kColTile;
        const int c = ct + col;
        if (c < dv) {
          float sum = 0.f;
#pragma unroll
          for (int wp = 0; wp < kWarps; ++wp) sum += part[(wp * HT + hh) * kColTile + col];
          out[(gi * H + h0 + hh) * (int64_t)dv + c] = sum / den[hh];
        }
      }
      __syncthreads();
    }
  }

  // Every read of the old slot is done: overwrite it and move the ring.
  float* wk = s.win_k + (g * w + slot) * (int64_t)d;
  float* wv = s.win_v + (g * w + slot) * (int64_t)dv;
  for (int c = tid; c < d4; c += kThreads) st4(wk + 4 * c, ld4(knew + 4 * c));
  for (int c = tid; c < dv4; c += kThreads) st4(wv + 4 * c, ld4(vnew + 4 * c));
  if (tid == 0) {
    if (full) ints[kIntWinHead] = (win_head + 1) % w;
    else ints[kIntWinLen] = win_len + 1;
  }
}

template <int HT>
cudaError_t launch_tile(const DevState& s, int64_t g0, int64_t n,
                        const float* q, const float* k, const float* v,
                        float* out, cudaStream_t stream) {
  const StepSmem L(HT, s.d, s.dv, s.sink + s.w, s.m);
  const size_t bytes = (size_t)L.total * sizeof(float);
  cudaError_t e = ensure_smem<step_kernel<HT>>(bytes);
  if (e != cudaSuccess) return e;
  step_kernel<HT><<<(unsigned)n, kThreads, bytes, stream>>>(s, g0, q, k, v, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step(const DevState& s, int64_t g0, int64_t n,
                        const float* q, const float* k, const float* v,
                        float* out, cudaStream_t stream, int debug_skip) {
  if (n <= 0) return cudaSuccess;
  // Geometries the persistent TMA kernel covers take it; the rest (H > 8,
  // dv > 128, rows that are not 16-byte multiples) run the kernel below.
  alignas(16) unsigned char plan[kPlanBytes];
  if (step_tma_plan_bytes() <= sizeof(plan) && plan_step_tma(s, plan))
    return launch_step_tma(s, plan, g0, n, q, k, v, out, stream, debug_skip);
  if (s.heads == 1) return launch_tile<1>(s, g0, n, q, k, v, out, stream);
  if (s.heads == 2) return launch_tile<2>(s, g0, n, q, k, v, out, stream);
  if (s.heads <= 4) return launch_tile<4>(s, g0, n, q, k, v, out, stream);
  return launch_tile<8>(s, g0, n, q, k, v, out, stream);
}

}  // namespace nys
