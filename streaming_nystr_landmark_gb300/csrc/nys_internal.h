// Internal declarations shared by the libnys translation units: the device
// view of a state buffer and the kernel launchers.  Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "nys.h"

namespace nys {

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
  kIntsPerGroup = 8
};
enum : int { kModeEmpty = 0, kModeSealed = 1 };

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
  int32_t* far_len;
  int32_t* ints;
  int32_t m, w, sink, heads, d, dv, rect;
  float scale;  // 1/sqrt(d) evaluated in f32
};

// One decode token for groups [g0, g0+n): one kernel launch on `stream`.
cudaError_t launch_step(const DevState& s, int64_t g0, int64_t n,
                        const float* q, const float* k, const float* v,
                        float* out, cudaStream_t stream);

// Bytes of f64 workspace the seal needs per group (key landmarks and every
// head's query landmarks before rounding).
size_t seal_workspace_bytes_per_group(const DevState& s);

// Seal groups [g0, g0+n) with prompt length t and m_eff landmarks, using
// `ws` (seal_workspace_bytes_per_group * n bytes) as f64 scratch.  Three
// kernel launches on `stream`.
cudaError_t launch_seal(const DevState& s, int64_t g0, int64_t n, int t,
                        int m_eff, const float* q, const float* k,
                        const float* v, double* ws, cudaStream_t stream);

}  // namespace nys
