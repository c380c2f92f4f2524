// nys_seal_static: the seal without device allocation (see include/nys.h).
//
// The f64 landmark workspace lives in a file-scope device array instead of a
// cudaMallocAsync buffer.  Host code cannot use the array's name as a device
// address (on the host it names a shadow object), so the first call on each
// device looks the real address up with cudaGetSymbolAddress, with that
// device current, and caches it per device ordinal.
#include <algorithm>
#include <mutex>

#include "nys_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;  // 4 MiB, stated in nys.h
constexpr int kMaxDevices = 64;

static __device__ __align__(256) double g_seal_scratch[kScratchBytes / sizeof(double)];

std::mutex g_scratch_mu;
double* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_seal_scratch on the current device, or nullptr.
double* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_seal_scratch) != cudaSuccess || !p) {
      // Clear the runtime's sticky last error so that the next call of the
      // library (which checks cudaGetLastError after its launches) does not
      // report this failure as its own.
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<double*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int nys_seal_static(nys_states* st, int64_t g0, int64_t n, int32_t t,
                               const float* q, const float* k, const float* v,
                               void* stream) {
  // The same checks and mode choice as nys_seal, from the same function.
  nys::SealPlan plan;
  int rc = nys::plan_seal(st, g0, n, t, q, k, v, &plan);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Exact-only prompts copy the prompt into the state: no workspace at all.
  if (plan.exact) return nys::run_exact_seal(st, g0, n, t, k, v, s);
  const nys::DevState& ds = plan.ds;
  const size_t per = nys::seal_workspace_bytes_per_group(ds);
  if (per > kScratchBytes) return NYS_E_SCRATCH;
  if (n == 0) return NYS_OK;
  double* ws = scratch_address();
  if (!ws) return NYS_E_CUDA;
  // Each chunk's kernels finish reading the workspace before the next chunk's
  // first kernel overwrites it: all of them are ordered on `stream`.  Every
  // workspace element a kernel reads was written earlier in the same chunk,
  // so nothing left by a previous call is ever read.
  const int64_t chunk = std::min<int64_t>(n, (int64_t)(kScratchBytes / per));
  const int64_t H = ds.heads;
  for (int64_t a = 0; a < n; a += chunk) {
    const int64_t nb = std::min(chunk, n - a);
    if (nys::launch_seal(ds, g0 + a, nb, t, plan.m_eff, q + a * H * (int64_t)t * ds.d,
                         k + a * (int64_t)t * ds.d, v + a * (int64_t)t * ds.dv, ws, s) !=
        cudaSuccess)
      return NYS_E_CUDA;
  }
  nys::record_sealed(st, g0, n);
  return NYS_OK;
}
