// One attention layer's O(1) override for a batch of sequences: the
// lifecycle of Struct LayerKvCache (docs.rs, cortiq-engine 0.5.71), methods
// o1_begin, o1_push_q, o1_sealed, o1_seal, o1_step, o1_views and
// o1_memory_bytes, over the batched group states of this library.
//
//  begin   arm query collection: a device trace of max_prompt positions for
//          every (sequence, query head);
//  push_q  record one position's queries of every sequence (one strided copy);
//  seal    if the page's preconditions hold -- a full query trace, a GQA
//          fan-out that divides, densely stored KV rows (f32 by this API) --
//          build one state per (sequence, KV head) with nys_seal and release
//          the trace; otherwise report "not sealed" and keep everything, so
//          the caller's layer stays exact;
//  step    one decode token for every (sequence, KV group): head h of a
//          sequence belongs to group h / (num_heads / num_kv_heads).
// Host code only: every operation on the data runs in the library's kernels
// or in CUDA copies.
#include <cstring>
#include <new>

#include "nys_internal.h"

struct nys_o1 {
  nys_config cfg;   // heads_per_kv is filled in at seal time
  int32_t batch, num_heads, num_kv_heads, max_prompt;
  int32_t pushed;   // positions recorded so far
  float* trace;     // [batch][num_heads][max_prompt][d], null once sealed
  nys_states* states;
};

extern "C" {

int nys_o1_begin(const nys_config* cfg, int32_t batch, int32_t num_heads,
                 int32_t num_kv_heads, int32_t max_prompt, nys_o1** out) {
  if (!cfg || !out || batch < 1 || num_heads < 1 || num_kv_heads < 1 || max_prompt < 1)
    return NYS_E_INVAL;
  *out = nullptr;
  nys_config c = *cfg;
  c.heads_per_kv = 1;  // validated here with a placeholder; fixed at seal
  size_t probe = 0;
  int rc = nys_memory_bytes(&c, 1, &probe);
  if (rc) return rc;
  nys_o1* o = new (std::nothrow) nys_o1();
  if (!o) return NYS_E_INVAL;
  o->cfg = *cfg;
  o->batch = batch;
  o->num_heads = num_heads;
  o->num_kv_heads = num_kv_heads;
  o->max_prompt = max_prompt;
  o->pushed = 0;
  o->states = nullptr;
  const size_t bytes = (size_t)batch * num_heads * max_prompt * cfg->d * sizeof(float);
  if (cudaMalloc(&o->trace, bytes) != cudaSuccess) {
    delete o;
    return NYS_E_CUDA;
  }
  *out = o;
  return NYS_OK;
}

int nys_o1_push_q(nys_o1* o, const float* q_all, void* stream) {
  if (!o || !q_all) return NYS_E_INVAL;
  if (!o->trace) return NYS_OK;  // not collecting (already sealed): a no-op, as on the page
  if (o->pushed >= o->max_prompt) return NYS_E_RANGE;
  const size_t row = (size_t)o->cfg.d * sizeof(float);
  // q_all [batch][num_heads][d] -> trace[b][h][pushed][:]
  if (cudaMemcpy2DAsync(o->trace + (size_t)o->pushed * o->cfg.d, (size_t)o->max_prompt * row,
                        q_all, row, row, (size_t)o->batch * o->num_heads,
                        cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return NYS_E_CUDA;
  ++o->pushed;
  return NYS_OK;
}

int nys_o1_seal(nys_o1* o, const float* k, const float* v, int32_t kv_len, int32_t kv_dense,
                void* stream, int32_t* sealed) {
  if (!o || !sealed || !k || !v) return NYS_E_INVAL;
  *sealed = 0;
  if (o->states) {
    *sealed = 1;
    return NYS_OK;
  }
  const nys_config& c0 = o->cfg;
  // Preconditions of o1_seal: a GQA fan-out that divides, densely stored KV,
  // a full query trace.  Failing any keeps the layer exact.
  if (o->num_heads % o->num_kv_heads != 0 || !kv_dense || kv_len < 1 || o->pushed != kv_len)
    return NYS_OK;
  // A short prompt takes the exact-only mode, which needs the exact region.
  if ((int64_t)kv_len <= (int64_t)c0.w + c0.sink + 8 && c0.exact_cap < kv_len) return NYS_OK;
  nys_config c = c0;
  c.heads_per_kv = o->num_heads / o->num_kv_heads;
  const int64_t groups = (int64_t)o->batch * o->num_kv_heads;
  nys_states* st = nullptr;
  int rc = nys_alloc_states(&c, groups, nullptr, 0, &st);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Compact the trace to [batch][num_heads][kv_len][d] = [groups][hpk][t][d].
  const size_t row = (size_t)c.d * sizeof(float);
  void* q = nullptr;
  if (cudaMallocAsync(&q, (size_t)o->batch * o->num_heads * kv_len * row, s) != cudaSuccess) {
    nys_free_states(st);
    return NYS_E_CUDA;
  }
  if (cudaMemcpy2DAsync(q, (size_t)kv_len * row, o->trace, (size_t)o->max_prompt * row,
                        (size_t)kv_len * row, (size_t)o->batch * o->num_heads,
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    cudaFreeAsync(q, s);
    nys_free_states(st);
    return NYS_E_CUDA;
  }
  rc = nys_seal(st, 0, groups, kv_len, static_cast<const float*>(q), k, v, stream);
  const cudaError_t fe = cudaFreeAsync(q, s);
  if (rc || fe != cudaSuccess) {
    nys_free_states(st);
    return rc ? rc : NYS_E_CUDA;
  }
  // The trace is no longer needed once the seal's reads are done.
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    nys_free_states(st);
    return NYS_E_CUDA;
  }
  cudaFree(o->trace);
  o->trace = nullptr;
  o->states = st;
  *sealed = 1;
  return NYS_OK;
}

int nys_o1_sealed(const nys_o1* o, int32_t* sealed) {
  if (!o || !sealed) return NYS_E_INVAL;
  *sealed = o->states != nullptr;
  return NYS_OK;
}

int nys_o1_step(nys_o1* o, const float* q_all, const float* k_new, const float* v_new,
                float* out, void* stream) {
  if (!o) return NYS_E_INVAL;
  if (!o->states) return NYS_E_NOT_SEALED;
  return nys_step_batch(o->states, 0, (int64_t)o->batch * o->num_kv_heads, q_all, k_new, v_new,
                        out, stream);
}

int nys_o1_memory_bytes(const nys_o1* o, size_t* bytes) {
  if (!o || !bytes) return NYS_E_INVAL;
  if (o->states) {
    nys_config c;
    int64_t g = 0;
    nys_config_of(o->states, &c, &g);
    return nys_memory_bytes(&c, g, bytes);
  }
  *bytes = (size_t)o->batch * o->num_heads * o->pushed * o->cfg.d * sizeof(float);
  return NYS_OK;
}

int nys_o1_states(const nys_o1* o, nys_states** st) {
  if (!o || !st) return NYS_E_INVAL;
  *st = o->states;
  return o->states ? NYS_OK : NYS_E_NOT_SEALED;
}

int nys_o1_free(nys_o1* o) {
  if (!o) return NYS_OK;
  int rc = NYS_OK;
  if (o->trace && cudaFree(o->trace) != cudaSuccess) rc = NYS_E_CUDA;
  if (o->states) {
    const int r2 = nys_free_states(o->states);
    if (r2) rc = r2;
  }
  delete o;
  return rc;
}

}  // extern "C"
