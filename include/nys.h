/*
 * nys.h -- C ABI of libnys: batched streaming Nystrom (landmark) attention
 * for GQA decode on one NVIDIA GB300 (sm_103a).
 *
 * The operator is the one defined in the module documentation of
 * cortiq_engine's nystrom.rs (docs.rs source view, cortiq-engine 0.5.71):
 *
 *   out(q) = (sum_near e_j v_j + F M T_far) / (sum_near e_j + F M Z_far)
 *   e_j = exp(q.k_j/sqrt(d)),  F_a = exp(q.k~_a/sqrt(d)),
 *   M = pinv_reg(exp(Q~ K~^T/sqrt(d))),
 *   T_far = sum_far exp(Q~ k_j/sqrt(d)) v_j^T,  Z_far = sum_far exp(Q~ k_j/sqrt(d)),
 *
 * with an exact ring window of the last w keys, `sink` permanent exact keys,
 * delayed insertion of a key into the far field at the step it leaves the
 * window, per-landmark running maxima, and one joint division.
 *
 * Conventions for every entry point:
 *  - Return 0 (NYS_OK) on success, a negative nys_status otherwise.  The
 *    library never aborts, never traps the GPU and never prints except the
 *    one-time landmark-clamp notice described at nys_seal.
 *  - Every float pointer is a DEVICE pointer to fp32, row-major, 16-byte
 *    aligned, owned by the caller; the library reads inputs and writes only
 *    `out` and the state buffer.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it.  Host-side validation
 *    happens before anything is enqueued, so an error return means nothing
 *    was launched (except NYS_E_CUDA, which reports a failed launch).
 *  - A "group" is one (sequence, layer, KV head) state: the shared window,
 *    sinks and key landmarks plus heads_per_kv private query-head parts.
 *    Query head h of group g is global head g*heads_per_kv + h, so a group's
 *    heads are contiguous in q and out (Struct LayerKvCache, o1_step).
 */
#ifndef NYS_H
#define NYS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NYS_OK = 0,
  NYS_E_INVAL = -1,      /* bad geometry (m<4, w<1, heads<1, sink<0, d or dv
                            not a positive multiple of 4, unknown rect) or a
                            NULL argument                                      */
  NYS_E_RANGE = -2,      /* group range outside the handle, or t <= sink      */
  NYS_E_NOT_SEALED = -3, /* decode step on a group that was never sealed      */
  NYS_E_EXACT_ONLY = -4, /* prompt t <= w + sink + 8: short-prompt mode, which
                            this GPU path does not carry                       */
  NYS_E_BUF = -5,        /* caller buffer smaller than nys_memory_bytes       */
  NYS_E_ALIGN = -6,      /* pointer not 16-byte aligned (state: 256-byte)     */
  NYS_E_CUDA = -7,       /* a CUDA call or kernel launch failed               */
  NYS_E_UNSUPPORTED = -8, /* geometry beyond the kernels' limits: m > 64,
                            d or dv > 256, heads_per_kv > 64, sink + w > 2048  */
  NYS_E_SCRATCH = -9,    /* nys_seal_static only: one group's workspace does
                            not fit the library's static scratch array         */
  NYS_E_CAPACITY = -10   /* an exact-only group would exceed exact_cap keys   */
} nys_status;

/* Rectifier of the skeleton's far mass (nystrom.rs, enum O1Rect).
 * AGGREGATE, the default (nystrom.rs, O1_DEFAULT_RECT): a row whose far
 * denominator is negative drops its far field.  FM: clamp u = F^ M at 0. */
typedef enum { NYS_RECT_AGGREGATE = 0, NYS_RECT_FM = 1 } nys_rect;

/* Geometry shared by every group of a handle (nystrom.rs,
 * NystromState::new_group(m, w, sink, q_heads) and with_rect; the page fixes
 * d and dv at seal time, this library at allocation, so that the state can
 * be laid out up front). */
typedef struct {
  int32_t m;            /* landmark budget, >= 4 (page default 32)            */
  int32_t w;            /* exact window width, >= 1 (page default 128)        */
  int32_t sink;         /* permanent exact sink keys, >= 0 (page default 4)   */
  int32_t heads_per_kv; /* query heads per group, >= 1                        */
  int32_t d;            /* query/key head dim, positive multiple of 4         */
  int32_t dv;           /* value head dim, positive multiple of 4             */
  int32_t rect;         /* nys_rect                                           */
  int32_t exact_cap;    /* keys an exact-only (short-prompt) group can hold; 0
                           (the default) refuses such prompts.  See nys_seal. */
} nys_config;

typedef struct nys_states nys_states; /* opaque host handle */

/* Device layout of the state buffer: the analogue of nystrom.rs
 * O1DeviceView / O1HeadView (every slice the device mirror needs, in the
 * layout the kernels index).  Offsets are bytes from the buffer base; every
 * region starts on a 256-byte boundary and is indexed [group][...] as below.
 * Storage is strided by the budget m: a group sealed with m_eff < m uses the
 * leading m_eff rows, and the top-left m_eff x m_eff block of mu (row
 * stride m).
 *
 *   win_k   f32 [G][w][d]        ring window keys   (shared per group)
 *   win_v   f32 [G][w][dv]       ring window values
 *   sink_k  f32 [G][sink][d]     sink keys
 *   sink_v  f32 [G][sink][dv]    sink values
 *   k_tilde f32 [G][m][d]        key landmarks K~
 *   q_tilde f32 [G][H][m][d]     query landmarks Q~ (per head)
 *   mu      f32 [G][H][m][m]     M: row = key landmark a, column = query
 *                                landmark b
 *   t_hat   f32 [G][H][m][dv]    far numerator at scale e^{-m_max} (high part)
 *   z_hat   f32 [G][H][m]        far denominator, same scale (high part)
 *   m_max   f32 [G][H][m]        per-landmark running max of far logits
 *   t_lo    bf16 [G][H][m][dv]   low part of the far numerator
 *   z_lo    f32 [G][H][m]        low part of the far denominator
 *   exact_k f32 [G][exact_cap][d]   keys of exact-only groups (absent if 0)
 *   exact_v f32 [G][exact_cap][dv]  their values
 *   far_len i32 [G][H]           keys absorbed per head
 *   ints    i32 [G][8]           {win_head, win_len, m_eff, t, mode, status, 0, 0},
 *                                mode 0 = empty, 1 = sealed (landmark path),
 *                                2 = sealed exact-only (win_len = keys held);
 *                                status 0 = fine, nonzero = a bounded wait in a
 *                                decode kernel gave up (every wait is limited
 *                                to 2 s); that group's state is then invalid
 *
 * The far accumulators are carried as unevaluated sums T^ = t_hat + t_lo and
 * Z^ = z_hat + z_lo.  The page keeps them as plain f32; every decode token
 * rounds them once more, and the ill-conditioned mixing F^ M amplifies that
 * drift roughly fifty-fold in the output, so over a thousand tokens plain f32
 * leaves the exact result by ~1e-4.  The low parts hold the rounding error of
 * each update (exact product and sum errors via FMA), which keeps the far
 * field within ~1e-7 of exact at 12.5% more state bytes.
 */
typedef struct {
  size_t total_bytes;
  size_t off_win_k, off_win_v, off_sink_k, off_sink_v, off_k_tilde;
  size_t off_q_tilde, off_mu, off_t_hat, off_z_hat, off_m_max;
  size_t off_t_lo, off_z_lo;
  size_t off_far_len, off_ints;
  size_t off_exact_k, off_exact_v;
  int64_t n_groups;
  int32_t ints_per_group; /* 8 */
} nys_layout;

/* Host-visible summary of one group (nystrom.rs, NystromState::far_len and
 * the O1DeviceView scalars). */
typedef struct {
  int32_t mode;     /* 0 empty, 1 sealed                                      */
  int32_t m_eff;    /* effective landmark count, clamp(t/8, 4, m)             */
  int32_t t;        /* prompt length the group was sealed with                */
  int32_t win_len;  /* keys in the window (w once sealed)                     */
  int32_t win_head; /* ring slot of the oldest window key                     */
  int32_t status;   /* 0 when healthy; 1 when a decode launch's bounded wait
                       gave up before this group was stepped (its state is
                       stale and its last outputs are not valid); 3 when the
                       tensor-core replay of its seal gave up (its far field
                       is not valid).  Sealing again clears it.              */
} nys_group_info;

/* Bytes of device memory a handle of n_groups groups needs (nystrom.rs,
 * NystromState::memory_bytes: window, sinks and K~ once per group; far field,
 * Q~ and M per head.  The page's per-head score scratch is not carried: the
 * kernels keep it on chip).  Writes *device_bytes.  Host arithmetic only;
 * needs no GPU.  Errors: NYS_E_INVAL, NYS_E_UNSUPPORTED. */
int nys_memory_bytes(const nys_config* cfg, int64_t n_groups,
                     size_t* device_bytes);

/* Create a handle for n_groups groups (nystrom.rs, NystromState::new_group,
 * once per group).  dev_buf == NULL: the library cudaMallocs
 * nys_memory_bytes bytes and frees them in nys_free_states.  Otherwise
 * dev_buf is a caller-owned device buffer of at least that size (e.g. a torch
 * tensor), 256-byte aligned, which must outlive the handle.  The buffer is
 * zeroed synchronously, so every group starts empty.  *out receives the
 * handle.  Errors: NYS_E_INVAL, NYS_E_UNSUPPORTED, NYS_E_BUF, NYS_E_ALIGN,
 * NYS_E_CUDA. */
int nys_alloc_states(const nys_config* cfg, int64_t n_groups, void* dev_buf,
                     size_t buf_bytes, nys_states** out);

/* Destroy a handle, and the buffer if the library allocated it, and the
 * second stream and two events its seals use.  The caller must make sure no
 * enqueued work still uses it.  NULL is a no-op. */
int nys_free_states(nys_states* st);

/* Seal groups [g0, g0+n) on a prompt of t positions (nystrom.rs,
 * NystromState::prefill_group, prefill_shared, NystromHead::seal,
 * seg_means, ridge_pinv, cholesky; Struct NystromState, prefill_group):
 *  - sinks = keys/values 0..sink; m_eff = clamp(t/8, 4, m), with one notice
 *    on stderr per process when m_eff < m, as the page warns once;
 *  - K~ = segment means of the keys, Q~_h = segment means of head h's
 *    queries (f64 accumulation, stored f32);
 *  - M_h = (A^T A + lambda I)^-1 A^T of A = exp(Q~ K~^T / sqrt(d)) in f64,
 *    lambda = 1e-6 * mean diag(A^T A), tenfold growth after a failed
 *    Cholesky, at most twelve attempts, stored f32;
 *  - positions sink..t-1 replayed through the window: the last w sit in the
 *    ring, keys sink..t-w-1 are in every head's far field with per-landmark
 *    running max, far_len = t - sink - w.
 * Inputs: q [n][heads_per_kv][t][d], k [n][t][d], v [n][t][dv] (device).
 * Short prompts, t <= w + sink + 8, take the page's exact-only mode
 * (nystrom.rs, prefill_shared and seal_exact): every key stays an exact key
 * in a growing window, with no sinks, landmarks or far field; each decode
 * token appends its key and attends over all keys so far.  That needs
 * cfg.exact_cap >= t (else NYS_E_EXACT_ONLY when exact_cap is 0, NYS_E_RANGE
 * when t > exact_cap); nys_step_batch returns NYS_E_CAPACITY before a token
 * that would exceed exact_cap keys.
 * All n groups share t.  Re-sealing a group replaces its state.  Allocates a
 * temporary f64 workspace of n*m*d*8 bytes with cudaMallocAsync on `stream`
 * and frees it there.  The pinv kernel runs on a second stream owned by the
 * handle (made at its first seal), forked from `stream` and joined back
 * before the call returns, so all of the seal's work is ordered on `stream`
 * as usual; calls on one handle must not overlap.  Writes no attention
 * output (the page's prefill writes none).
 * Errors: NYS_E_INVAL, NYS_E_RANGE, NYS_E_EXACT_ONLY, NYS_E_ALIGN,
 * NYS_E_CUDA. */
int nys_seal(nys_states* st, int64_t g0, int64_t n, int32_t t,
             const float* q, const float* k, const float* v, void* stream);

/* nys_seal for a batch of prompts of different lengths, in one set of
 * launches (nystrom.rs, NystromState::prefill_group applied to each group
 * with its own t; prefill_shared fixes m_eff = clamp(t/8, 4, m) per group,
 * so the effective landmark count may differ between groups of the batch).
 * t_host: host array of n prompt lengths, each > w + sink + 8.
 * Inputs are packed back to back in group order: with off_i = t_0 + ... +
 * t_{i-1}, group g0+i's keys are rows off_i .. off_i + t_i - 1 of
 * k [sum t][d], its values the same rows of v [sum t][dv], and its queries
 * the H*t_i rows starting at row H*off_i of q [H * sum t][d], laid out
 * [H][t_i][d] (all device).  Allocates the f64 workspace and an n*16-byte
 * table of per-group lengths, landmark counts and offsets with
 * cudaMallocAsync on `stream`, and frees both there.
 * Errors: those of nys_seal; NYS_E_EXACT_ONLY or NYS_E_RANGE if any t_i is
 * outside the landmark path (nothing is launched then). */
int nys_seal_ragged(nys_states* st, int64_t g0, int64_t n, const int32_t* t_host,
                    const float* q, const float* k, const float* v, void* stream);

/* One decode token for groups [g0, g0+n) (nystrom.rs,
 * NystromState::step_group and advance, NystromHead::step and far_insert;
 * Struct NystromState, step_group): insert each group's (k, v) once -- a full
 * ring first evicts its oldest key into every head's far field -- then write
 * every head's output.
 * Inputs: q [n][heads_per_kv][d], k [n][d], v [n][dv]; output
 * out [n][heads_per_kv][dv] (all device).  One kernel launch.
 * Groups sealed in exact-only mode run a second, exact-attention kernel.
 * Errors: NYS_E_INVAL, NYS_E_RANGE, NYS_E_NOT_SEALED, NYS_E_ALIGN,
 * NYS_E_CAPACITY, NYS_E_CUDA. */
int nys_step_batch(nys_states* st, int64_t g0, int64_t n, const float* q,
                   const float* k, const float* v, float* out, void* stream);

/* nys_seal without any device allocation.  The pages have no counterpart:
 * this entry point exists for callers that must not allocate device memory
 * while they run -- a serving loop that has reserved all memory up front, an
 * allocator that forbids cudaMalloc/cudaMallocAsync inside its critical
 * section, or code embedded in a host application that owns every buffer.
 * It computes exactly what nys_seal computes (same kernels, the same checks
 * from one shared function, bit-identical states), but its f64 landmark
 * workspace is a 4 MiB array that the
 * library places in device global memory at load time (every GPU that loads
 * the library keeps those 4 MiB until the process exits).  Groups are sealed
 * in chunks that fit the array, one after another on `stream`.
 *  - The first call on a device looks the array's device address up
 *    (cudaGetSymbolAddress) with that device current and caches it; make
 *    that first call before any stream capture on the device.  The cached
 *    address belongs to the device's context as it was then: after a
 *    cudaDeviceReset (or any teardown of that context) it is stale, so do
 *    not call nys_seal_static again in a process that reset the device.
 *  - Exact-only prompts (t <= w + sink + 8 on a handle with exact_cap > 0)
 *    need no workspace; they are sealed exactly as nys_seal seals them.
 *  - Every call on a device shares the one array, and each call overwrites
 *    what the previous one left there.  Calls that may run at the same time
 *    on the GPU (different streams without ordering between them) race on
 *    it: order them on one stream or with events.
 *  - A geometry whose single-group workspace, (1 + heads_per_kv) * m * d * 8
 *    bytes, exceeds 4 MiB is rejected with NYS_E_SCRATCH before anything is
 *    enqueued.
 * Arguments, layouts and the other errors are those of nys_seal (NYS_E_INVAL,
 * NYS_E_RANGE, NYS_E_EXACT_ONLY, NYS_E_ALIGN, NYS_E_CUDA). */
int nys_seal_static(nys_states* st, int64_t g0, int64_t n, int32_t t,
                    const float* q, const float* k, const float* v,
                    void* stream);

/* Read one group's counters to the host (nystrom.rs, NystromState::far_len,
 * and the O1DeviceView scalars).  far_len, if not NULL, receives
 * heads_per_kv entries.  Synchronises `stream`.  Errors: NYS_E_INVAL,
 * NYS_E_RANGE, NYS_E_CUDA. */
int nys_query(const nys_states* st, int64_t g, nys_group_info* info,
              int32_t* far_len, void* stream);

/* The state buffer's base pointer and layout (see nys_layout), so that a
 * caller can read or write any group's state in place, as the page's
 * device_view exposes a sealed group for upload.  Errors: NYS_E_INVAL. */
int nys_layout_of(const nys_states* st, void** base, nys_layout* layout);

/* Declare groups [g0, g0+n) sealed after the caller wrote a complete sealed
 * state into them through nys_layout_of (their ints.mode must be 1 and their
 * ring full).  Host bookkeeping only; nothing is launched.
 * Errors: NYS_E_INVAL, NYS_E_RANGE. */
int nys_mark_sealed(nys_states* st, int64_t g0, int64_t n);

/* Test hook, no counterpart on the pages: the next nys_step_batch on this
 * handle makes its first CTA withhold ring stage `stage` (counted from 0 over
 * that CTA's groups), so that CTA's bounded waits run out after 2 s and it
 * marks its groups' status words.  Exercises the decode kernel's timeout path
 * without faulting or hanging the GPU; the context stays usable and re-sealing
 * clears the status.  Only the fast decode kernel (d, dv <= 128, heads <= 8)
 * waits on anything.  Errors: NYS_E_INVAL. */
int nys_debug_stall_once(nys_states* st, int32_t stage);

/* Test hook, no counterpart on the pages: in the next nys_seal on this
 * handle, the tensor-core replay (groups whose prompt leaves >= 256 keys to
 * fold, m >= 32) skips issuing the first MMAs of its first CTA, so that
 * CTA's bounded waits run out after 2 s and its group's status word becomes
 * 3.  Exercises the replay's timeout path without faulting or hanging the
 * GPU; sealing again clears the status.  Errors: NYS_E_INVAL. */
int nys_debug_stall_replay_once(nys_states* st);

/* The geometry a handle was created with.  Errors: NYS_E_INVAL. */
int nys_config_of(const nys_states* st, nys_config* cfg, int64_t* n_groups);

/* ---- One layer's O(1) override over a batch of sequences ------------------
 * The lifecycle of Struct LayerKvCache (o1_begin, o1_push_q, o1_sealed,
 * o1_seal, o1_step, o1_views, o1_memory_bytes) on top of the calls above.
 * A layer has num_heads query heads over num_kv_heads KV heads for each of
 * `batch` sequences; query head h of a sequence belongs to KV group
 * h / (num_heads / num_kv_heads), so q/out rows are [batch][num_heads][d]. */
typedef struct nys_o1 nys_o1; /* opaque */

/* Arm query collection for a fresh prompt pass (o1_begin): cfg gives m, w,
 * sink, rect, d, dv and exact_cap (heads_per_kv is ignored: it is fixed at
 * seal time from the fan-out).  Allocates a device query trace of
 * batch*num_heads*max_prompt*d floats.  Errors: NYS_E_INVAL,
 * NYS_E_UNSUPPORTED, NYS_E_CUDA. */
int nys_o1_begin(const nys_config* cfg, int32_t batch, int32_t num_heads,
                 int32_t num_kv_heads, int32_t max_prompt, nys_o1** out);

/* Record one prompt position's queries of every sequence (o1_push_q):
 * q_all [batch][num_heads][d] (device), one strided copy on `stream`.  A
 * no-op once the layer is sealed; NYS_E_RANGE after max_prompt positions. */
int nys_o1_push_q(nys_o1* o, const float* q_all, void* stream);

/* Freeze the prompt (o1_seal): k [batch][num_kv_heads][kv_len][d] and v
 * [..][dv] are the layer's prompt keys/values (device, f32).  *sealed = 1
 * when the states were built -- the caller may then drop its KV for this
 * layer; *sealed = 0 (status NYS_OK) when a precondition of the page fails
 * and the layer must stay exact: the query trace is not complete (positions
 * pushed != kv_len), the GQA fan-out does not divide, the KV is not densely
 * stored (kv_dense = 0), or a short prompt (kv_len <= w + sink + 8) has no
 * exact_cap room.  Synchronises `stream`, then releases the trace.
 * Errors: those of nys_alloc_states and nys_seal. */
int nys_o1_seal(nys_o1* o, const float* k, const float* v, int32_t kv_len,
                int32_t kv_dense, void* stream, int32_t* sealed);

/* *sealed = 1 once nys_o1_seal built the states (o1_sealed). */
int nys_o1_sealed(const nys_o1* o, int32_t* sealed);

/* One decode token of the whole layer (o1_step): q_all [batch][num_heads][d],
 * k_new/v_new [batch][num_kv_heads][d|dv], out [batch][num_heads][dv].
 * Errors: NYS_E_NOT_SEALED, and those of nys_step_batch. */
int nys_o1_step(nys_o1* o, const float* q_all, const float* k_new,
                const float* v_new, float* out, void* stream);

/* Device bytes held (o1_memory_bytes): the query trace recorded so far while
 * collecting, the states once sealed. */
int nys_o1_memory_bytes(const nys_o1* o, size_t* bytes);

/* The sealed states (the o1_views analogue; see nys_layout_of), or
 * NYS_E_NOT_SEALED.  Owned by the nys_o1. */
int nys_o1_states(const nys_o1* o, nys_states** st);

/* Release the trace and the states.  NULL is a no-op. */
int nys_o1_free(nys_o1* o);

/* Static description of a status code.  Never NULL. */
const char* nys_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* NYS_H */
