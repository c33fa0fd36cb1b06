/*
 * gdn.h -- C ABI of libgdn: the chunked gated delta rule (GDN) forward and
 * backward over packed variable-length sequences, and the single-token decode
 * step over a slot-indexed state pool, on NVIDIA GB300 (sm_103a).
 *
 * What is computed.  Per sequence n and value head hv, with key head
 * h = hv / (HV / H):
 *     qhat_t = scale * q_t / sqrt(sum_i q_{t,i}^2 + 1e-6)
 *     khat_t =         k_t / sqrt(sum_i k_{t,i}^2 + 1e-6)     (k is never scaled)
 *     S_t    = exp(g_t) S_{t-1} (I - beta_t khat_t khat_t^T) + beta_t v_t khat_t^T
 *     o_t    = S_t qhat_t
 * with S (V x K) starting from the transpose of initial_state[n, hv] (or 0).
 * Sources (page title, section):
 *   - "cake_gdn: deterministic chunked GDN training kernels" (miles #3597),
 *     Summary: chunk 64, K = V = 128, in-kernel q/k L2 norm, cu_seqlens
 *     packing, per-chunk state h stored in bf16 with an fp32 running state,
 *     reductions without device atomics (bit-identical repeats).
 *   - "[Cake 1/13] gdn: chunked gated delta rule, det and fast, with KCP and
 *     FLA-CP" (miles-ext-kernels #1), API and flags: q/k [B,T,H,K],
 *     v [B,T,HV,V], HV % H == 0, bf16 q/k/v, packed varlen B = 1, fp32
 *     initial/final state [N,HV,K,V], host cu_seqlens with no device-to-host
 *     sync, a call without tokens passes the state through; extents checked
 *     before any launch.
 *   - "C6: GDN decode-step goldens and recurrent/conv state contract"
 *     (RL-Kernel #469), What / Provider: the L2 norm divides by the sqrt,
 *     scale multiplies q after the norm, key head = hv // (HV // H), state pool
 *     [num_blocks, HV, V, K] addressed by ssm_state_indices, every index <= 0
 *     is skipped and its output row written as zeros, fp32 accumulator.
 *
 * Conventions for every entry point:
 *   - All tensors are dense, row-major, on the device of the current CUDA
 *     context, except cu_seqlens_host (host memory).  bf16 = IEEE bfloat16 bits.
 *   - Calls are asynchronous and ordered on `stream`.  The library allocates
 *     no memory, keeps no pointer after it returns and has no global mutable
 *     state; the caller owns every buffer.
 *   - Arguments are validated on the host before any launch; an invalid call
 *     returns an error and launches nothing.  GDN_ERR_CUDA reports a failed
 *     launch (cudaGetLastError) and may leave outputs partly written.
 *   - Results are deterministic: the same inputs give the same bits on any
 *     stream and in any process (no device atomics, fixed reduction orders).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL = the legacy default stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,          /* null pointer, bad extents, bad cu_seqlens */
    GDN_ERR_UNSUPPORTED = 2,          /* K or V != 128, HV % H != 0 */
    GDN_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below the size query */
    GDN_ERR_CUDA = 4                  /* a CUDA launch or call failed */
} gdn_status;

/* Element types of beta / dbeta in the chunk calls ("[Cake 1/13] gdn: chunked
 * gated delta rule, det and fast, with KCP and FLA-CP", Performance (3/5): the
 * training kernels are timed with BF16 beta and with FP32 beta). */
#define GDN_DTYPE_BF16 0
#define GDN_DTYPE_F32 1

/* A packed variable-length problem (B = 1).  Sequence n holds tokens
 * [cu[n], cu[n+1]) of the packed arrays.  Chunks of 64 tokens never span two
 * sequences; the last chunk of a sequence may be partial. */
typedef struct {
    int32_t num_seqs;                 /* N >= 1 */
    int64_t total_tokens;             /* T >= 0, T == cu[N]; T < 2^31 */
    int32_t num_k_heads;              /* H >= 1 */
    int32_t num_v_heads;              /* HV >= 1, HV % H == 0 */
    int32_t head_dim_k;               /* K, must be 128 */
    int32_t head_dim_v;               /* V, must be 128 */
    float scale;                      /* > 0, or <= 0 to select 1/sqrt(K) */
    int32_t beta_dtype;               /* GDN_DTYPE_BF16 (0, the default of a
                                         zeroed struct) or GDN_DTYPE_F32: the
                                         element type of beta and dbeta; any
                                         other value is GDN_ERR_INVALID_ARG */
    const int32_t *cu_seqlens_host;   /* host [N+1]: 0 = c0 <= c1 <= ... <= cN = T */
    const int32_t *cu_seqlens_dev;    /* device [N+1], the same values */
    int32_t *device_status;           /* device int32, or NULL: the chunk calls OR
                                         GDN_DEVICE_* bits into it when a kernel
                                         finds something wrong (see below); the
                                         library never clears it */
    int32_t scan_segment_chunks;      /* plan of the state scans (see
                                         gdn_chunk_scan_plan): 0 (the default of a
                                         zeroed struct) = the library's plan, -1 =
                                         never split, L > 0 = segments of L chunks;
                                         other values are GDN_ERR_INVALID_ARG */
} gdn_problem;

/* Bits of gdn_problem.device_status ("[Cake 1/13] gdn: chunked gated delta rule,
 * det and fast, with KCP and FLA-CP", API and flags: failures are reported, not
 * silent).  The word is written by the kernels, so it is valid once the call's
 * work on `stream` has finished; a set bit means the outputs of that call are
 * not to be trusted.
 *   GDN_DEVICE_CU_SEQLENS_MISMATCH  cu_seqlens_dev disagrees with the host copy
 *                                   (the chunk table is clamped to the host's
 *                                   extents, so no access leaves the buffers)
 *   GDN_DEVICE_WAIT_TIMEOUT         a bounded wait for a tensor-core product or
 *                                   a TMA copy ran out (one second); the kernel
 *                                   drained its copies, freed its tensor memory
 *                                   and returned early
 *   GDN_DEVICE_INDEX_OUT_OF_RANGE   (builds with GDN_CHECKED only) a global
 *                                   index fell outside its buffer; the access
 *                                   was skipped */
#define GDN_DEVICE_CU_SEQLENS_MISMATCH 1
#define GDN_DEVICE_WAIT_TIMEOUT 2
#define GDN_DEVICE_INDEX_OUT_OF_RANGE 4

/* Bytes of the `saved` buffer gdn_chunk_fwd fills for gdn_chunk_bwd (per-chunk
 * states in bf16, the WY matrices, v_new and the norm / gate prefix sums).
 * Returns 0 for an invalid problem.  Pure host function. */
size_t gdn_chunk_saved_bytes(const gdn_problem *p);

/* Bytes of scratch the calls need.  for_backward = 0: gdn_chunk_fwd (this
 * includes room for the saved tensors, used when `saved` is NULL);
 * for_backward = 1: gdn_chunk_bwd with a `saved` buffer; for_backward = 2:
 * gdn_chunk_bwd in recompute-state mode (`saved` NULL: the workspace also
 * holds the recomputed forward tensors).  Returns 0 for an invalid problem or
 * another for_backward value. */
size_t gdn_chunk_workspace_bytes(const gdn_problem *p, int for_backward);

/* How the forward state scan of this problem is run (a pure host function of
 * the problem; the same plan on every device, so the same bits).  A scan walks
 * the chunks of a sequence one after another; when a few long sequences would
 * leave the GPU idle, every sequence is cut into segments of *seg_len chunks
 * (segment-parallel scan: the transitions of the segments are scanned at once,
 * stitched, and the segments re-scanned from their start states, as the
 * pre-scan + stitch of the context-parallel state scans in "[Cake 1/13] gdn:
 * ...", Review items, and the GDN context-parallel m-scan of "Qwen3.5-397B RL
 * trainer on 128 v7x").  *seg_len = 0 and *num_segments = 1 when the scan is
 * not split; otherwise *num_segments is the largest segment count of any
 * sequence.  The split changes the rounding of the states (not their values
 * beyond it) and adds its buffers to both workspace queries.  The problem's
 * scan_segment_chunks field overrides the plan: -1 never splits, L > 0 cuts
 * every sequence into segments of L chunks whenever some sequence then has 3 or
 * more (and the segment count stays within 4096). */
gdn_status gdn_chunk_scan_plan(const gdn_problem *p, int32_t *seg_len, int32_t *num_segments);

/* Forward of chunk_gated_delta_rule.
 *   q, k           bf16 [T, H, 128]
 *   v              bf16 [T, HV, 128]
 *   g              fp32 [T, HV]  log decay per token and value head
 *   beta           [T, HV], bf16 or fp32 as p->beta_dtype says
 *   initial_state  fp32 [N, HV, 128(K), 128(V)] K-major, or NULL for zeros
 *   o              bf16 [T, HV, 128]           (out)
 *   final_state    fp32 [N, HV, 128, 128] (out), or NULL
 *   saved          gdn_chunk_saved_bytes() bytes (out), or NULL when no
 *                  backward follows
 *   workspace      ws_bytes >= gdn_chunk_workspace_bytes(p, 0), 256-byte aligned
 * T == 0 writes final_state = initial_state (or zeros) and nothing else. */
gdn_status gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *initial_state,
                         void *o, float *final_state, void *saved, void *workspace,
                         size_t ws_bytes, gdn_stream_t stream);

/* gdn_chunk_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for callers such as code
 * inside a pre-planned memory arena that forbids new allocations after
 * start-up, host plugins that receive only their input and output buffers, and
 * latency-critical paths that must avoid the synchronisation cudaMalloc and
 * cudaFree can cause.  Inputs and outputs are as in gdn_chunk_fwd; no `saved`
 * buffer is produced (forward only).  The scratch is a fixed 64 MiB device
 * array inside the library (every GPU that loads libgdn.so holds it until the
 * process exits); a problem whose forward workspace
 * (gdn_chunk_workspace_bytes(p, 0)) exceeds 64 MiB is rejected with
 * GDN_ERR_WORKSPACE_TOO_SMALL before any launch.  Nothing is allocated.  The
 * first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls on a device share the array: calls
 * that overlap on the GPU race and give undefined results, so order them on
 * one stream. */
gdn_status gdn_chunk_fwd_noalloc(const gdn_problem *p, const void *q, const void *k,
                                 const void *v, const float *g, const void *beta,
                                 const float *initial_state, void *o, float *final_state,
                                 gdn_stream_t stream);

/* Paged chunk prefill ("Replace Qwen3.5 FLA paths with Attention Gym"
 * (torchtitan #4389), GDN prefill ablation and Paged-state continuity): the
 * forward of gdn_chunk_fwd whose states live in the decode state pool, so a
 * prefill advances the slots in place with no gather / scatter copies.
 *   q, k, v, g, beta, o   as in gdn_chunk_fwd (forward only: nothing saved)
 *   state_pool            fp32 [num_slots, HV, V, K] (V-major, the layout of
 *                         gdn_decode_step), updated in place
 *   state_indices         int32 [N] on the device: the slot of sequence n; a
 *                         slot <= 0 is none: the sequence starts from zeros
 *                         and its final state is dropped; a slot >= num_slots
 *                         is skipped the same way and flagged in device_status
 *   has_initial_state     int32 [N] on the device, or NULL (= all nonzero):
 *                         nonzero resumes from the slot's state, 0 starts the
 *                         sequence fresh from zeros; the final state of every
 *                         sequence with a slot is written to that slot
 *   device_status         int32 on the device, or NULL
 *   workspace             ws_bytes >= gdn_chunk_workspace_bytes(p, 0)
 * Two sequences naming the same slot race (a caller error).  The results are
 * the bits of gdn_chunk_fwd with initial_state[n] = the transpose of the slot
 * (or zeros) and final_state[n] copied back transposed. */
gdn_status gdn_chunk_prefill_paged(const gdn_problem *p, const void *q, const void *k,
                                   const void *v, const float *g, const void *beta,
                                   float *state_pool, int32_t num_slots,
                                   const int32_t *state_indices, const int32_t *has_initial_state,
                                   void *o, int32_t *device_status, void *workspace,
                                   size_t ws_bytes, gdn_stream_t stream);

/* Backward of chunk_gated_delta_rule.  q ... initial_state exactly as passed
 * to the gdn_chunk_fwd that filled `saved` (not modified since).
 *   saved          the buffer gdn_chunk_fwd filled, or NULL for recompute-state
 *                  mode ("[Cake 1/13] gdn: ...", API and flags: the recompute
 *                  option rebuilds w, u, h and v_new in the backward): the call
 *                  first reruns the forward's norm / gate pass, WY pass and
 *                  state scan into the workspace (no o, no final state), then
 *                  the backward; the results are bit-identical to those of the
 *                  saved mode, since the same kernels run in the same order
 *   d_o            bf16 [T, HV, 128]
 *   d_final_state  fp32 [N, HV, 128, 128], or NULL for zeros
 *   dq, dk         bf16 [T, H, 128]   (out; summed over the HV/H value heads)
 *   dv             bf16 [T, HV, 128]  (out)
 *   dg             fp32 [T, HV]       (out)
 *   dbeta          [T, HV] (out), beta's dtype
 *   dh0            fp32 [N, HV, 128, 128] (out), or NULL
 *   workspace      ws_bytes >= gdn_chunk_workspace_bytes(p, 1) with `saved`,
 *                  >= gdn_chunk_workspace_bytes(p, 2) without; 256-byte aligned
 * The reverse state recurrence follows "Qwen3.5-397B RL trainer on 128 v7x"
 * (maxtext #5799), GDN context-parallel dh-scan commit. */
gdn_status gdn_chunk_bwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *initial_state,
                         const void *saved, const void *d_o, const float *d_final_state,
                         void *dq, void *dk, void *dv, float *dg, void *dbeta, float *dh0,
                         void *workspace, size_t ws_bytes, gdn_stream_t stream);

/* One decode token per row over a slot-indexed fp32 state pool
 * ("C6: GDN decode-step goldens ...", Provider and State contract).
 *   q, k           bf16 [batch, H, K]
 *   v              bf16 [batch, HV, V]
 *   g, beta        fp32 [batch, HV]
 *   state_pool     fp32 [num_slots, HV, V, K] (V-major: row v of S holds K
 *                  floats), updated in place
 *   state_indices  int32 [batch] on the device: the slot of each row; a slot
 *                  <= 0 is null: the row is skipped, its output row is zeros
 *                  and no slot is touched
 *   o              bf16 [batch, HV, V] (out)
 *   device_status  int32 on the device, or NULL: set to 1 when a row's slot
 *                  was >= num_slots (that row is then treated as null)
 * Two active rows naming the same slot race (undefined result): a caller error.
 * K and V must be 128. */
gdn_status gdn_decode_step(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                           int32_t head_dim_k, int32_t head_dim_v, float scale,
                           const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float *state_pool, int32_t num_slots,
                           const int32_t *state_indices, void *o, int32_t *device_status,
                           gdn_stream_t stream);

/* Host-side check of a decode batch's slot indices ("C6: GDN decode-step goldens
 * and recurrent/conv state contract", State contract: one slot per active row).
 * gdn_decode_step cannot see a repeated slot without a device-to-host copy, so
 * it races on one instead; callers that want the rule enforced run this on the
 * host copy of the indices before the step.  Reads only host memory, launches
 * nothing, needs no GPU.
 *   state_indices  int32 [batch] on the HOST
 *   num_slots      pool size (>= 1)
 *   bad_row        out, or NULL: the first row that breaks the rule, -1 if none
 * Rows with an index <= 0 are null and may repeat.  Returns GDN_OK when every
 * active index is < num_slots and no active index repeats; GDN_ERR_INVALID_ARG
 * otherwise (also for batch < 0, num_slots < 1 or a NULL array with batch > 0).
 * A repeat is reported at the later of the two rows. */
gdn_status gdn_check_indices(const int32_t *state_indices, int32_t batch, int32_t num_slots,
                             int32_t *bad_row);

/* Fused gating ("C6: GDN decode-step goldens and recurrent/conv state
 * contract" (RL-Kernel #469), What and Provider): the decay and beta are
 * computed inside the kernels, in fp32, from their pre-activations:
 *     beta_t = sigmoid(b_t)
 *     g_t    = -exp(A_log[hv]) * softplus(a_t + dt_bias[hv]),
 *     softplus(x) = x for x > 20, log(1 + exp(x)) otherwise.
 *   a, b           bf16 [T, HV] (decode: [batch, HV])
 *   A_log, dt_bias fp32 [HV]
 * The *_gated calls take these in place of g and beta; every other argument
 * is as in the call without the suffix, and p->beta_dtype must be
 * GDN_DTYPE_BF16.  The backward returns, in place of dg and dbeta:
 *   da, db            bf16 [T, HV]: da = dg * (-exp(A_log)) * softplus'(a + dt_bias)
 *                     with softplus' = 1 above the threshold and sigmoid below;
 *                     db = dbeta * beta (1 - beta)
 *   dA_log, ddt_bias  fp32 [HV] (out, required): sums over every token of the
 *                     call of dg * g and of da, in a fixed order (zeros when
 *                     T == 0)
 * A backward after gdn_chunk_fwd_gated must be gdn_chunk_bwd_gated (the saved
 * buffer holds the cumulative decay of the fused gate).  Recompute-state mode
 * (saved NULL) works as in gdn_chunk_bwd. */
gdn_status gdn_chunk_fwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const void *a, const void *b, const float *A_log,
                               const float *dt_bias, const float *initial_state, void *o,
                               float *final_state, void *saved, void *workspace,
                               size_t ws_bytes, gdn_stream_t stream);
gdn_status gdn_chunk_bwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const void *a, const void *b, const float *A_log,
                               const float *dt_bias, const float *initial_state,
                               const void *saved, const void *d_o, const float *d_final_state,
                               void *dq, void *dk, void *dv, void *da, void *db, float *dA_log,
                               float *ddt_bias, float *dh0, void *workspace, size_t ws_bytes,
                               gdn_stream_t stream);
gdn_status gdn_decode_step_gated(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, float scale,
                                 const void *q, const void *k, const void *v, const void *a,
                                 const void *b, const float *A_log, const float *dt_bias,
                                 float *state_pool, int32_t num_slots,
                                 const int32_t *state_indices, void *o, int32_t *device_status,
                                 gdn_stream_t stream);

/* Optional per-kernel timing, for profiling tools and benchmarks.  The caller
 * creates `capacity` pairs of CUDA events (cudaEvent_t, passed as void*) and
 * passes the struct to a *_timed entry point; the library records
 * start_events[i] / stop_events[i] on `stream` around the i-th kernel it
 * launches, stores that kernel's id (GDN_KERNEL_*) in kernel_ids[i] and the
 * number of pairs used in `count`.  Launches past `capacity` are not timed.
 * Recording adds one event pair per launch; results are unchanged. */
typedef struct {
    int32_t capacity;
    int32_t count;           /* out */
    void **start_events;     /* cudaEvent_t[capacity] */
    void **stop_events;      /* cudaEvent_t[capacity] */
    int32_t *kernel_ids;     /* out, [capacity] */
} gdn_kernel_timer;

enum {
    GDN_KERNEL_PLAN = 0,     /* chunk table from cu_seqlens */
    GDN_KERNEL_PREP,         /* q/k norms, chunk-local cumsum of g */
    GDN_KERNEL_INTRA,        /* WY pass: A, (I + A)^-1, w, u */
    GDN_KERNEL_STATE,        /* forward state scan: v_new, per-chunk h, final state */
    GDN_KERNEL_OUT,          /* output o */
    GDN_KERNEL_DVLOC,        /* backward: tril(Qhat Khat^T (.) decay)^T dO */
    GDN_KERNEL_BSTATE,       /* backward reverse state scan: dh, dv_new, dh0 */
    GDN_KERNEL_BINTRA_A,     /* backward: terms through h and dh; dq (summed over the
                                value heads of a key head, L2-norm backward applied) */
    GDN_KERNEL_BINTRA_B,     /* backward: intra-chunk terms, WY pullback, dg, and dk
                                (the khat gradient summed over the value heads of a
                                key head, L2-norm backward applied) */
    GDN_KERNEL_DECODE,       /* decode step */
    GDN_KERNEL_SEG_STITCH,   /* segment-parallel state scan: start states of the segments */
    GDN_KERNEL_COUNT
};

/* Name of a GDN_KERNEL_* id ("unknown" otherwise). */
const char *gdn_kernel_name(int32_t kernel_id);

/* gdn_chunk_fwd / gdn_chunk_bwd / gdn_decode_step with a kernel timer
 * (timer may be NULL, then identical to the plain call). */
gdn_status gdn_chunk_fwd_timed(const gdn_problem *p, const void *q, const void *k,
                               const void *v, const float *g, const void *beta,
                               const float *initial_state, void *o, float *final_state,
                               void *saved, void *workspace, size_t ws_bytes,
                               gdn_stream_t stream, gdn_kernel_timer *timer);
gdn_status gdn_chunk_bwd_timed(const gdn_problem *p, const void *q, const void *k,
                               const void *v, const float *g, const void *beta,
                               const float *initial_state, const void *saved, const void *d_o,
                               const float *d_final_state, void *dq, void *dk, void *dv,
                               float *dg, void *dbeta, float *dh0, void *workspace,
                               size_t ws_bytes, gdn_stream_t stream, gdn_kernel_timer *timer);
gdn_status gdn_decode_step_timed(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, float scale,
                                 const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, float *state_pool, int32_t num_slots,
                                 const int32_t *state_indices, void *o, int32_t *device_status,
                                 gdn_stream_t stream, gdn_kernel_timer *timer);

/* Diagnostic: runs one kernel that waits, with the same bounded mbarrier wait
 * the chunk kernels use, on a barrier that nothing ever arrives on.  After
 * limit_ns nanoseconds (1e3 .. 1e9) the wait gives up and the kernel ORs
 * GDN_DEVICE_WAIT_TIMEOUT into *device_status (device int32, required), as a
 * chunk kernel does when one of its waits runs out; the context stays usable.
 * Returns GDN_ERR_INVALID_ARG for a NULL or misaligned word or a limit outside
 * the range.  The pages have no counterpart: it exists so that the failure path
 * of the bounded waits can be tested without faulting or hanging a GPU. */
gdn_status gdn_selftest_bounded_wait(int32_t *device_status, uint64_t limit_ns,
                                     gdn_stream_t stream);

/* A static, human-readable name of a status code. */
const char *gdn_status_string(gdn_status s);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
