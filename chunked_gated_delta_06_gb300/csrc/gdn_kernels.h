// gdn_kernels.h -- host-side launchers of the libgdn kernels (internal C++ interface).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"

namespace gdn {

// Per (chunk, value head): the scalars the two state scans apply per token, written by
// the WY pass (k_intra_tc) and copied into shared memory by the scans with their tiles (one 16-byte
// aligned bulk copy), so that no scan step waits on scattered global loads.
struct alignas(16) ScRec {
    float kc[kChunk];   // e^{G_L - G_t} / r_k,t, 0 past L
    float qc[kChunk];   // e^{G_t} scale / r_q,t, 0 past L
    float egl;          // e^{G_L}
    float pad[3];
};
static_assert(sizeof(ScRec) % 16 == 0, "bulk copies move multiples of 16 bytes");
constexpr int kScRec = (int)(sizeof(ScRec) / sizeof(float));

// Everything one chunk call touches.  Pointers the call does not use are null.
struct ChunkArgs {
    int N, T, H, HV, num_chunks;
    float scale;
    // inputs
    const bf16 *q, *k, *v;
    const float *g;
    const void *beta;       // [T,HV] bf16 or fp32 (beta_mode 0 / 1)
    int beta_mode;          // 0: bf16 beta; 1: fp32 beta; 2: fused gating (beta = sigmoid(gb))
    // fused gating (beta_mode 2): g and beta come from these instead of g / beta
    const bf16 *ga, *gb;    // [T,HV] pre-activations of the gate and of beta
    const float *A_log, *dt_bias;  // [HV]
    const float *h0;        // [N,HV,K,V] or null
    const int *cu_dev;      // [N+1]
    // forward outputs
    bf16 *o;
    float *ht;              // or null
    // paged prefill: the initial state of sequence n is read from, and its final state
    // written to, pool slot pool_idx[n] ([num_slots,HV,V,K], V-major) in place
    float *pool;            // null = h0 / ht above
    int num_slots;
    const int *pool_idx;    // [N] device; <= 0: no slot (zero start, final state dropped)
    const int *pool_resume; // [N] device or null: 0 = fresh (zero start) although a slot is named
    int *pool_status;       // device or null: set to 1 when an index >= num_slots was skipped
    // saved by the forward, read by the backward
    bf16 *hc;               // [C_total,HV,K,V] state at each chunk start
    bf16 *vnew;             // [T,HV,V]
    bf16 *w;                // w^T per chunk: [C,HV,K,64] (row k holds the chunk's 64 tokens; zero past L)
    bf16 *Tm;               // [C_total,HV,64,64] (I + A)^-1
    float *rq, *rk;         // [T,H] sqrt(|x|^2 + eps)
    float *G;               // [T,HV] chunk-local cumulative log decay
    float *sc;              // [C,HV] records of kScRec floats: the scans' per-token scalars
                            // kc_t = e^{G_L-G_t} / r_k,t, qc_t = e^{G_t} scale / r_q,t (0 past
                            // L) and e^{G_L} (see ScRec)
    // chunk table (device, rebuilt by every call)
    int *seq_chunk_off, *chunk_start, *chunk_len;
    int max_seq_chunks;     // chunks of the longest sequence (host copy of cu_seqlens)
    int *seq_order;         // [N] sequences by decreasing length (scans start the longest first)
    int *status;            // the caller's device status word or null: bit 1 = inconsistent
                            // device cu_seqlens, bit 2 = a bounded wait ran out
    // segment-parallel forward state scan (seg_len = 0: one piece per sequence)
    int seg_len;            // chunks per segment
    int seg_max;            // largest segment count of any sequence (>= 3 when seg_len > 0)
    float *seg_end;         // [N,seg_max-1,HV,K,2K] end states of segment 0 and the pre-scans: [h | Phi]
    float *seg_start;       // [N,seg_max-1,HV,K,V] start states of segments 1 .. S-1
    // forward scratch
    bf16 *u;                // u^T per chunk: [C,HV,V,64] (as w)
    // backward
    const bf16 *d_o;
    const float *d_ht;      // or null
    bf16 *dq, *dk, *dv;
    void *dbeta;            // [T,HV], beta's dtype; with fused gating db (bf16)
    bf16 *da;               // [T,HV] fused gating: gradient of the gate pre-activation
    float *dA_log, *ddt_bias;  // [HV] fused gating: sums over all tokens
    float *gpart;           // [C_total,HV,2] per-chunk sums of dg g and of da (fused gating)
    float *dg, *dh0;        // dh0 may be null
    bf16 *dvloc;            // [T,HV,V]  tril(M)^T dO
    bf16 *dvnew;            // [T,HV,V]  full gradient of v_new
    bf16 *dhc;              // [C_total,HV,K,V] gradient of the state after each chunk
    bf16 *dW;               // [T,HV,K]
    bf16 *dkpart;           // [T,H,K] the h / dh' and Q K^T terms of the khat gradient,
                            // summed over the value heads of each key head
                            // the same way
    float *dGp;             // [T,HV]
    gdn_kernel_timer *timer;  // optional per-kernel events
};

// Element extents of the buffers a chunk call touches (for in_range()).
__device__ __forceinline__ long long n_tok_h(const ChunkArgs &a) { return (long long)a.T * a.H; }
__device__ __forceinline__ long long n_tok_hv(const ChunkArgs &a) { return (long long)a.T * a.HV; }
__device__ __forceinline__ long long n_rows_h(const ChunkArgs &a) { return (long long)a.T * a.H * kDim; }
__device__ __forceinline__ long long n_rows_hv(const ChunkArgs &a) { return (long long)a.T * a.HV * kDim; }
__device__ __forceinline__ long long n_states(const ChunkArgs &a) {
    return (long long)a.N * a.HV * kDim * kDim;
}

// beta_i in the form the call gives it (a uniform branch per load).
__device__ __forceinline__ float load_beta(const ChunkArgs &a, size_t i) {
    if (!in_range(i, 1, n_tok_hv(a), a.status)) return 0.f;
    if (a.beta_mode == 2) return gate_sigmoid(bf2f(a.gb[i]));
    return a.beta_mode ? static_cast<const float *>(a.beta)[i] : bf2f(static_cast<const bf16 *>(a.beta)[i]);
}
// The same in two steps, so that a prefetch does not wait for its load: the raw bits
// (fp32, or bf16 in the low half) now, the value when it is used.
__device__ __forceinline__ uint32_t load_beta_raw(const ChunkArgs &a, size_t i) {
    if (!in_range(i, 1, n_tok_hv(a), a.status)) return 0u;
    if (a.beta_mode == 1) return __float_as_uint(static_cast<const float *>(a.beta)[i]);
    const bf16 *p = a.beta_mode == 2 ? a.gb : static_cast<const bf16 *>(a.beta);
    return (uint32_t)__bfloat16_as_ushort(p[i]);
}
__device__ __forceinline__ float beta_from_raw(const ChunkArgs &a, uint32_t bits) {
    if (a.beta_mode == 1) return __uint_as_float(bits);
    const float x = __uint_as_float(bits << 16);
    return a.beta_mode == 2 ? gate_sigmoid(x) : x;
}
// dbeta_i = x in beta's dtype; with fused gating db_i = x beta_i (1 - beta_i) (bf16).
__device__ __forceinline__ void store_dbeta(const ChunkArgs &a, size_t i, float x, float beta) {
    if (!in_range(i, 1, n_tok_hv(a), a.status)) return;
    if (a.beta_mode == 1) static_cast<float *>(a.dbeta)[i] = x;
    else static_cast<bf16 *>(a.dbeta)[i] = f2bf(a.beta_mode == 2 ? x * (beta * (1.f - beta)) : x);
}
// g_i: the input, or -exp(A_log) softplus(a + dt_bias) with fused gating.
__device__ __forceinline__ float load_g(const ChunkArgs &a, size_t i, int hv) {
    if (!in_range(i, 1, n_tok_hv(a), a.status) || !in_range(hv, 1, a.HV, a.status)) return 0.f;
    if (a.beta_mode != 2) return a.g[i];
    return -expf(a.A_log[hv]) * gate_softplus(bf2f(a.ga[i]) + a.dt_bias[hv]);
}

// Records the caller's event pair around one launch (no-op without a timer).
struct TimerScope {
    gdn_kernel_timer *t;
    cudaStream_t s;
    int slot = -1;
    TimerScope(gdn_kernel_timer *t_, int id, cudaStream_t s_) : t(t_), s(s_) {
        if (t && t->count < t->capacity) {
            slot = t->count++;
            t->kernel_ids[slot] = id;
            cudaEventRecord(static_cast<cudaEvent_t>(t->start_events[slot]), s);
        }
    }
    ~TimerScope() {
        if (slot >= 0) cudaEventRecord(static_cast<cudaEvent_t>(t->stop_events[slot]), s);
    }
};

// Number of SMs of the current device (grid sizing of the persistent kernels).
inline cudaError_t sm_count(int *n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
}

cudaError_t launch_plan(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_prep(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_fwd_chunks(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_recompute_chunks(const ChunkArgs &a, cudaStream_t s);  // WY pass + state scan
cudaError_t launch_gate_reduce(const ChunkArgs &a, cudaStream_t s);       // dA_log, ddt_bias
cudaError_t launch_bwd_chunks(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_state_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_bstate_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_seg_stitch(const ChunkArgs &a, cudaStream_t s);  // segment start states
cudaError_t launch_bintra_a_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_out_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_dvloc_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_bintra_b_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_intra_tc(const ChunkArgs &a, cudaStream_t s);

// Fused-gating inputs of the decode step (a null = g and beta are given).
struct DecodeGate {
    const bf16 *a, *b;             // [B,HV]
    const float *A_log, *dt_bias;  // [HV]
};
cudaError_t launch_decode(int B, int H, int HV, float scale, const bf16 *q, const bf16 *k,
                          const bf16 *v, const float *g, const float *beta, const DecodeGate &gate,
                          float *pool, int num_slots, const int32_t *idx, bf16 *o, int32_t *status,
                          cudaStream_t s, gdn_kernel_timer *timer);

}  // namespace gdn
