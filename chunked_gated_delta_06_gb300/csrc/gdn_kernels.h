// gdn_kernels.h -- host-side launchers of the libgdn kernels (internal C++ interface).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"
#include "gdn_common.cuh"

namespace gdn {

// Everything one chunk call touches.  Pointers the call does not use are null.
struct ChunkArgs {
    int N, T, H, HV, num_chunks;
    float scale;
    // inputs
    const bf16 *q, *k, *v;
    const float *g;
    const void *beta;       // [T,HV] bf16, or fp32 when beta_f32
    int beta_f32;           // the dtype of beta and dbeta
    const float *h0;        // [N,HV,K,V] or null
    const int *cu_dev;      // [N+1]
    // forward outputs
    bf16 *o;
    float *ht;              // or null
    // saved by the forward, read by the backward
    bf16 *hc;               // [C_total,HV,K,V] state at each chunk start
    bf16 *vnew;             // [T,HV,V]
    bf16 *w;                // [T,HV,K]
    bf16 *Tm;               // [C_total,HV,64,64] (I + A)^-1
    float *rq, *rk;         // [T,H] sqrt(|x|^2 + eps)
    float *G;               // [T,HV] chunk-local cumulative log decay
    // chunk table (device, rebuilt by every call)
    int *seq_chunk_off, *chunk_seq, *chunk_start, *chunk_len;
    int *seq_order;         // [N] sequences by decreasing length (scans start the longest first)
    int *status;            // device int, nonzero = inconsistent device cu_seqlens
    // forward scratch
    bf16 *u;                // [T,HV,V]
    // backward
    const bf16 *d_o;
    const float *d_ht;      // or null
    bf16 *dq, *dk, *dv;
    void *dbeta;            // [T,HV], beta's dtype
    float *dg, *dh0;        // dh0 may be null
    bf16 *dvloc;            // [T,HV,V]  tril(M)^T dO
    bf16 *dvnew;            // [T,HV,V]  full gradient of v_new
    bf16 *dhc;              // [C_total,HV,K,V] gradient of the state after each chunk
    bf16 *dW;               // [T,HV,K]
    bf16 *dqp, *dkp;        // [T,HV,K] per-value-head gradients of qhat (all terms) and
                            // khat (h / dh' and Q K^T terms)
    bf16 *dkp2;             // [T,HV,K] the WY-pullback terms of the khat gradient
    float *dGp;             // [T,HV]
    gdn_kernel_timer *timer;  // optional per-kernel events
};

// beta_i and dbeta_i in the dtype the call names (a uniform branch per load).
__device__ __forceinline__ float load_beta(const ChunkArgs &a, size_t i) {
    return a.beta_f32 ? static_cast<const float *>(a.beta)[i] : bf2f(static_cast<const bf16 *>(a.beta)[i]);
}
__device__ __forceinline__ void store_dbeta(const ChunkArgs &a, size_t i, float x) {
    if (a.beta_f32) static_cast<float *>(a.dbeta)[i] = x;
    else static_cast<bf16 *>(a.dbeta)[i] = f2bf(x);
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

cudaError_t launch_plan(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_prep(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_fwd_chunks(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_recompute_chunks(const ChunkArgs &a, cudaStream_t s);  // WY pass + state scan
cudaError_t launch_bwd_chunks(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_state_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_bstate_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_bintra_a_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_out_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_dvloc_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_bintra_b_tc(const ChunkArgs &a, cudaStream_t s);
cudaError_t launch_intra_tc(const ChunkArgs &a, cudaStream_t s);

cudaError_t launch_decode(int B, int H, int HV, float scale, const bf16 *q, const bf16 *k,
                          const bf16 *v, const float *g, const float *beta, float *pool,
                          int num_slots, const int32_t *idx, bf16 *o, int32_t *status,
                          cudaStream_t s, gdn_kernel_timer *timer);

}  // namespace gdn
