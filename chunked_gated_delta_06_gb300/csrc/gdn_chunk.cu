// gdn_chunk.cu -- the small CUDA-core kernels of the chunk path and the launch
// order of the forward and backward.
//
//   k_plan   chunk table from the device copy of cu_seqlens (chunks of 64
//            tokens never span sequences, the last one of a sequence may be
//            partial), "[Cake 1/13] gdn: chunked gated delta rule ...", API;
//   k_prep   q / k norms r = sqrt(sum x^2 + 1e-6) ("C6: GDN decode-step
//            goldens ...", Provider: divide by the sqrt) and the chunk-local
//            cumulative sum G of g.
// The tensor-core kernels of the chunked (WY) form live in gdn_*_tc.cu.
// Every reduction runs in a fixed order and no kernel uses atomics, so results
// are bit-identical from run to run.
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// Chunk table from the device cu_seqlens (one block).  The host sized every buffer
// from its own copy of cu_seqlens (total_chunks chunks, at most max_seq_chunks in one
// sequence, T tokens).  The device copy is accepted only when it fits those extents:
// cu[0] = 0, cu[N] = T, non-decreasing, total_chunks chunks in all and no sequence
// longer than max_seq_chunks.  Otherwise bit 1 is ORed into the caller's status word
// (when there is one) and the table written is empty (every sequence without chunks,
// every chunk of length 0), which every kernel turns into no work, so a bad device
// copy never leads to an access outside the buffers.
__global__ void k_plan(const int *__restrict__ cu, int N, int T, int total_chunks, int max_seq_chunks,
                       int *seq_off, int *chunk_start, int *chunk_len, int *seq_order, int *status) {
    __shared__ int sums[1024];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (N + nt - 1) / nt;
    const int b = min(N, tid * per), e = min(N, b + per);
    int cnt = 0;
    bool bad = tid == 0 && (cu[0] != 0 || cu[N] != T);
    for (int n = b; n < e; ++n) {
        const int L = cu[n + 1] - cu[n];
        const int ch = (max(L, 0) + kChunk - 1) / kChunk;
        bad = bad || L < 0 || ch > max_seq_chunks;
        cnt += ch;
    }
    sums[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {
        int x = tid >= off ? sums[tid - off] : 0;
        __syncthreads();
        sums[tid] += x;
        __syncthreads();
    }
    bad = __syncthreads_or(bad || sums[nt - 1] != total_chunks);
    if (bad) {
        if (tid == 0 && status) atomicOr(status, 1);
        for (int c = tid; c < total_chunks; c += nt) {
            chunk_start[c] = 0;
            chunk_len[c] = 0;
        }
        for (int n = tid; n <= N; n += nt) seq_off[n] = 0;
        for (int n = tid; n < N; n += nt) seq_order[n] = n;
        return;
    }
    // the table: chunk c of sequence n starts at cu[n] + 64 j (consecutive 64-token
    // blocks inside [0, T), the last one partial)
    int base = sums[tid] - cnt;
    for (int n = b; n < e; ++n) {
        seq_off[n] = base;
        const int L = cu[n + 1] - cu[n];
        for (int j = 0; j * kChunk < L; ++j) {
            if (!in_range(base + j, 1, total_chunks, status)) break;
            chunk_start[base + j] = cu[n] + j * kChunk;
            chunk_len[base + j] = min(kChunk, L - j * kChunk);
        }
        base += (L + kChunk - 1) / kChunk;
    }
    if (tid == nt - 1) seq_off[N] = total_chunks;
    // longest sequences first (ties by index), so the scans start the longest
    // chunk chains first; identity order beyond 4096 sequences
    for (int n = b; n < e; ++n) {
        int rank = n;
        if (N <= 4096) {
            const int Ln = cu[n + 1] - cu[n];
            rank = 0;
            for (int m = 0; m < N; ++m) {
                const int Lm = cu[m + 1] - cu[m];
                rank += (Lm > Ln || (Lm == Ln && m < n)) ? 1 : 0;
            }
        }
        if (in_range(rank, 1, N, status)) seq_order[rank] = n;
    }
}

// ---------------------------------------------------------------------------
// Norms of q and k rows and the chunk-local cumsum of g (g from the fused gate when
// the call passes its pre-activations).  grid (chunks, H).
__global__ void __launch_bounds__(kThreads) k_prep(ChunkArgs a) {
    const int c = blockIdx.x, h = blockIdx.y;
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // warp w takes rows w, w + 8, ..., w + 56: all 16 row slices (8 bytes a lane) are
    // loaded before the first sum
    constexpr int kRows = kChunk / (kThreads / 32);
    uint2 xq[kRows], xk[kRows];
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = warp + 8 * m;
        xq[m] = xk[m] = make_uint2(0u, 0u);
        if (i < L) {
            const size_t row = ((size_t)(t0 + i) * a.H + h) * kDim + lane * 4;
            if (in_range(row, 4, n_rows_h(a), a.status)) {
                xq[m] = *reinterpret_cast<const uint2 *>(a.q + row);
                xk[m] = *reinterpret_cast<const uint2 *>(a.k + row);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kRows; ++m) {
        const int i = warp + 8 * m;
        const float2 q0 = bf2_to_f2(xq[m].x), q1 = bf2_to_f2(xq[m].y);
        const float2 k0 = bf2_to_f2(xk[m].x), k1 = bf2_to_f2(xk[m].y);
        float sq = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
        float sk = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0 && i < L && in_range((size_t)(t0 + i) * a.H + h, 1, n_tok_h(a), a.status)) {
            a.rq[(size_t)(t0 + i) * a.H + h] = sqrtf(sq + kNormEps);
            a.rk[(size_t)(t0 + i) * a.H + h] = sqrtf(sk + kNormEps);
        }
    }
    const int r = a.HV / a.H;
    for (int j = warp; j < r; j += kThreads / 32) {
        const int hv = h * r + j;
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        float x0 = i0 < L ? load_g(a, (size_t)(t0 + i0) * a.HV + hv, hv) : 0.f;
        float x1 = i1 < L ? load_g(a, (size_t)(t0 + i1) * a.HV + hv, hv) : 0.f;
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        float excl = s - (x0 + x1);
        if (i0 < L && in_range((size_t)(t0 + i0) * a.HV + hv, 1, n_tok_hv(a), a.status))
            a.G[(size_t)(t0 + i0) * a.HV + hv] = excl + x0;
        if (i1 < L && in_range((size_t)(t0 + i1) * a.HV + hv, 1, n_tok_hv(a), a.status))
            a.G[(size_t)(t0 + i1) * a.HV + hv] = excl + x0 + x1;
    }
}

}  // namespace

cudaError_t launch_plan(const ChunkArgs &a, cudaStream_t s) {
    TimerScope ts(a.timer, GDN_KERNEL_PLAN, s);
    k_plan<<<1, 1024, 0, s>>>(a.cu_dev, a.N, a.T, a.num_chunks, a.max_seq_chunks, a.seq_chunk_off,
                              a.chunk_start, a.chunk_len, a.seq_order, a.status);
    return cudaGetLastError();
}

cudaError_t launch_prep(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    TimerScope ts(a.timer, GDN_KERNEL_PREP, s);
    k_prep<<<dim3(a.num_chunks, a.H), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd_chunks(const ChunkArgs &a, cudaStream_t s) {
    cudaError_t e;
    if ((e = launch_intra_tc(a, s)) != cudaSuccess) return e;
    if ((e = launch_state_tc(a, s)) != cudaSuccess) return e;
    if ((e = launch_out_tc(a, s)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_recompute_chunks(const ChunkArgs &a, cudaStream_t s) {
    cudaError_t e;
    if ((e = launch_intra_tc(a, s)) != cudaSuccess) return e;
    return launch_state_tc(a, s);  // a.ht is null: no final state
}

// Fused-gating backward, last step: dA_log[hv] and ddt_bias[hv] as sums of the
// per-chunk partials of the WY-pullback kernel.  One warp per value head: lane l
// adds the chunks c = l, l + 32, ... in order (fp64), then a fixed butterfly.
__global__ void k_gate_reduce(ChunkArgs a) {
    const int hv = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (hv >= a.HV) return;
    const float2 *part = reinterpret_cast<const float2 *>(a.gpart);
    double sa = 0.0, sd = 0.0;
    for (int c = lane; c < a.num_chunks; c += 32) {
        if (!in_range(((size_t)c * a.HV + hv) * 2, 2, (long long)a.num_chunks * a.HV * 2, a.status)) break;
        const float2 p = part[(size_t)c * a.HV + hv];
        sa += p.x;
        sd += p.y;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        sa += __shfl_xor_sync(0xffffffffu, sa, o);
        sd += __shfl_xor_sync(0xffffffffu, sd, o);
    }
    if (lane == 0) {
        a.dA_log[hv] = (float)sa;
        a.ddt_bias[hv] = (float)sd;
    }
}

cudaError_t launch_gate_reduce(const ChunkArgs &a, cudaStream_t s) {
    k_gate_reduce<<<(a.HV + 7) / 8, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunks(const ChunkArgs &a, cudaStream_t s) {
    cudaError_t e;
    if ((e = launch_dvloc_tc(a, s)) != cudaSuccess) return e;
    if ((e = launch_bstate_tc(a, s)) != cudaSuccess) return e;
    if (a.num_chunks == 0) return cudaSuccess;
    if ((e = launch_bintra_a_tc(a, s)) != cudaSuccess) return e;
    return launch_bintra_b_tc(a, s);  // ends with dk (the L2-norm backward of khat)
}

}  // namespace gdn
