// gdn_chunk_simt.cu -- chunked gated delta rule, forward and backward, as plain
// fp32 CUDA-core kernels over shared-memory tiles.
//
// The chunked (WY) form follows "Qwen3.5-397B RL trainer on 128 v7x"
// (maxtext #5799), GDN context-parallel m-scan / dh-scan commits, and the chunk
// pipeline of "cake_gdn: deterministic chunked GDN training kernels"
// (miles #3597), Summary and section 2 (norm + cumsum, WY pass, state scan,
// output; reverse state scan "dhu", "dqkwg", WY pullback).  Per chunk of
// L <= 64 tokens with h the K x V state at the chunk start, qhat / khat the
// normalised rows (scale on q only) and G the chunk-local cumsum of g:
//   A     = strict_tril(diag(beta) Khat Khat^T (.) exp(G_i - G_j))
//   Tm    = (I + A)^-1
//   w     = Tm diag(beta e^G) Khat,      u = Tm diag(beta) V
//   v_new = u - w h
//   o     = diag(e^G) Qhat h + tril(Qhat Khat^T (.) exp(G_i - G_j)) v_new
//   h'    = e^{G_L} h + (diag(e^{G_L - G}) Khat)^T v_new
// Every reduction runs in a fixed order and no kernel uses atomics, so results
// are bit-identical from run to run.
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kP = 129;  // padded pitch of 128-wide fp32 tiles
constexpr int kQ = 65;   // padded pitch of 64-wide fp32 tiles
constexpr int kSlab = 32;

// ---------------------------------------------------------------------------
// Chunk table from the device cu_seqlens (one block).  Host code computed the
// chunk count from the host copy; a mismatch sets *status.
__global__ void k_plan(const int *__restrict__ cu, int N, int T, int total_chunks, int *seq_off,
                       int *chunk_seq, int *chunk_start, int *chunk_len, int *status) {
    __shared__ int sums[1024];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (N + nt - 1) / nt;
    const int b = min(N, tid * per), e = min(N, b + per);
    int cnt = 0;
    for (int n = b; n < e; ++n) cnt += (max(cu[n + 1] - cu[n], 0) + kChunk - 1) / kChunk;
    sums[tid] = cnt;
    __syncthreads();
    for (int off = 1; off < nt; off <<= 1) {
        int x = tid >= off ? sums[tid - off] : 0;
        __syncthreads();
        sums[tid] += x;
        __syncthreads();
    }
    int base = sums[tid] - cnt;
    for (int n = b; n < e; ++n) {
        seq_off[n] = base;
        int L = max(cu[n + 1] - cu[n], 0);
        for (int j = 0; j * kChunk < L; ++j) {
            int c = base + j;
            if (c < total_chunks) {
                // clamp to [0, T): a device copy of cu_seqlens that disagrees with
                // the host copy yields empty chunks and a status flag, never an
                // out-of-bounds access
                const int st = min(max(cu[n] + j * kChunk, 0), T);
                chunk_seq[c] = n;
                chunk_start[c] = st;
                chunk_len[c] = max(0, min(min(kChunk, L - j * kChunk), T - st));
            }
        }
        base += (L + kChunk - 1) / kChunk;
    }
    __syncthreads();
    if (tid == nt - 1) {
        seq_off[N] = min(sums[tid], total_chunks);
        if (status) *status = (sums[tid] != total_chunks || cu[N] != T) ? 1 : 0;
    }
    // keep every sequence's chunk range inside [0, total_chunks]
    for (int n = b; n < e; ++n) seq_off[n] = min(seq_off[n], total_chunks);
}

// ---------------------------------------------------------------------------
// Norms of q and k rows and the chunk-local cumsum of g.  grid (chunks, H).
__global__ void __launch_bounds__(kThreads) k_prep(ChunkArgs a) {
    const int c = blockIdx.x, h = blockIdx.y;
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < L; i += kThreads / 32) {
        const size_t row = ((size_t)(t0 + i) * a.H + h) * kDim;
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float x = bf2f(a.q[row + lane * 4 + e]);
            float y = bf2f(a.k[row + lane * 4 + e]);
            sq += x * x;
            sk += y * y;
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        if (lane == 0) {
            a.rq[(size_t)(t0 + i) * a.H + h] = sqrtf(sq + kNormEps);
            a.rk[(size_t)(t0 + i) * a.H + h] = sqrtf(sk + kNormEps);
        }
    }
    const int r = a.HV / a.H;
    for (int j = warp; j < r; j += kThreads / 32) {
        const int hv = h * r + j;
        const int i0 = 2 * lane, i1 = 2 * lane + 1;
        float x0 = i0 < L ? a.g[(size_t)(t0 + i0) * a.HV + hv] : 0.f;
        float x1 = i1 < L ? a.g[(size_t)(t0 + i1) * a.HV + hv] : 0.f;
        float s = x0 + x1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        float excl = s - (x0 + x1);
        if (i0 < L) a.G[(size_t)(t0 + i0) * a.HV + hv] = excl + x0;
        if (i1 < L) a.G[(size_t)(t0 + i1) * a.HV + hv] = excl + x0 + x1;
    }
}

// Load normalised rows: dst[i][c] = mul * x[t0+i, h, c] / r[t0+i, h]  (0 past L).
__device__ void load_rows_norm(float *dst, const bf16 *x, const float *r, int t0, int L, int H,
                               int h, float mul) {
    for (int idx = threadIdx.x; idx < kChunk * kDim; idx += kThreads) {
        int i = idx >> 7, c = idx & 127;
        float val = 0.f;
        if (i < L) {
            size_t t = (size_t)(t0 + i) * H + h;
            val = mul * bf2f(x[t * kDim + c]) / r[t];
        }
        dst[i * kP + c] = val;
    }
}

// ---------------------------------------------------------------------------
// WY pass: A, Tm = (I + A)^-1, w, u.  grid (chunks, H); loops over the value
// heads of key head h so Khat Khat^T is formed once.
__global__ void __launch_bounds__(kThreads) k_intra(ChunkArgs a) {
    extern __shared__ float sm[];
    float *Kn = sm;
    float *KK = Kn + kChunk * kP;
    float *A = KK + kChunk * kQ;
    float *Tm = A + kChunk * kQ;
    float *Gs = Tm + kChunk * kQ;
    float *bs = Gs + kChunk;
    float *ws = bs + kChunk;
    const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const int r = a.HV / a.H;
    load_rows_norm(Kn, a.k, a.rk, t0, L, a.H, h, 1.f);
    __syncthreads();
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float s = 0.f;
        for (int e = 0; e < kDim; ++e) s += Kn[i * kP + e] * Kn[j * kP + e];
        KK[i * kQ + j] = s;
    }
    for (int jv = 0; jv < r; ++jv) {
        const int hv = h * r + jv;
        __syncthreads();
        if (tid < kChunk) {
            bool in = tid < L;
            float gg = in ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
            float bb = in ? bf2f(a.beta[(size_t)(t0 + tid) * a.HV + hv]) : 0.f;
            Gs[tid] = gg;
            bs[tid] = bb;
            ws[tid] = in ? bb * expf(gg) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
            int i = idx >> 6, j = idx & 63;
            A[i * kQ + j] = (j < i && i < L) ? bs[i] * KK[i * kQ + j] * expf(Gs[i] - Gs[j]) : 0.f;
        }
        __syncthreads();
        if (tid < kChunk) {  // column j of the inverse by forward substitution
            const int j = tid;
            for (int i = 0; i < kChunk; ++i) {
                float x;
                if (i < j || i >= L) x = 0.f;
                else if (i == j) x = 1.f;
                else {
                    x = 0.f;
                    for (int m = j; m < i; ++m) x -= A[i * kQ + m] * Tm[m * kQ + j];
                }
                Tm[i * kQ + j] = x;
            }
        }
        __syncthreads();
        for (int idx = tid; idx < L * kDim; idx += kThreads) {
            int i = idx >> 7, e = idx & 127;
            float sw = 0.f, su = 0.f;
            for (int j = 0; j <= i; ++j) {
                float t = Tm[i * kQ + j];
                sw += t * ws[j] * Kn[j * kP + e];
                su += t * bs[j] * bf2f(a.v[((size_t)(t0 + j) * a.HV + hv) * kDim + e]);
            }
            size_t o = ((size_t)(t0 + i) * a.HV + hv) * kDim + e;
            a.w[o] = f2bf(sw);
            a.u[o] = f2bf(su);
        }
        float *Tdst = a.Tm + ((size_t)c * a.HV + hv) * kChunk * kChunk;
        for (int idx = tid; idx < kChunk * kChunk; idx += kThreads)
            Tdst[idx] = Tm[(idx >> 6) * kQ + (idx & 63)];
    }
}

// M[i][j] = (Qn_i . Kn_j) exp(G_i - G_j) for j <= i < L, else 0.
__device__ void build_M(float *M, const float *Qn, const float *Kn, const float *Gs, int L) {
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float s = 0.f;
        if (j <= i && i < L) {
            for (int e = 0; e < kDim; ++e) s += Qn[i * kP + e] * Kn[j * kP + e];
            s *= expf(Gs[i] - Gs[j]);
        }
        M[i * kQ + j] = s;
    }
}

// ---------------------------------------------------------------------------
// Output.  grid (chunks, HV).
__global__ void __launch_bounds__(kThreads) k_out(ChunkArgs a) {
    extern __shared__ float sm[];
    float *Qn = sm;
    float *Kn = Qn + kChunk * kP;
    float *Vn = Kn + kChunk * kP;
    float *M = Vn + kChunk * kP;
    float *Gs = M + kChunk * kQ;
    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    load_rows_norm(Qn, a.q, a.rq, t0, L, a.H, h, a.scale);
    load_rows_norm(Kn, a.k, a.rk, t0, L, a.H, h, 1.f);
    for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
        int i = idx >> 7, e = idx & 127;
        Vn[i * kP + e] = i < L ? bf2f(a.vnew[((size_t)(t0 + i) * a.HV + hv) * kDim + e]) : 0.f;
    }
    if (tid < kChunk) Gs[tid] = tid < L ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
    __syncthreads();
    build_M(M, Qn, Kn, Gs, L);
    __syncthreads();
    const bf16 *hc = a.hc + ((size_t)c * a.HV + hv) * kDim * kDim;
    for (int idx = tid; idx < L * kDim; idx += kThreads) {
        int i = idx >> 7, e = idx & 127;
        float inter = 0.f;
        for (int r = 0; r < kDim; ++r) inter += Qn[i * kP + r] * bf2f(hc[(size_t)r * kDim + e]);
        float s = expf(Gs[i]) * inter;
        for (int j = 0; j <= i; ++j) s += M[i * kQ + j] * Vn[j * kP + e];
        a.o[((size_t)(t0 + i) * a.HV + hv) * kDim + e] = f2bf(s);
    }
}

// ---------------------------------------------------------------------------
// Backward, step 1: dv_local = tril(M)^T dO.  grid (chunks, HV).
__global__ void __launch_bounds__(kThreads) k_dvloc(ChunkArgs a) {
    extern __shared__ float sm[];
    float *Qn = sm;
    float *Kn = Qn + kChunk * kP;
    float *dO = Kn + kChunk * kP;
    float *M = dO + kChunk * kP;
    float *Gs = M + kChunk * kQ;
    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    load_rows_norm(Qn, a.q, a.rq, t0, L, a.H, h, a.scale);
    load_rows_norm(Kn, a.k, a.rk, t0, L, a.H, h, 1.f);
    for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
        int i = idx >> 7, e = idx & 127;
        dO[i * kP + e] = i < L ? bf2f(a.d_o[((size_t)(t0 + i) * a.HV + hv) * kDim + e]) : 0.f;
    }
    if (tid < kChunk) Gs[tid] = tid < L ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
    __syncthreads();
    build_M(M, Qn, Kn, Gs, L);
    __syncthreads();
    for (int idx = tid; idx < L * kDim; idx += kThreads) {
        int j = idx >> 7, e = idx & 127;
        float s = 0.f;
        for (int i = j; i < L; ++i) s += M[i * kQ + j] * dO[i * kP + e];
        a.dvloc[((size_t)(t0 + j) * a.HV + hv) * kDim + e] = s;
    }
}

// ---------------------------------------------------------------------------
// Backward, step 5: sum the per-value-head gradients of qhat / khat over the
// HV / H value heads of each key head (fixed order) and apply the L2-norm
// backward dx = (dn - n (n . dn)) / r.  One warp per (token, key head).
__global__ void __launch_bounds__(kThreads) k_bnorm(ChunkArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t item = (size_t)blockIdx.x * (kThreads / 32) + warp;
    if (item >= (size_t)a.T * a.H) return;
    const int t = (int)(item / a.H), h = (int)(item % a.H);
    const int r = a.HV / a.H;
    float dq[4] = {0, 0, 0, 0}, dk[4] = {0, 0, 0, 0}, xq[4], xk[4];
    for (int j = 0; j < r; ++j) {
        const size_t o = ((size_t)t * a.HV + h * r + j) * kDim + lane * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            dq[u] += a.dqp[o + u];
            dk[u] += a.dkp[o + u];
        }
    }
    const size_t row = ((size_t)t * a.H + h) * kDim + lane * 4;
    const float rq = a.rq[(size_t)t * a.H + h], rk = a.rk[(size_t)t * a.H + h];
    float nq = 0.f, nk = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        xq[u] = bf2f(a.q[row + u]) / rq;
        xk[u] = bf2f(a.k[row + u]) / rk;
        dq[u] *= a.scale;
        nq += xq[u] * dq[u];
        nk += xk[u] * dk[u];
    }
    nq = warp_sum(nq);
    nk = warp_sum(nk);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        a.dq[row + u] = f2bf((dq[u] - xq[u] * nq) / rq);
        a.dk[row + u] = f2bf((dk[u] - xk[u] * nk) / rk);
    }
}

template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

constexpr size_t kSmemIntra = sizeof(float) * (kChunk * kP + 3 * kChunk * kQ + 3 * kChunk);
constexpr size_t kSmemOut = sizeof(float) * (3 * kChunk * kP + kChunk * kQ + kChunk);

}  // namespace

cudaError_t launch_plan(const ChunkArgs &a, cudaStream_t s) {
    TimerScope ts(a.timer, GDN_KERNEL_PLAN, s);
    k_plan<<<1, 1024, 0, s>>>(a.cu_dev, a.N, a.T, a.num_chunks, a.seq_chunk_off, a.chunk_seq,
                              a.chunk_start, a.chunk_len, a.status);
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

cudaError_t launch_bwd_chunks(const ChunkArgs &a, cudaStream_t s) {
    cudaError_t e;
    if ((e = launch_dvloc_tc(a, s)) != cudaSuccess) return e;
    if ((e = launch_bstate_tc(a, s)) != cudaSuccess) return e;
    if (a.num_chunks == 0) return cudaSuccess;
    if ((e = launch_bintra_a_tc(a, s)) != cudaSuccess) return e;
    if ((e = launch_bintra_b_tc(a, s)) != cudaSuccess) return e;
    {
        const size_t items = (size_t)a.T * a.H;
        const unsigned blocks = (unsigned)((items + kThreads / 32 - 1) / (kThreads / 32));
        TimerScope ts(a.timer, GDN_KERNEL_BNORM, s);
        k_bnorm<<<blocks, kThreads, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
