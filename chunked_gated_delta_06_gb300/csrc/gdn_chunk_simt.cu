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
__global__ void k_plan(const int *__restrict__ cu, int N, int total_chunks, int *seq_off,
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
                chunk_seq[c] = n;
                chunk_start[c] = cu[n] + j * kChunk;
                chunk_len[c] = min(kChunk, L - j * kChunk);
            }
        }
        base += (L + kChunk - 1) / kChunk;
    }
    if (tid == nt - 1) {
        seq_off[N] = sums[tid];
        if (status) *status = (sums[tid] != total_chunks) ? 1 : 0;
    }
}

// ---------------------------------------------------------------------------
// Norms of q and k rows and the chunk-local cumsum of g.  grid (chunks, H).
__global__ void __launch_bounds__(kThreads) k_prep(ChunkArgs a) {
    const int c = blockIdx.x, h = blockIdx.y;
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
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

// ---------------------------------------------------------------------------
// Forward state scan.  grid (N, HV, V / 32): one 128 x 32 slab of the fp32
// state per block, sequential over the sequence's chunks.
__global__ void __launch_bounds__(kThreads) k_state(ChunkArgs a) {
    extern __shared__ float sm[];
    float *hs = sm;                 // [128][33]
    float *vn = hs + kDim * 33;     // [64][33]
    float *kt = vn + kChunk * 33;   // [64][129]
    const int n = blockIdx.x, hv = blockIdx.y, v0 = blockIdx.z * kSlab, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim;
    for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
        int r = idx >> 5, j = idx & 31;
        hs[r * 33 + j] = a.h0 ? a.h0[sbase + (size_t)r * kDim + v0 + j] : 0.f;
    }
    __syncthreads();
    const int cb = a.seq_chunk_off[n], ce = a.seq_chunk_off[n + 1];
    for (int c = cb; c < ce; ++c) {
        const int t0 = a.chunk_start[c], L = a.chunk_len[c];
        bf16 *hdst = a.hc + ((size_t)c * a.HV + hv) * kDim * kDim;
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            hdst[(size_t)r * kDim + v0 + j] = f2bf(hs[r * 33 + j]);
        }
        for (int idx = tid; idx < L * kSlab; idx += kThreads) {
            int i = idx >> 5, j = idx & 31;
            size_t row = ((size_t)(t0 + i) * a.HV + hv) * kDim;
            float s = bf2f(a.u[row + v0 + j]);
            for (int e = 0; e < kDim; ++e) s -= bf2f(a.w[row + e]) * hs[e * 33 + j];
            vn[i * 33 + j] = s;
            a.vnew[row + v0 + j] = f2bf(s);
        }
        const float Gl = a.G[(size_t)(t0 + L - 1) * a.HV + hv];
        for (int idx = tid; idx < L * kDim; idx += kThreads) {
            int i = idx >> 7, e = idx & 127;
            size_t t = (size_t)(t0 + i) * a.H + h;
            kt[i * kP + e] = expf(Gl - a.G[(size_t)(t0 + i) * a.HV + hv]) / a.rk[t] *
                             bf2f(a.k[t * kDim + e]);
        }
        __syncthreads();
        const float egl = expf(Gl);
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            float s = egl * hs[r * 33 + j];
            for (int i = 0; i < L; ++i) s += kt[i * kP + r] * vn[i * 33 + j];
            hs[r * 33 + j] = s;
        }
        __syncthreads();
    }
    if (a.ht) {
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            a.ht[sbase + (size_t)r * kDim + v0 + j] = hs[r * 33 + j];
        }
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

// Backward, step 2: reverse state scan ("dhu").  grid (N, HV, V / 32).
//   dv_new = dv_local + Ktil dh',  Ktil_i = exp(G_L - G_i) khat_i
//   dh     = e^{G_L} dh' + Qtil^T dO - w^T dv_new,  Qtil_i = e^{G_i} qhat_i
__global__ void __launch_bounds__(kThreads) k_bstate(ChunkArgs a) {
    extern __shared__ float sm[];
    float *dh = sm;                  // [128][33]
    float *dvn = dh + kDim * 33;     // [64][33]
    float *dos = dvn + kChunk * 33;  // [64][33]
    float *kt = dos + kChunk * 33;   // [64][129]
    float *qt = kt + kChunk * kP;    // [64][129]
    const int n = blockIdx.x, hv = blockIdx.y, v0 = blockIdx.z * kSlab, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim;
    for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
        int r = idx >> 5, j = idx & 31;
        dh[r * 33 + j] = a.d_ht ? a.d_ht[sbase + (size_t)r * kDim + v0 + j] : 0.f;
    }
    __syncthreads();
    const int cb = a.seq_chunk_off[n], ce = a.seq_chunk_off[n + 1];
    for (int c = ce - 1; c >= cb; --c) {
        const int t0 = a.chunk_start[c], L = a.chunk_len[c];
        bf16 *ddst = a.dhc + ((size_t)c * a.HV + hv) * kDim * kDim;
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            ddst[(size_t)r * kDim + v0 + j] = f2bf(dh[r * 33 + j]);
        }
        const float Gl = a.G[(size_t)(t0 + L - 1) * a.HV + hv];
        for (int idx = tid; idx < L * kDim; idx += kThreads) {
            int i = idx >> 7, e = idx & 127;
            size_t t = (size_t)(t0 + i) * a.H + h;
            float Gi = a.G[(size_t)(t0 + i) * a.HV + hv];
            kt[i * kP + e] = expf(Gl - Gi) / a.rk[t] * bf2f(a.k[t * kDim + e]);
            qt[i * kP + e] = expf(Gi) * a.scale / a.rq[t] * bf2f(a.q[t * kDim + e]);
        }
        for (int idx = tid; idx < L * kSlab; idx += kThreads) {
            int i = idx >> 5, j = idx & 31;
            dos[i * 33 + j] = bf2f(a.d_o[((size_t)(t0 + i) * a.HV + hv) * kDim + v0 + j]);
        }
        __syncthreads();
        for (int idx = tid; idx < L * kSlab; idx += kThreads) {
            int i = idx >> 5, j = idx & 31;
            size_t row = ((size_t)(t0 + i) * a.HV + hv) * kDim;
            float s = a.dvloc[row + v0 + j];
            for (int e = 0; e < kDim; ++e) s += kt[i * kP + e] * dh[e * 33 + j];
            dvn[i * 33 + j] = s;
            a.dvnew[row + v0 + j] = s;
        }
        __syncthreads();
        const float egl = expf(Gl);
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            float s = egl * dh[r * 33 + j];
            for (int i = 0; i < L; ++i) {
                float wv = bf2f(a.w[((size_t)(t0 + i) * a.HV + hv) * kDim + r]);
                s += qt[i * kP + r] * dos[i * 33 + j] - wv * dvn[i * 33 + j];
            }
            dh[r * 33 + j] = s;
        }
        __syncthreads();
    }
    if (a.dh0) {
        for (int idx = tid; idx < kDim * kSlab; idx += kThreads) {
            int r = idx >> 5, j = idx & 31;
            a.dh0[sbase + (size_t)r * kDim + v0 + j] = dh[r * 33 + j];
        }
    }
}

// Deterministic block sum (fixed tree) of one float per thread.
__device__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float s = 0.f;
    if (threadIdx.x == 0) {
        for (int w = 0; w < kThreads / 32; ++w) s += red[w];
        red[kThreads / 32] = s;
    }
    __syncthreads();
    return red[kThreads / 32];
}

// ---------------------------------------------------------------------------
// Backward, step 3 ("dqkwg", the terms with h and dh').  grid (chunks, HV).
//   dqhat_i  = e^{G_i} dO_i h^T                        -> dqp
//   dW       = -dv_new h^T                             -> dW
//   dKtil_j  = v_new_j dh'^T; dkhat_j = e^{G_L-G_j} dKtil_j  -> dkp
//   dG_i    += qhat_i . dqhat_i
//   dG_j    -= xi_j,  dG_L += sum_j xi_j + e^{G_L} <h, dh'>,  xi_j = khat_j . dkhat_j
__global__ void __launch_bounds__(kThreads) k_bintra_a(ChunkArgs a) {
    extern __shared__ float sm[];
    float *dO = sm;                  // [64][129]
    float *dvn = dO + kChunk * kP;   // [64][129]
    float *vn = dvn + kChunk * kP;   // [64][129]
    float *Gs = vn + kChunk * kP;    // [64]
    float *dG = Gs + kChunk;         // [64]
    float *red = dG + kChunk;        // [9]
    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
        int i = idx >> 7, e = idx & 127;
        size_t o = ((size_t)(t0 + i) * a.HV + hv) * kDim + e;
        bool in = i < L;
        dO[i * kP + e] = in ? bf2f(a.d_o[o]) : 0.f;
        dvn[i * kP + e] = in ? a.dvnew[o] : 0.f;
        vn[i * kP + e] = in ? bf2f(a.vnew[o]) : 0.f;
    }
    if (tid < kChunk) Gs[tid] = tid < L ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
    __syncthreads();
    const bf16 *hc = a.hc + ((size_t)c * a.HV + hv) * kDim * kDim;
    const bf16 *dhc = a.dhc + ((size_t)c * a.HV + hv) * kDim * kDim;
    const float Gl = Gs[L - 1];
    // thread -> (i = idx % 64, r = idx / 64): h / dh' rows r are warp-uniform
    for (int idx = tid; idx < kChunk * kDim; idx += kThreads) {
        int i = idx & 63, r = idx >> 6;
        if (i >= L) continue;
        float sq = 0.f, sw = 0.f, sk = 0.f;
        for (int e = 0; e < kDim; ++e) {
            float hv_ = bf2f(hc[(size_t)r * kDim + e]);
            float dh_ = bf2f(dhc[(size_t)r * kDim + e]);
            sq += dO[i * kP + e] * hv_;
            sw += dvn[i * kP + e] * hv_;
            sk += vn[i * kP + e] * dh_;
        }
        size_t o = ((size_t)(t0 + i) * a.HV + hv) * kDim + r;
        a.dqp[o] = expf(Gs[i]) * sq;
        a.dW[o] = -sw;
        a.dkp[o] = expf(Gl - Gs[i]) * sk;
    }
    // <h, dh'>
    float part = 0.f;
    for (int idx = tid; idx < kDim * kDim; idx += kThreads) part += bf2f(hc[idx]) * bf2f(dhc[idx]);
    float hdh = block_sum(part, red);  // includes __syncthreads: dqp / dkp visible
    if (tid < kChunk) {
        const int i = tid;
        float dg = 0.f, xi = 0.f;
        if (i < L) {
            size_t t = (size_t)(t0 + i) * a.H + h;
            size_t o = ((size_t)(t0 + i) * a.HV + hv) * kDim;
            float qi = 0.f;
            const float qs = a.scale / a.rq[t], ks = 1.f / a.rk[t];
            for (int e = 0; e < kDim; ++e) {
                qi += bf2f(a.q[t * kDim + e]) * qs * a.dqp[o + e];
                xi += bf2f(a.k[t * kDim + e]) * ks * a.dkp[o + e];
            }
            dg = qi - xi;
            a.dGp[(size_t)(t0 + i) * a.HV + hv] = dg;
        }
        dG[i] = xi;  // 0 past L
    }
    __syncthreads();
    if (tid == 0) {
        float sx = 0.f;
        for (int i = 0; i < L; ++i) sx += dG[i];
        size_t o = (size_t)(t0 + L - 1) * a.HV + hv;
        a.dGp[o] += sx + expf(Gl) * hdh;
    }
}

// ---------------------------------------------------------------------------
// Backward, step 4 (the intra-chunk terms and the WY pullback).  grid (chunks, HV).
__global__ void __launch_bounds__(kThreads) k_bintra_b(ChunkArgs a) {
    extern __shared__ float sm[];
    float *Qn = sm;                    // [64][129]
    float *Kn = Qn + kChunk * kP;      // [64][129]
    float *Tm = Kn + kChunk * kP;      // [64][65]
    float *dMG = Tm + kChunk * kQ;     // [64][65]  dM (.) Gamma, j <= i
    float *P = dMG + kChunk * kQ;      // [64][65]  work
    float *dT = P + kChunk * kQ;       // [64][65]
    float *B = dT + kChunk * kQ;       // [64][65]  dA (.) beta_i Gamma, j < i
    float *Gs = B + kChunk * kQ;       // [64]
    float *bs = Gs + kChunk;           // [64]
    float *dG = bs + kChunk;           // [64]
    float *dbs = dG + kChunk;          // [64]
    const int c = blockIdx.x, hv = blockIdx.y, tid = threadIdx.x;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    load_rows_norm(Qn, a.q, a.rq, t0, L, a.H, h, a.scale);
    load_rows_norm(Kn, a.k, a.rk, t0, L, a.H, h, 1.f);
    const float *Tsrc = a.Tm + ((size_t)c * a.HV + hv) * kChunk * kChunk;
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads)
        Tm[(idx >> 6) * kQ + (idx & 63)] = Tsrc[idx];
    if (tid < kChunk) {
        bool in = tid < L;
        Gs[tid] = in ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
        bs[tid] = in ? bf2f(a.beta[(size_t)(t0 + tid) * a.HV + hv]) : 0.f;
        dG[tid] = in ? a.dGp[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
        dbs[tid] = 0.f;
    }
    __syncthreads();
    auto rowv = [&](const bf16 *base, int i) { return base + ((size_t)(t0 + i) * a.HV + hv) * kDim; };
    auto rowf = [&](const float *base, int i) { return base + ((size_t)(t0 + i) * a.HV + hv) * kDim; };
    // dM (.) Gamma and P1 = dM (.) M
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float dmg = 0.f, p1 = 0.f;
        if (j <= i && i < L) {
            const bf16 *dOi = rowv(a.d_o, i), *vj = rowv(a.vnew, j);
            float dm = 0.f, qk = 0.f;
            for (int e = 0; e < kDim; ++e) {
                dm += bf2f(dOi[e]) * bf2f(vj[e]);
                qk += Qn[i * kP + e] * Kn[j * kP + e];
            }
            float gam = expf(Gs[i] - Gs[j]);
            dmg = dm * gam;
            p1 = dm * qk * gam;
        }
        dMG[i * kQ + j] = dmg;
        P[i * kQ + j] = p1;
    }
    // dT (strictly lower) = dW_i . Wt_j + dv_new_i . Ut_j
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float s = 0.f;
        if (j < i && i < L) {
            const float *dWi = rowf(a.dW, i), *dvi = rowf(a.dvnew, i);
            const bf16 *vj = rowv(a.v, j);
            float s1 = 0.f, s2 = 0.f;
            for (int e = 0; e < kDim; ++e) {
                s1 += dWi[e] * Kn[j * kP + e];
                s2 += dvi[e] * bf2f(vj[e]);
            }
            s = bs[j] * (expf(Gs[j]) * s1 + s2);
        }
        dT[i * kQ + j] = s;
    }
    __syncthreads();
    if (tid < kChunk) {  // dG from P1: row sums minus column sums
        const int i = tid;
        float s = 0.f;
        for (int j = 0; j < kChunk; ++j) s += P[i * kQ + j] - P[j * kQ + i];
        dG[i] += s;
    }
    // X = dT Tm^T  (into B temporarily):  X_aj = sum_b dT_ab Tm_jb
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int r = idx >> 6, j = idx & 63;
        float s = 0.f;
        for (int b = 0; b < kChunk; ++b) s += dT[r * kQ + b] * Tm[j * kQ + b];
        B[r * kQ + j] = s;
    }
    __syncthreads();
    // dA_ij = -sum_r Tm_ri X_rj, strictly lower; then B = dA (.) beta_i Gamma, P2 = dA (.) A
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float da = 0.f;
        if (j < i && i < L) {
            for (int r = i; r < L; ++r) da -= Tm[r * kQ + i] * B[r * kQ + j];
        }
        dT[i * kQ + j] = da;  // dT now holds dA
    }
    __syncthreads();
    for (int idx = tid; idx < kChunk * kChunk; idx += kThreads) {
        int i = idx >> 6, j = idx & 63;
        float b = 0.f, p2 = 0.f;
        if (j < i && i < L) {
            float kk = 0.f;
            for (int e = 0; e < kDim; ++e) kk += Kn[i * kP + e] * Kn[j * kP + e];
            float gam = expf(Gs[i] - Gs[j]);
            float da = dT[i * kQ + j];
            b = da * bs[i] * gam;
            p2 = da * kk * gam;  // dA_ij * (A_ij / beta_i)
        }
        B[i * kQ + j] = b;
        P[i * kQ + j] = p2;
    }
    __syncthreads();
    if (tid < kChunk) {
        const int i = tid;
        float rs = 0.f, cs = 0.f;
        for (int j = 0; j < kChunk; ++j) {
            rs += P[i * kQ + j];
            cs += bs[j] * P[j * kQ + i];
        }
        dbs[i] += rs;                 // d beta_i from A
        dG[i] += bs[i] * rs - cs;     // P2 = dA (.) A: row sums minus column sums
    }
    __syncthreads();
    // per-row outputs: warp w takes rows m = w, w + 8, ...; lane takes 4 columns
    const int warp = tid >> 5, lane = tid & 31;
    for (int m = warp; m < L; m += kThreads / 32) {
        float sk = 0.f, su = 0.f;
        const float egm = expf(Gs[m]);
        float dq[4], dk[4], dv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = lane * 4 + u;
            float q_ = 0.f, k_ = 0.f, wt = 0.f, ut = 0.f;
            for (int j = 0; j <= m; ++j) {
                q_ += dMG[m * kQ + j] * Kn[j * kP + e];
                k_ += B[m * kQ + j] * Kn[j * kP + e];
            }
            for (int i = m; i < L; ++i) {
                k_ += dMG[i * kQ + m] * Qn[i * kP + e] + B[i * kQ + m] * Kn[i * kP + e];
                const float t = Tm[i * kQ + m];
                wt += t * rowf(a.dW, i)[e];
                ut += t * rowf(a.dvnew, i)[e];
            }
            k_ += bs[m] * egm * wt;
            sk += Kn[m * kP + e] * wt;
            su += bf2f(rowv(a.v, m)[e]) * ut;
            dq[u] = q_;
            dk[u] = k_;
            dv[u] = bs[m] * ut;
        }
        sk = warp_sum(sk);
        su = warp_sum(su);
        const size_t o = ((size_t)(t0 + m) * a.HV + hv) * kDim + lane * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            a.dqp[o + u] += dq[u];
            a.dkp[o + u] += dk[u];
            a.dv[o + u] = f2bf(dv[u]);
        }
        if (lane == 0) {
            dbs[m] += egm * sk + su;
            dG[m] += bs[m] * egm * sk;
        }
    }
    __syncthreads();
    if (tid == 0) {  // dg = reverse cumsum of dG within the chunk
        float acc = 0.f;
        for (int i = L - 1; i >= 0; --i) {
            acc += dG[i];
            a.dg[(size_t)(t0 + i) * a.HV + hv] = acc;
            a.dbeta[(size_t)(t0 + i) * a.HV + hv] = f2bf(dbs[i]);
        }
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
constexpr size_t kSmemState = sizeof(float) * (kDim * 33 + kChunk * 33 + kChunk * kP);
constexpr size_t kSmemOut = sizeof(float) * (3 * kChunk * kP + kChunk * kQ + kChunk);
constexpr size_t kSmemBstate = sizeof(float) * (kDim * 33 + 2 * kChunk * 33 + 2 * kChunk * kP);
constexpr size_t kSmemBa = sizeof(float) * (3 * kChunk * kP + 2 * kChunk + 16);
constexpr size_t kSmemBb = sizeof(float) * (2 * kChunk * kP + 5 * kChunk * kQ + 4 * kChunk);

}  // namespace

cudaError_t launch_plan(const ChunkArgs &a, cudaStream_t s) {
    TimerScope ts(a.timer, GDN_KERNEL_PLAN, s);
    k_plan<<<1, 1024, 0, s>>>(a.cu_dev, a.N, a.num_chunks, a.seq_chunk_off, a.chunk_seq,
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
    if ((e = set_smem(k_intra, kSmemIntra)) != cudaSuccess) return e;
    if ((e = set_smem(k_state, kSmemState)) != cudaSuccess) return e;
    if ((e = set_smem(k_out, kSmemOut)) != cudaSuccess) return e;
    if (a.num_chunks > 0) {
        TimerScope ts(a.timer, GDN_KERNEL_INTRA, s);
        k_intra<<<dim3(a.num_chunks, a.H), kThreads, kSmemIntra, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        TimerScope ts(a.timer, GDN_KERNEL_STATE, s);
        k_state<<<dim3(a.N, a.HV, kDim / kSlab), kThreads, kSmemState, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.num_chunks > 0) {
        TimerScope ts(a.timer, GDN_KERNEL_OUT, s);
        k_out<<<dim3(a.num_chunks, a.HV), kThreads, kSmemOut, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bwd_chunks(const ChunkArgs &a, cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem(k_dvloc, kSmemOut)) != cudaSuccess) return e;
    if ((e = set_smem(k_bstate, kSmemBstate)) != cudaSuccess) return e;
    if ((e = set_smem(k_bintra_a, kSmemBa)) != cudaSuccess) return e;
    if ((e = set_smem(k_bintra_b, kSmemBb)) != cudaSuccess) return e;
    if (a.num_chunks > 0) {
        TimerScope ts(a.timer, GDN_KERNEL_DVLOC, s);
        k_dvloc<<<dim3(a.num_chunks, a.HV), kThreads, kSmemOut, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
        k_bstate<<<dim3(a.N, a.HV, kDim / kSlab), kThreads, kSmemBstate, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.num_chunks == 0) return cudaSuccess;
    {
        TimerScope ts(a.timer, GDN_KERNEL_BINTRA_A, s);
        k_bintra_a<<<dim3(a.num_chunks, a.HV), kThreads, kSmemBa, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        TimerScope ts(a.timer, GDN_KERNEL_BINTRA_B, s);
        k_bintra_b<<<dim3(a.num_chunks, a.HV), kThreads, kSmemBb, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
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
