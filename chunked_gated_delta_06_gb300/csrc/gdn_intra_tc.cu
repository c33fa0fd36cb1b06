// gdn_intra_tc.cu -- WY pass of a chunk on the tensor cores ("WY pass" of
// "cake_gdn: deterministic chunked GDN training kernels", section 2; the
// chunk form of the GDN context-parallel scans in "Qwen3.5-397B RL trainer on
// 128 v7x", maxtext #5799).
//
// One CTA of 128 threads per (chunk, key head); it walks the HV/H value heads
// of the key head.  With Khat = diag(1 / r_k) K and Gamma_ij = exp(G_i - G_j):
//   KK = K K^T                                   (tcgen05, M=64 N=64 K=128, once)
//   A  = strict_tril(diag(beta) KKhat (.) Gamma) (CUDA cores, fp32)
//   T  = (I + A)^-1                              (fp32, recursive 2x2 blocking:
//        8x8 diagonal blocks by substitution, then T21 = -T22 (A21 T11) at block
//        sizes 8, 16 and 32)
//   w  = (T diag(beta e^G / r_k)) K,  u = (T diag(beta)) V
//                                                (tcgen05, M=64 N=128 K=64; K and
//                                                 V are raw MN-major TMA tiles)
// w and u go to HBM in bf16, T in fp32 (kept for the backward).  M=64 results
// sit in TMEM lanes 32 (m / 16) + m % 16: lanes 0..15 of warp w own rows
// 16w..16w+15.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 256;   // two warpgroups share the 128 TMEM lanes
constexpr uint32_t kHalf = 64 * 128;
constexpr uint32_t kTile = 2 * kHalf;
constexpr int kF = 65;

struct IntraSmem {
    unsigned char k[kTile];
    unsigned char v[2][kTile];     // double-buffered value tiles
    unsigned char op_w[kHalf];     // T_ij beta_j e^{G_j} / r_k,j  [i][j] K-major
    unsigned char op_u[kHalf];     // T_ij beta_j                  [i][j] K-major
    float A[64 * kF];
    float T[64 * kF];
    float X[64 * kF];
    float G[64], beta[64], wc[64], rk[64];
    uint64_t k_bar, v_bar[2], mma_bar;
    uint32_t tmem_base;
};

struct IntraMaps {
    CUtensorMap k, v;
};

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// T = (I + A)^-1 for a strictly lower A (64 x 64, rows/cols >= L are zero).
// All 128 threads take part.
__device__ void tri_inverse(const float *A, float *T, float *X) {
    const int tid = threadIdx.x;
    for (int idx = tid; idx < 64 * 64; idx += kThr) T[(idx >> 6) * kF + (idx & 63)] = 0.f;
    __syncthreads();
    if (tid < 64) {  // 8 diagonal 8x8 blocks, one column per thread
        const int b = tid >> 3, cc = tid & 7, base = b * 8;
        float col[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float x = (r == cc) ? 1.f : 0.f;
            if (r > cc) {
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m >= cc && m < r) x -= A[(base + r) * kF + base + m] * col[m];
            }
            col[r] = x;
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) T[(base + r) * kF + base + cc] = col[r];
    }
    __syncthreads();
    for (int s = 8; s < 64; s *= 2) {
        // for every merged block p of size 2s: X = A21 T11, then T21 = -T22 X
        const int nb = 64 / (2 * s), ent = nb * s * s;
        for (int e = tid; e < ent; e += kThr) {
            const int p = e / (s * s), rr = (e / s) % s, cc = e % s;
            const int r0 = p * 2 * s + s, c0 = p * 2 * s;
            float acc = 0.f;
            for (int m = cc; m < s; ++m) acc += A[(r0 + rr) * kF + c0 + m] * T[(c0 + m) * kF + c0 + cc];
            X[(r0 + rr) * kF + c0 + cc] = acc;
        }
        __syncthreads();
        for (int e = tid; e < ent; e += kThr) {
            const int p = e / (s * s), rr = (e / s) % s, cc = e % s;
            const int r0 = p * 2 * s + s, c0 = p * 2 * s;
            float acc = 0.f;
            for (int m = 0; m <= rr; ++m) acc += T[(r0 + rr) * kF + r0 + m] * X[(r0 + m) * kF + c0 + cc];
            T[(r0 + rr) * kF + c0 + cc] = -acc;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThr, 1) k_intra_tc(const ChunkArgs a,
                                                      const __grid_constant__ IntraMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    IntraSmem &sm = *reinterpret_cast<IntraSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                   ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y;
    const int r = a.HV / a.H;
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const bool active = lane < 16;
    const int grp = warp >> 2;              // warpgroup: which half of the columns
    const int row = (warp & 3) * 16 + lane;

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.k_bar, 1);
        mbar_init(&sm.v_bar[0], 1);
        mbar_init(&sm.v_bar[1], 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.k_bar, kTile);
        tma_load_3d(sm.k, &maps.k, 0, h, t0, &sm.k_bar);
        tma_load_3d(sm.k + kHalf, &maps.k, 64, h, t0, &sm.k_bar);
        mbar_arrive_expect_tx(&sm.v_bar[0], kTile);
        tma_load_3d(sm.v[0], &maps.v, 0, h * r, t0, &sm.v_bar[0]);
        tma_load_3d(sm.v[0] + kHalf, &maps.v, 64, h * r, t0, &sm.v_bar[0]);
    }
    if (tid < 64) sm.rk[tid] = tid < L ? a.rk[(size_t)(t0 + tid) * a.H + h] : 1.f;
    bool ok = __syncthreads_and(mbar_wait(&sm.k_bar, 0));
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t mphase = 0;
    if (tid == 0 && ok) {  // KK = K K^T into columns 0..63
        tc_fence_after();
        const uint32_t ks = smem_u32(sm.k);
        const uint32_t id = idesc_bf16(64, 64, 0, 0);
        for (int s = 0; s < 8; ++s) {
            const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
            mma_bf16(tb, sdesc(ks + off, 16, 1024), sdesc(ks + off, 16, 1024), id, s > 0);
        }
        mma_commit(&sm.mma_bar);
    }
    ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, mphase));
    mphase ^= 1;
    tc_fence_after();
    // KKhat row i, columns [32 grp, 32 grp + 32), stays in registers for all value heads
    float kk[32];
    if (ok) {
        tmem_ld32(t_row + grp * 32, kk);
        tmem_ld_wait();
        if (active) {
#pragma unroll
            for (int j = 0; j < 32; ++j) kk[j] /= (sm.rk[row] * sm.rk[grp * 32 + j]);
        }
    }
    for (int jv = 0; jv < r && ok; ++jv) {
        const int hv = h * r + jv, vb = jv & 1;
        if (tid == 0 && jv + 1 < r) {  // prefetch the next value head's tile
            mbar_arrive_expect_tx(&sm.v_bar[vb ^ 1], kTile);
            tma_load_3d(sm.v[vb ^ 1], &maps.v, 0, hv + 1, t0, &sm.v_bar[vb ^ 1]);
            tma_load_3d(sm.v[vb ^ 1] + kHalf, &maps.v, 64, hv + 1, t0, &sm.v_bar[vb ^ 1]);
        }
        if (tid < 64) {
            const bool in = tid < L;
            const size_t gi = (size_t)(t0 + tid) * a.HV + hv;
            const float gg = in ? a.G[gi] : 0.f, bb = in ? bf2f(a.beta[gi]) : 0.f;
            sm.G[tid] = gg;
            sm.beta[tid] = bb;
            sm.wc[tid] = in ? bb * __expf(gg) / sm.rk[tid] : 0.f;
        }
        __syncthreads();
        if (active) {  // A row i, this warpgroup's 32 columns
            const int i = row;
            const float Gi = sm.G[i], bi = sm.beta[i];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = grp * 32 + jj;
                const float msk = (j < i && i < L) ? 1.f : 0.f;
                sm.A[i * kF + j] = msk * bi * kk[jj] * __expf(fminf(Gi - sm.G[j], 0.f));
            }
        }
        __syncthreads();
        tri_inverse(sm.A, sm.T, sm.X);
        // operands T diag(beta e^G / r_k) (warpgroup 0, also T to HBM) and T diag(beta) (warpgroup 1)
        if (active) {
            const int i = row;
            float4 *Tdst = reinterpret_cast<float4 *>(a.Tm + ((size_t)c * a.HV + hv) * 64 * 64 + (size_t)i * 64);
            for (int half = 0; half < 2; ++half) {
                float x[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    const float t = sm.T[i * kF + j];
                    const float bj = sm.beta[j];
                    if (grp == 0) x[jj] = t * sm.wc[j];
                    else x[jj] = t * bj;
                }
                if (grp == 0) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        Tdst[half * 8 + q] = make_float4(sm.T[i * kF + half * 32 + 4 * q], sm.T[i * kF + half * 32 + 4 * q + 1],
                                                         sm.T[i * kF + half * 32 + 4 * q + 2], sm.T[i * kF + half * 32 + 4 * q + 3]);
                }
                unsigned char *op = grp == 0 ? sm.op_w : sm.op_u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = half * 32 + q * 8;
                    *reinterpret_cast<uint4 *>(op + sw128_off(i, col)) =
                        make_uint4(pack_bf2(x[q * 8], x[q * 8 + 1]), pack_bf2(x[q * 8 + 2], x[q * 8 + 3]),
                                   pack_bf2(x[q * 8 + 4], x[q * 8 + 5]), pack_bf2(x[q * 8 + 6], x[q * 8 + 7]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(mbar_wait(&sm.v_bar[vb], (jv >> 1) & 1))) { ok = false; break; }
        if (tid == 0) {  // w -> columns 64..191, u -> 192..319
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 128, 0, 1);
            const uint32_t ks = smem_u32(sm.k), vs = smem_u32(sm.v[vb]);
            const uint32_t ws = smem_u32(sm.op_w), us = smem_u32(sm.op_u);
            for (int s = 0; s < 4; ++s) {
                mma_bf16(tb + 64, sdesc(ws + s * 32, 16, 1024), sdesc(ks + s * 2048, kHalf, 1024), id, s > 0);
                mma_bf16(tb + 192, sdesc(us + s * 32, 16, 1024), sdesc(vs + s * 2048, kHalf, 1024), id, s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        ok = __syncthreads_and(mbar_wait(&sm.mma_bar, mphase));
        mphase ^= 1;
        tc_fence_after();
        if (ok) {  // warpgroup 0 writes w, warpgroup 1 writes u
            const int i = row;
            const bool live = active && i < L;
            const size_t o = ((size_t)(t0 + (live ? i : 0)) * a.HV + hv) * kDim;
            bf16 *dst = grp == 0 ? a.w : a.u;
            const uint32_t col0 = grp == 0 ? 64 : 192;
            for (int cc = 0; cc < 4; ++cc) {
                float w[32];
                tmem_ld32(t_row + col0 + cc * 32, w);
                tmem_ld_wait();
                if (live) {
                    uint4 *wp = reinterpret_cast<uint4 *>(dst + o + cc * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        wp[q] = make_uint4(pack_bf2(w[q * 8], w[q * 8 + 1]), pack_bf2(w[q * 8 + 2], w[q * 8 + 3]),
                                           pack_bf2(w[q * 8 + 4], w[q * 8 + 5]), pack_bf2(w[q * 8 + 6], w[q * 8 + 7]));
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (!ok && tid == 0 && a.status) atomicOr(a.status, 2);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

cudaError_t launch_intra_tc(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    IntraMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    if (!encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.v, a.v, a.HV, a.T, rowb, rowb * a.HV, 64))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(IntraSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(k_intra_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_INTRA, s);
    k_intra_tc<<<dim3(a.num_chunks, a.H), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
