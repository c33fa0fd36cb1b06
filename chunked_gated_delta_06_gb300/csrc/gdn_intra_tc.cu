// gdn_intra_tc.cu -- WY pass of a chunk on the tensor cores ("WY pass" of
// "cake_gdn: deterministic chunked GDN training kernels", section 2; the
// chunk form of the GDN context-parallel scans in "Qwen3.5-397B RL trainer on
// 128 v7x", maxtext #5799).
//
// One CTA of 256 threads per (chunk, key head).  Its two warpgroups work on
// two value heads of the key head at once (value heads 2p and 2p + 1), each
// with its own tiles, TMEM columns and named barrier.  With Khat = diag(1 / r_k) K and Gamma_ij = exp(G_i - G_j):
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

constexpr int kThr = 256;   // two warpgroups, each working on its own value head
constexpr uint32_t kHalf = 64 * 128;
constexpr uint32_t kTile = 2 * kHalf;
constexpr int kF = 65;

struct IntraSmem {
    unsigned char k[kTile];
    unsigned char v[2][2][kTile];     // [warpgroup][buffer] value tiles
    unsigned char op_w[2][kHalf];     // T_ij beta_j e^{G_j} / r_k,j  [i][j] K-major
    unsigned char op_u[2][kHalf];     // T_ij beta_j                  [i][j] K-major
    float A[2][64 * kF];
    float T[2][64 * kF];
    float X[2][64 * kF];
    float G[2][64], beta[2][64], wc[2][64], rk[64];
    uint64_t k_bar, v_bar[2][2], mma_bar[3];
    uint32_t tmem_base;
    int err[2];
};

struct IntraMaps {
    CUtensorMap k, v;
};

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// Barrier over the 128 threads of warpgroup g (named barrier 1 + g).
__device__ __forceinline__ void group_sync(int g) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}

// T = (I + A)^-1 for a strictly lower A (64 x 64, rows/cols >= L are zero),
// by the 128 threads of warpgroup g (gt = thread index within the group):
// 8x8 diagonal blocks by substitution, then T21 = -T22 (A21 T11) at block
// sizes 8, 16 and 32.
__device__ void tri_inverse(const float *A, float *T, float *X, int gt, int g) {
    for (int idx = gt; idx < 64 * 64; idx += 128) T[(idx >> 6) * kF + (idx & 63)] = 0.f;
    group_sync(g);
    if (gt < 64) {
        const int b = gt >> 3, cc = gt & 7, base = b * 8;
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
    group_sync(g);
    for (int s = 8; s < 64; s *= 2) {
        const int nb = 64 / (2 * s), ent = nb * s * s;
        for (int e = gt; e < ent; e += 128) {
            const int p = e / (s * s), rr = (e / s) % s, cc = e % s;
            const int r0 = p * 2 * s + s, c0 = p * 2 * s;
            float acc = 0.f;
            for (int m = cc; m < s; ++m) acc += A[(r0 + rr) * kF + c0 + m] * T[(c0 + m) * kF + c0 + cc];
            X[(r0 + rr) * kF + c0 + cc] = acc;
        }
        group_sync(g);
        for (int e = gt; e < ent; e += 128) {
            const int p = e / (s * s), rr = (e / s) % s, cc = e % s;
            const int r0 = p * 2 * s + s, c0 = p * 2 * s;
            float acc = 0.f;
            for (int m = 0; m <= rr; ++m) acc += T[(r0 + rr) * kF + r0 + m] * X[(r0 + m) * kF + c0 + cc];
            T[(r0 + rr) * kF + c0 + cc] = -acc;
        }
        group_sync(g);
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
    const int g = warp >> 2, gt = tid & 127;  // warpgroup, thread within it
    const bool active = lane < 16;
    const int row = (warp & 3) * 16 + lane;
    const int npairs = (r + 1) / 2;

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.k_bar, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sm.v_bar[x][0], 1);
            mbar_init(&sm.v_bar[x][1], 1);
        }
        for (int x = 0; x < 3; ++x) mbar_init(&sm.mma_bar[x], 1);
        fence_mbar_init();
        sm.err[0] = sm.err[1] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.k_bar, kTile);
        tma_load_3d(sm.k, &maps.k, 0, h, t0, &sm.k_bar);
        tma_load_3d(sm.k + kHalf, &maps.k, 64, h, t0, &sm.k_bar);
    }
    if (gt == 0 && g < r) {  // each warpgroup's first value-head tile
        const int hv = h * r + g;
        mbar_arrive_expect_tx(&sm.v_bar[g][0], kTile);
        tma_load_3d(sm.v[g][0], &maps.v, 0, hv, t0, &sm.v_bar[g][0]);
        tma_load_3d(sm.v[g][0] + kHalf, &maps.v, 64, hv, t0, &sm.v_bar[g][0]);
    }
    if (tid < 64) sm.rk[tid] = tid < L ? a.rk[(size_t)(t0 + tid) * a.H + h] : 1.f;
    bool ok = __syncthreads_and(mbar_wait(&sm.k_bar, 0));
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)((warp & 3) * 32) << 16);
    if (tid == 0 && ok) {  // KK = K K^T into columns 0..63
        tc_fence_after();
        const uint32_t ks = smem_u32(sm.k);
        const uint32_t id = idesc_bf16(64, 64, 0, 0);
        for (int s = 0; s < 8; ++s) {
            const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
            mma_bf16(tb, sdesc(ks + off, 16, 1024), sdesc(ks + off, 16, 1024), id, s > 0);
        }
        mma_commit(&sm.mma_bar[2]);
    }
    ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar[2], 0));
    tc_fence_after();
    // KKhat row i stays in registers for all value heads of this warpgroup
    float kk[64];
    if (ok) {
        float k0[32], k1[32];
        tmem_ld32(t_row, k0);
        tmem_ld32(t_row + 32, k1);
        tmem_ld_wait();
        const float rki = active ? 1.f / sm.rk[row] : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            kk[j] = k0[j] * rki / sm.rk[j];
            kk[32 + j] = k1[j] * rki / sm.rk[32 + j];
        }
    }
    tc_fence_before();
    __syncthreads();  // KK columns are free from here on
    tc_fence_after();
    const uint32_t cw = tb + g * 256, cu = tb + g * 256 + 128;   // this group's w / u columns
    uint32_t mphase = 0;
    for (int p = 0; p < npairs && ok; ++p) {
        const int jv = 2 * p + g;
        if (jv >= r) break;  // odd r: the second warpgroup has no last value head
        const int hv = h * r + jv, vb = p & 1;
        if (gt == 0 && jv + 2 < r) {  // prefetch this group's next value head
            mbar_arrive_expect_tx(&sm.v_bar[g][vb ^ 1], kTile);
            tma_load_3d(sm.v[g][vb ^ 1], &maps.v, 0, hv + 2, t0, &sm.v_bar[g][vb ^ 1]);
            tma_load_3d(sm.v[g][vb ^ 1] + kHalf, &maps.v, 64, hv + 2, t0, &sm.v_bar[g][vb ^ 1]);
        }
        if (gt < 64) {
            const bool in = gt < L;
            const size_t gi = (size_t)(t0 + gt) * a.HV + hv;
            const float gg = in ? a.G[gi] : 0.f, bb = in ? bf2f(a.beta[gi]) : 0.f;
            sm.G[g][gt] = gg;
            sm.beta[g][gt] = bb;
            sm.wc[g][gt] = in ? bb * __expf(gg) / sm.rk[gt] : 0.f;
        }
        group_sync(g);
        float *A = sm.A[g], *T = sm.T[g];
        if (active) {  // A row i
            const int i = row;
            const float Gi = sm.G[g][i], bi = sm.beta[g][i];
#pragma unroll 8
            for (int j = 0; j < 64; ++j) {
                const float msk = (j < i && i < L) ? 1.f : 0.f;
                A[i * kF + j] = msk * bi * kk[j] * __expf(fminf(Gi - sm.G[g][j], 0.f));
            }
        }
        group_sync(g);
        tri_inverse(A, T, sm.X[g], gt, g);
        if (active) {  // operands, and T to HBM
            const int i = row;
            float4 *Tdst = reinterpret_cast<float4 *>(a.Tm + ((size_t)c * a.HV + hv) * 64 * 64 + (size_t)i * 64);
            for (int half = 0; half < 2; ++half) {
                float xw[32], xu[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    const float t = T[i * kF + j];
                    xw[jj] = t * sm.wc[g][j];
                    xu[jj] = t * sm.beta[g][j];
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    Tdst[half * 8 + q] = make_float4(T[i * kF + half * 32 + 4 * q], T[i * kF + half * 32 + 4 * q + 1],
                                                     T[i * kF + half * 32 + 4 * q + 2], T[i * kF + half * 32 + 4 * q + 3]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int col = half * 32 + q * 8;
                    *reinterpret_cast<uint4 *>(sm.op_w[g] + sw128_off(i, col)) =
                        make_uint4(pack_bf2(xw[q * 8], xw[q * 8 + 1]), pack_bf2(xw[q * 8 + 2], xw[q * 8 + 3]),
                                   pack_bf2(xw[q * 8 + 4], xw[q * 8 + 5]), pack_bf2(xw[q * 8 + 6], xw[q * 8 + 7]));
                    *reinterpret_cast<uint4 *>(sm.op_u[g] + sw128_off(i, col)) =
                        make_uint4(pack_bf2(xu[q * 8], xu[q * 8 + 1]), pack_bf2(xu[q * 8 + 2], xu[q * 8 + 3]),
                                   pack_bf2(xu[q * 8 + 4], xu[q * 8 + 5]), pack_bf2(xu[q * 8 + 6], xu[q * 8 + 7]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (!mbar_wait(&sm.v_bar[g][vb], (p >> 1) & 1)) sm.err[g] = 1;
        group_sync(g);
        if (sm.err[g]) { ok = false; break; }
        if (gt == 0) {  // w and u of this value head
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 128, 0, 1);
            const uint32_t ks = smem_u32(sm.k), vs = smem_u32(sm.v[g][vb]);
            const uint32_t ws = smem_u32(sm.op_w[g]), us = smem_u32(sm.op_u[g]);
            for (int s = 0; s < 4; ++s) {
                mma_bf16(cw, sdesc(ws + s * 32, 16, 1024), sdesc(ks + s * 2048, kHalf, 1024), id, s > 0);
                mma_bf16(cu, sdesc(us + s * 32, 16, 1024), sdesc(vs + s * 2048, kHalf, 1024), id, s > 0);
            }
            mma_commit(&sm.mma_bar[g]);
        }
        if (!mbar_wait(&sm.mma_bar[g], mphase)) sm.err[g] = 1;
        mphase ^= 1;
        tc_fence_after();
        group_sync(g);
        if (sm.err[g]) { ok = false; break; }
        {
            const int i = row;
            const bool live = active && i < L;
            const size_t o = ((size_t)(t0 + (live ? i : 0)) * a.HV + hv) * kDim;
            for (int wu = 0; wu < 2; ++wu) {
                bf16 *dst = wu == 0 ? a.w : a.u;
                const uint32_t col0 = (wu == 0 ? cw : cu) - tb;
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
        }
        tc_fence_before();
        group_sync(g);
    }
    if (!ok && gt == 0 && a.status) atomicOr(a.status, 2);
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
    static_assert(sizeof(IntraSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k_intra_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_INTRA, s);
    k_intra_tc<<<dim3(a.num_chunks, a.H), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
