// gdn_bintra_b_tc.cu -- intra-chunk backward and WY pullback on the tensor
// cores ("dqkwg" / "WY pullback" of "cake_gdn: deterministic chunked GDN
// training kernels", section 2 and the round-11 kernel notes).
//
// One CTA of 128 threads per (chunk, value head).  All products are M=64
// tcgen05 MMAs whose rows are tokens; an M=64 result row m lives in TMEM lane
// 32 (m / 16) + m % 16, so lanes 0..15 of warp w own rows 16w..16w+15.
// With Qhat = diag(scale / r_q) Q, Khat = diag(1 / r_k) K, Gamma_ij =
// exp(G_i - G_j) and the WY inverse T (saved by the forward):
//   phase 1 (K = 128):  dM = dO v_new^T, QK = Q K^T, KK = K K^T,
//                       D1 = dW K^T, D2 = dv_new V^T
//     M_ij  = QK_ij scale / (r_q,i r_k,j) Gamma_ij       (j <= i)
//     dMG   = dM (.) Gamma,  P1 = dM (.) M  -> dG
//     dT_ij = beta_j (e^{G_j} D1_ij / r_k,j + D2_ij)     (j < i)
//   phase 1b/1c (K = 64): X = dT T^T,  dA = -T^T X (strictly lower)
//     B = dA (.) beta_i Gamma,  P2 = dA (.) KKhat Gamma -> dbeta, dG
//   phase 2 (K = 64):   dq  = dMG diag(1/r_k) K
//                       dk  = (diag(scale/r_q) dMG)^T Q + B diag(1/r_k) K
//                             + (diag(1/r_k) B)^T K
//                       dWt = T^T dW,   dUt = T^T dv_new
//     dkhat_m += beta_m e^{G_m} dWt_m,  dv_m = beta_m dUt_m,
//     dbeta_m += e^{G_m} khat_m . dWt_m + v_m . dUt_m,
//     dG_m    += beta_m e^{G_m} khat_m . dWt_m,   dg = reverse cumsum of dG.
// dq / dk go to their own buffers; the head-sum kernel adds them to the
// per-value-head gradients of qhat / khat that the h / dh' kernel wrote, then
// applies the L2-norm backward.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 256;   // two warpgroups share the 128 TMEM lanes
constexpr uint32_t kTile = 2 * 64 * 128;  // 64 rows x 128 bf16: two 8 KB k-halves
constexpr uint32_t kHalf = 64 * 128;
constexpr int kF = 65;                     // fp32 64 x 64 pitch

// TMEM columns
constexpr uint32_t cDM = 0, cQK = 64, cKK = 128, cD1 = 192, cD2 = 256, cX = 320, cA = 384;
constexpr uint32_t cDQ = 0, cDK = 128, cWT = 256, cUT = 384;

struct BbSmem {
    unsigned char q[kTile], k[kTile], v[kTile], dO[kTile], vn[kTile], dvn[kTile], dw[kTile];
    unsigned char op_dmg[kHalf];    // dMG_ij / r_k,j        [m][j]  K-major A
    unsigned char op_dmgt[kHalf];   // dMG_ij scale / r_q,i  [i][m]  MN-major A
    unsigned char op_b[kHalf];      // B_mj / r_k,j          [m][j]  K-major A
    unsigned char op_bt[kHalf];     // B_im / r_k,i          [i][m]  MN-major A
    unsigned char op_t[kHalf];      // T_ij rows i: K-major B of X, MN-major A of T^T X, T^T dW
    unsigned char op_dt[kHalf];     // dT_rb rows r: K-major A of X = dT T^T
    unsigned char op_x[kHalf];      // X_rj rows r: MN-major B of T^T X
    float C[64 * kF];               // P1_ij + beta_i P2_ij (column sums give dG)
    float G[64], beta[64], rq[64], rk[64], dG[64], dbeta[64];
    float rki[64], eg[64], qsc[64];  // 1 / r_k, e^{G}, scale / r_q (0 / 1 past L)
    float rs[2][64];                // per-warpgroup partial row sums of P2
    float cs[4][64];                // partial column sums of C
    float sk[2][64], su[2][64];     // per-warpgroup partial row dots
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

struct BbMaps {
    CUtensorMap q, k, v, dO, vn, dvn, dw;
};

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// Write 32 consecutive fp32 values of row `row`, columns [col0, col0 + 32), as
// bf16 into a 64-wide SW128 tile.
__device__ __forceinline__ void put_row32(unsigned char *tile, int row, int col0, const float *x) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(tile + sw128_off(row, col0 + q * 8)) =
            make_uint4(pack_bf2(x[q * 8 + 0], x[q * 8 + 1]), pack_bf2(x[q * 8 + 2], x[q * 8 + 3]),
                       pack_bf2(x[q * 8 + 4], x[q * 8 + 5]), pack_bf2(x[q * 8 + 6], x[q * 8 + 7]));
}

__device__ __forceinline__ float tile_at(const unsigned char *tile, int row, int col) {
    return bf2f(*reinterpret_cast<const bf16 *>(tile + (col >> 6) * kHalf + sw128_off(row, col & 63)));
}

__global__ void __launch_bounds__(kThr, 1) k_bintra_b_tc(const ChunkArgs a,
                                                         const __grid_constant__ BbMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BbSmem &sm = *reinterpret_cast<BbSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, hv = blockIdx.y;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const bool active = lane < 16;          // lane holds an M=64 result row
    const int grp = warp >> 2;              // warpgroup: which half of the work
    const int row = (warp & 3) * 16 + lane; // that row (valid when active)

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.tma_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        mbar_arrive_expect_tx(&sm.tma_bar, 7 * kTile);
        const CUtensorMap *mk[7] = {&maps.q, &maps.k, &maps.v, &maps.dO, &maps.vn, &maps.dvn, &maps.dw};
        unsigned char *dst[7] = {sm.q, sm.k, sm.v, sm.dO, sm.vn, sm.dvn, sm.dw};
        const int hh[7] = {h, h, hv, hv, hv, hv, hv};
        for (int i = 0; i < 7; ++i) {
            tma_load_3d(dst[i], mk[i], 0, hh[i], t0, &sm.tma_bar);
            tma_load_3d(dst[i] + kHalf, mk[i], 64, hh[i], t0, &sm.tma_bar);
        }
    }
    if (tid < 64) {
        const bool in = tid < L;
        const size_t r = (size_t)(t0 + tid) * a.H + h;
        const size_t gi = (size_t)(t0 + tid) * a.HV + hv;
        sm.G[tid] = in ? a.G[gi] : 0.f;
        sm.beta[tid] = in ? bf2f(a.beta[gi]) : 0.f;
        sm.rq[tid] = in ? a.rq[r] : 1.f;
        sm.rk[tid] = in ? a.rk[r] : 1.f;
        sm.dG[tid] = in ? a.dGp[gi] : 0.f;
        sm.dbeta[tid] = 0.f;
        sm.rki[tid] = 1.f / sm.rk[tid];
        sm.eg[tid] = in ? __expf(sm.G[tid]) : 0.f;
        sm.qsc[tid] = in ? a.scale / sm.rq[tid] : 0.f;
    }
    {  // T (fp32, saved by the forward) -> bf16 rows
        const float *Tsrc = a.Tm + ((size_t)c * a.HV + hv) * 64 * 64;
        for (int idx = tid; idx < 64 * 32; idx += kThr) {
            const int i = idx >> 5, j2 = (idx & 31) * 2;
            const float2 t2 = __ldg(reinterpret_cast<const float2 *>(Tsrc + i * 64 + j2));
            *reinterpret_cast<uint32_t *>(sm.op_t + sw128_off(i, j2)) = pack_bf2(t2.x, t2.y);
        }
    }
    fence_proxy_async_smem();
    bool ok = __syncthreads_and(mbar_wait(&sm.tma_bar, 0));
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t phase = 0;
    auto commit_wait = [&](bool &okr) {
        okr = __syncthreads_and(okr && mbar_wait(&sm.mma_bar, phase));
        phase ^= 1;
        tc_fence_after();
    };
    // ---- phase 1: five 64 x 64 products, contraction 128
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 64, 0, 0);
        const uint32_t A[5] = {smem_u32(sm.dO), smem_u32(sm.q), smem_u32(sm.k), smem_u32(sm.dw),
                               smem_u32(sm.dvn)};
        const uint32_t B[5] = {smem_u32(sm.vn), smem_u32(sm.k), smem_u32(sm.k), smem_u32(sm.k),
                               smem_u32(sm.v)};
        const uint32_t col[5] = {cDM, cQK, cKK, cD1, cD2};
        for (int p = 0; p < 5; ++p)
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
                mma_bf16(tb + col[p], sdesc(A[p] + off, 16, 1024), sdesc(B[p] + off, 16, 1024), id,
                         s > 0);
            }
        mma_commit(&sm.mma_bar);
    }
    commit_wait(ok);
    const int i = row;
    const bool live = active && i < L;
    const float Gi = active ? sm.G[i] : 0.f;
    if (ok) {
        if (grp == 0) {  // dM, QK -> M, dMG, P1 and the dMG operands
            const float qsi = active ? sm.qsc[i] : 0.f;
            float rsum = 0.f;
            for (int half = 0; half < 2; ++half) {
                float dm[32], qk[32];
                tmem_ld32(t_row + cDM + half * 32, dm);
                tmem_ld32(t_row + cQK + half * 32, qk);
                tmem_ld_wait();
                float x1[32], x2[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    // branch-free mask; the exponent is clamped to <= 0 so masked
                    // entries never form inf * 0
                    const float msk = (live && j <= i) ? 1.f : 0.f;
                    const float gam = msk * __expf(fminf(Gi - sm.G[j], 0.f));
                    const float rkj = sm.rki[j];
                    const float dmg = dm[jj] * gam;
                    const float p1 = dmg * qk[jj] * qsi * rkj;
                    rsum += p1;
                    if (active) sm.C[i * kF + j] = p1;
                    x1[jj] = dmg * rkj;
                    x2[jj] = dmg * qsi;
                }
                if (active) {
                    put_row32(sm.op_dmg, i, half * 32, x1);
                    put_row32(sm.op_dmgt, i, half * 32, x2);
                }
            }
            if (active) sm.dG[i] += rsum;
        } else {  // dW K^T, dv_new V^T -> dT row (bf16 operand)
            for (int half = 0; half < 2; ++half) {
                float d1[32], d2[32];
                tmem_ld32(t_row + cD1 + half * 32, d1);
                tmem_ld32(t_row + cD2 + half * 32, d2);
                tmem_ld_wait();
                float dt[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    const float msk = (live && j < i) ? 1.f : 0.f;
                    dt[jj] = msk * sm.beta[j] * (sm.eg[j] * sm.rki[j] * d1[jj] + d2[jj]);
                }
                if (active) put_row32(sm.op_dt, i, half * 32, dt);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- phase 1b: X = dT T^T  (A = dT rows, B = T rows as [N][K])
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 64, 0, 0);
        for (int s = 0; s < 4; ++s)
            mma_bf16(tb + cX, sdesc(smem_u32(sm.op_dt) + s * 32, 16, 1024),
                     sdesc(smem_u32(sm.op_t) + s * 32, 16, 1024), id, s > 0);
        mma_commit(&sm.mma_bar);
    }
    commit_wait(ok);
    if (ok) {  // X rows -> bf16 (each warpgroup one half of the columns)
        float x[32];
        tmem_ld32(t_row + cX + grp * 32, x);
        tmem_ld_wait();
        if (active) put_row32(sm.op_x, i, grp * 32, x);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- phase 1c: T^T X  (A = T rows read MN-major, B = X rows read MN-major)
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 64, 1, 1);
        for (int s = 0; s < 4; ++s)
            mma_bf16(tb + cA, sdesc(smem_u32(sm.op_t) + s * 2048, kHalf, 1024),
                     sdesc(smem_u32(sm.op_x) + s * 2048, kHalf, 1024), id, s > 0);
        mma_commit(&sm.mma_bar);
    }
    commit_wait(ok);
    if (ok) {  // dA = -(T^T X): B, P2, and their operands; warpgroup g takes columns [32g, 32g+32)
        float ta[32], kk[32];
        tmem_ld32(t_row + cA + grp * 32, ta);
        tmem_ld32(t_row + cKK + grp * 32, kk);
        tmem_ld_wait();
        float b1[32], b2[32], rsp = 0.f;
        const float bi = active ? sm.beta[i] : 0.f;
        const float rkii = active ? sm.rki[i] : 1.f;
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int j = grp * 32 + jj;
            const float msk = (live && j < i) ? 1.f : 0.f;
            const float dag = -ta[jj] * msk * __expf(fminf(Gi - sm.G[j], 0.f));
            const float rkj = sm.rki[j];
            const float b = dag * bi;
            const float p2 = dag * kk[jj] * rkii * rkj;
            rsp += p2;
            if (active) sm.C[i * kF + j] += bi * p2;
            b1[jj] = b * rkj;
            b2[jj] = b * rkii;
        }
        if (active) {
            put_row32(sm.op_b, i, grp * 32, b1);
            put_row32(sm.op_bt, i, grp * 32, b2);
            sm.rs[grp][i] = rsp;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- phase 2: 64 x 128 products, contraction 64
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t kA = smem_u32(sm.k), qA = smem_u32(sm.q), dwA = smem_u32(sm.dw),
                       dvA = smem_u32(sm.dvn);
        const uint32_t id_km = idesc_bf16(64, 128, 0, 1);  // A K-major, B MN-major
        const uint32_t id_mm = idesc_bf16(64, 128, 1, 1);  // A MN-major, B MN-major
        for (int s = 0; s < 4; ++s) {
            const uint64_t bK = sdesc(kA + s * 2048, kHalf, 1024), bQ = sdesc(qA + s * 2048, kHalf, 1024);
            const uint64_t bW = sdesc(dwA + s * 2048, kHalf, 1024), bV = sdesc(dvA + s * 2048, kHalf, 1024);
            const bool acc = s > 0;
            mma_bf16(tb + cDQ, sdesc(smem_u32(sm.op_dmg) + s * 32, 16, 1024), bK, id_km, acc);
            mma_bf16(tb + cDK, sdesc(smem_u32(sm.op_dmgt) + s * 2048, kHalf, 1024), bQ, id_mm, acc);
            mma_bf16(tb + cDK, sdesc(smem_u32(sm.op_b) + s * 32, 16, 1024), bK, id_km, true);
            mma_bf16(tb + cDK, sdesc(smem_u32(sm.op_bt) + s * 2048, kHalf, 1024), bK, id_mm, true);
            mma_bf16(tb + cWT, sdesc(smem_u32(sm.op_t) + s * 2048, kHalf, 1024), bW, id_mm, acc);
            mma_bf16(tb + cUT, sdesc(smem_u32(sm.op_t) + s * 2048, kHalf, 1024), bV, id_mm, acc);
        }
        mma_commit(&sm.mma_bar);
    }
    // meanwhile: row sums of P2 and column sums of C = P1 + beta_i P2
    if (ok) {
        if (tid < 64 && tid < L) {
            const float r2 = sm.rs[0][tid] + sm.rs[1][tid];
            sm.dbeta[tid] += r2;
            sm.dG[tid] += sm.beta[tid] * r2;
        }
        const int jcol = tid & 63, part = tid >> 6;
        float cs = 0.f;
        for (int r = part * 16; r < part * 16 + 16; ++r) cs += sm.C[r * kF + jcol];
        sm.cs[part][jcol] = cs;
    }
    __syncthreads();
    if (ok && tid < 64) sm.dG[tid] -= sm.cs[0][tid] + sm.cs[1][tid] + sm.cs[2][tid] + sm.cs[3][tid];
    commit_wait(ok);
    if (ok) {
        const int m = row;
        const bool mlive = active && m < L;
        const float em = mlive ? sm.eg[m] : 0.f;
        const float bm = mlive ? sm.beta[m] : 0.f;
        float sk = 0.f, su = 0.f;
        const size_t o = ((size_t)(t0 + (mlive ? m : 0)) * a.HV + hv) * kDim;
        for (int cc = 2 * grp; cc < 2 * grp + 2; ++cc) {  // this warpgroup's 64 columns
            float dq[32], dk[32], wt[32], ut[32];
            tmem_ld32(t_row + cDQ + cc * 32, dq);
            tmem_ld32(t_row + cDK + cc * 32, dk);
            tmem_ld32(t_row + cWT + cc * 32, wt);
            tmem_ld32(t_row + cUT + cc * 32, ut);
            tmem_ld_wait();
            if (mlive) {  // plain stores: the head-sum kernel adds them to the h / dh' terms
                float4 *qp = reinterpret_cast<float4 *>(a.dqp2 + o + cc * 32);
                float4 *kp = reinterpret_cast<float4 *>(a.dkp2 + o + cc * 32);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    qp[u] = make_float4(dq[4 * u + 0], dq[4 * u + 1], dq[4 * u + 2], dq[4 * u + 3]);
                    kp[u] = make_float4(dk[4 * u + 0] + bm * em * wt[4 * u + 0],
                                        dk[4 * u + 1] + bm * em * wt[4 * u + 1],
                                        dk[4 * u + 2] + bm * em * wt[4 * u + 2],
                                        dk[4 * u + 3] + bm * em * wt[4 * u + 3]);
                }
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) pk[j / 2] = pack_bf2(bm * ut[j], bm * ut[j + 1]);
                uint4 *dvp = reinterpret_cast<uint4 *>(a.dv + o + cc * 32);
#pragma unroll
                for (int u = 0; u < 4; ++u) dvp[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    sk += tile_at(sm.k, m, cc * 32 + j) * wt[j];
                    su += tile_at(sm.v, m, cc * 32 + j) * ut[j];
                }
            }
        }
        if (active) {
            sm.sk[grp][m] = sk;
            sm.su[grp][m] = su;
        }
    } else if (tid == 0 && a.status) {
        atomicOr(a.status, 2);
    }
    __syncthreads();
    if (ok && warp == 0) {  // dbeta, dG of the WY terms; dg = reverse cumsum of dG (warp scan)
        float dgv[2], dbv[2];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int m = 2 * lane + z;
            float dgm = 0.f, dbm = 0.f;
            if (m < L) {
                const float em = sm.eg[m], bm = sm.beta[m];
                const float sk = (sm.sk[0][m] + sm.sk[1][m]) * sm.rki[m];
                const float su = sm.su[0][m] + sm.su[1][m];
                dbm = sm.dbeta[m] + em * sk + su;
                dgm = sm.dG[m] + bm * em * sk;
            }
            dgv[z] = dgm;
            dbv[z] = dbm;
        }
        // suffix sums over m: reverse inclusive scan of dG
        float pair = dgv[0] + dgv[1];
        float suf = pair;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf += y;
        }
        const float after = suf - pair;  // sum over elements 2*lane+2 ...
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int m = 2 * lane + z;
            if (m < L) {
                const size_t gi = (size_t)(t0 + m) * a.HV + hv;
                a.dg[gi] = (z == 0 ? dgv[0] + dgv[1] : dgv[1]) + after;
                a.dbeta[gi] = f2bf(dbv[z]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

cudaError_t launch_bintra_b_tc(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    BbMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    if (!encode_rows_bf16(&m.q, a.q, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.v, a.v, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dO, a.d_o, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.vn, a.vnew, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dvn, a.dvnew, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dw, a.dW, a.HV, a.T, rowb, rowb * a.HV, 64))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BbSmem) + 1024;
    static_assert(sizeof(BbSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k_bintra_b_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BINTRA_B, s);
    k_bintra_b_tc<<<dim3(a.num_chunks, a.HV), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
