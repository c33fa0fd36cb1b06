// gdn_out_tc.cu -- chunk output o (forward) and dv_local (backward) on the
// tensor cores.
//
// One CTA of 128 threads per (chunk, value head).  Both modes start from the
// intra-chunk attention matrix
//   M[t][j] = (qhat_t . khat_j) exp(G_t - G_j),  j <= t < L   (else 0)
// formed by one product Q K^T (M=64 N=64 K=128) and scaled by
// scale / (r_q,t r_k,j) in an epilogue that reads it as 16x256b fragments
// (all four warps, two rows and eight columns per lane).
//   forward : o[t][v] = c_t (Q h)[t][v] + (M v_new)[t][v],
//             c_t = e^{G_t} scale / r_q,t            (o = diag(e^G) Qhat h + M v_new)
//   backward: dv_loc[t][v] = (M^T dO)[t][v]
// as token-row products (M=64, N=128); h_c [k][v], v_new and dO are read as
// MN-major operands straight from their TMA tiles, and the results are read as
// 16x256b fragments so that every lane writes bf16 pairs of two token rows.
#include <stddef.h>
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_epi.cuh"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
constexpr uint32_t kBox = 64 * 128;    // 64 rows x 128 B
constexpr uint32_t kBig = 128 * 128;   // 128 rows x 128 B

// The backward mode needs no h_c tile and half the TMEM columns, so three of its
// CTAs share an SM (two in the forward mode).
template <bool kForward>
struct OutSmem {
    unsigned char kq[2 * kBig];   // [K; Q] per k-half: K rows 0..63, Q rows 64..127 (one TMA box each)
    unsigned char tv[2 * kBox];   // v_new (forward) or dO (backward) [t][v] per v-half
    unsigned char mm[kBox];       // M, row i at row i (bf16)
    unsigned char stg[2 * kBox];  // a full chunk's output rows per v-half, for two TMA stores
    unsigned char hc[kForward ? 2 * kBig : 16];   // h_c [k][v] per v-half (forward only)
    float G[64], rq[64], rk[64];
    float qsc[64], rki[64], ct[64];  // scale / r_q, 1 / r_k, e^{G} scale / r_q
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

// Every TMA / SW128 tile starts on a 1024-byte boundary of the (1024-aligned) struct.
static_assert(offsetof(OutSmem<true>, tv) % 1024 == 0 && offsetof(OutSmem<true>, mm) % 1024 == 0 &&
                  offsetof(OutSmem<true>, stg) % 1024 == 0 && offsetof(OutSmem<true>, hc) % 1024 == 0 &&
                  offsetof(OutSmem<false>, stg) % 1024 == 0,
              "SW128 tiles on 1024-byte boundaries");

struct OutMaps {
    CUtensorMap q, k, h, tv, out;   // out: o (forward) or dv_loc (backward)
};

template <bool kForward>
constexpr uint32_t kTmemCols = kForward ? 256 : 128;

struct OutUnit {
    int c, hv, h, t0, L;
};

__device__ __forceinline__ OutUnit out_unit(const ChunkArgs &a, int u) {
    OutUnit x;
    x.c = u / a.HV;
    x.hv = u - x.c * a.HV;
    x.h = x.hv / (a.HV / a.H);
    const bool in = in_range(x.c, 1, a.num_chunks, a.status);
    x.t0 = in ? a.chunk_start[x.c] : 0;
    x.L = in ? a.chunk_len[x.c] : 0;
    return x;
}
// Unit u + 1 after unit x = u; the chunk table is read only when the chunk changes.
__device__ __forceinline__ OutUnit out_next(const ChunkArgs &a, const OutUnit &x) {
    if (x.hv + 1 < a.HV) {
        OutUnit y = x;
        y.hv = x.hv + 1;
        y.h = y.hv / (a.HV / a.H);
        return y;
    }
    return out_unit(a, (x.c + 1) * a.HV);
}

template <bool kForward>
__device__ __forceinline__ void out_issue(const OutMaps &m, OutSmem<kForward> &sm, const ChunkArgs &a,
                                          const OutUnit &x) {
    const uint32_t bytes = 2 * kBig + 2 * kBox + (kForward ? 2 * kBig : 0);
    mbar_arrive_expect_tx(&sm.tma_bar, bytes);
    tma_load_3d(sm.kq, &m.k, 0, x.h, x.t0, &sm.tma_bar);
    tma_load_3d(sm.kq + kBox, &m.q, 0, x.h, x.t0, &sm.tma_bar);
    tma_load_3d(sm.kq + kBig, &m.k, 64, x.h, x.t0, &sm.tma_bar);
    tma_load_3d(sm.kq + kBig + kBox, &m.q, 64, x.h, x.t0, &sm.tma_bar);
    tma_load_3d(sm.tv, &m.tv, 0, x.hv, x.t0, &sm.tma_bar);
    tma_load_3d(sm.tv + kBox, &m.tv, 64, x.hv, x.t0, &sm.tma_bar);
    if constexpr (kForward) {
        const int row = (x.c * a.HV + x.hv) * 128;
        tma_load_3d(sm.hc, &m.h, 0, 0, row, &sm.tma_bar);
        tma_load_3d(sm.hc + kBig, &m.h, 64, 0, row, &sm.tma_bar);
    }
}

// Persistent: CTA b walks the units [b per, (b + 1) per) (unit u = chunk u / HV, value
// head u % HV); the next unit's tiles load as soon as the second product has read
// this unit's, and its per-token scalars a unit ahead.
template <bool kForward>
__global__ void __launch_bounds__(kThr, kForward ? 2 : 3) k_out_tc(const ChunkArgs a,
                                                                   const __grid_constant__ OutMaps maps,
                                                                   int per) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    OutSmem<kForward> &sm = smem_struct<OutSmem<kForward>>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nunits = a.num_chunks * a.HV;
    const int ub = blockIdx.x * per, ue = min(nunits, ub + per);
    if (ub >= ue) return;
    if (tid == 0) tma_prefetch_maps(maps);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, kTmemCols<kForward>);
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
    OutUnit x = out_unit(a, ub);
    if (tid == 0) out_issue<kForward>(maps, sm, a, x);
    // per-token scalars of thread tid < 64 (raw), fetched one unit ahead
    float pG = 0.f, pRq = 1.f, pRk = 1.f;
    bool pin = false;
    auto fetch = [&](const OutUnit &y) {
        pin = tid < 64 && tid < y.L &&
              in_range((size_t)(y.t0 + tid) * a.HV + y.hv, 1, n_tok_hv(a), a.status);
        if (pin) {
            const size_t r = (size_t)(y.t0 + tid) * a.H + y.h;
            pG = a.G[(size_t)(y.t0 + tid) * a.HV + y.hv];
            pRq = a.rq[r];
            pRk = a.rk[r];
        }
    };
    fetch(x);
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)(warp * 32) << 16);
    uint32_t phase = 0;
    int issued = 1, waited = 0;
    bool ok = true;
    for (int u = ub; u < ue; ++u) {
        const bool has_next = u + 1 < ue;
        const int hv = x.hv, t0 = x.t0, L = x.L;
        if (tid < 64) {  // tokens past L: G = 0, r = 1, e^G term 0
            const float rq = pin ? pRq : 1.f, rk = pin ? pRk : 1.f, gg = pin ? pG : 0.f;
            sm.G[tid] = gg;
            sm.rq[tid] = rq;
            sm.rk[tid] = rk;
            sm.qsc[tid] = a.scale / rq;
            sm.rki[tid] = 1.f / rk;
            sm.ct[tid] = pin ? __expf(gg) * (a.scale / rq) : 0.f;
        }
        ok = __syncthreads_and(ok && mbar_wait(&sm.tma_bar, waited & 1));
        ++waited;
        if (!ok) break;
        // QK = Q K^T (M=64; Q rows sit at kBox inside each k-half of the [K; Q] tile)
        if (tid == 0 && ok) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 64, 0, 0);
            const uint32_t as = smem_u32(sm.kq);
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * kBig + (s & 3) * 32;
                mma_bf16(tb, sdesc(as + kBox + off, 16, 1024), sdesc(as + off, 16, 1024), id, s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        const OutUnit nx = has_next ? out_next(a, x) : x;
        if (has_next) fetch(nx);
        ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, phase));
        phase ^= 1;
        tc_fence_after();
        if (ok) {  // M from 16x256b fragments of QK: rows ra, rb = ra + 8 of warp w's block,
                   // columns 32 c + 8k + cq + {0, 1}
            const int lane = tid & 31;
            const int ra = 16 * warp + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
            const float qa = sm.qsc[ra], qb = sm.qsc[rb], Ga = sm.G[ra], Gb = sm.G[rb];
            const bool la = ra < L, lb = rb < L;
    #pragma unroll
            for (int c = 0; c < 2; ++c) {
                float r[16];
                epi::tmem_ld16x256_x4(t_row + 32 * c, r);
                tmem_ld_wait();
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = 32 * c + 8 * k + cq;
                    float m[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int jj = j + (e & 1);
                        const bool up = e & 2;
                        const int row = up ? rb : ra;
                        const float msk = (jj <= row && (up ? lb : la)) ? 1.f : 0.f;
                        m[e] = msk * r[4 * k + e] * (up ? qb : qa) * sm.rki[jj] *
                               __expf(fminf((up ? Gb : Ga) - sm.G[jj], 0.f));
                    }
                    // row t of M at row t: the forward reads it as K-major [t][j] (B = M^T
                    // operand of v_new^T M^T), the backward as MN-major [j][t] (B = M of dO^T M)
                    epi::put_pair(sm.mm, ra, j, m[0], m[1]);
                    epi::put_pair(sm.mm, rb, j, m[2], m[3]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {  // token-row products (M=64, N=128), rows t of the results
            tc_fence_after();
            const uint32_t tvs = smem_u32(sm.tv), mms = smem_u32(sm.mm);
            if constexpr (kForward) {
                // O1 = Q h : A = Q [t][k] (K-major), B = h_c [k][v] (MN-major, v halves 16 KB apart)
                const uint32_t id1 = idesc_bf16(64, 128, 0, 1);
                const uint32_t hs = smem_u32(sm.hc), qs = smem_u32(sm.kq + kBox);
                for (int s = 0; s < 8; ++s)
                    mma_bf16(tb, sdesc(qs + (s >> 2) * kBig + (s & 3) * 32, 16, 1024), sdesc(hs + s * 2048, kBig, 1024),
                             id1, s > 0);
                // O2 = M v_new : A = M [t][j] (K-major), B = v_new [j][v] (MN-major, v halves 8 KB apart)
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tb + 128, sdesc(mms + s * 32, 16, 1024), sdesc(tvs + s * 2048, kBox, 1024), id1, s > 0);
            } else {
                // DL = M^T dO : A = M [j][t] (MN-major), B = dO [j][v] (MN-major)
                const uint32_t id2 = idesc_bf16(64, 128, 1, 1);
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tb, sdesc(mms + s * 2048, kBox, 1024), sdesc(tvs + s * 2048, kBox, 1024), id2, s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        if (tid == 0) tma_store_wait_read();  // the last unit's staged rows have been read
        ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, phase));
        phase ^= 1;
        tc_fence_after();
        if (tid == 0 && ok && has_next) out_issue<kForward>(maps, sm, a, nx);  // the tiles have been read
        if (ok && has_next) ++issued;
        if (ok) {  // 16x256b fragments: rows ra, ra + 8, columns v = 32 c + 8k + cq + {0, 1}
            const int lane = tid & 31;
            const int ra = 16 * warp + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
            const bool la = ra < L, lb = rb < L;
            const float ca = sm.ct[ra], cb = sm.ct[rb];
            bf16 *dst = kForward ? a.o : a.dvloc;
            bf16 *da = dst + ((size_t)(t0 + (la ? ra : 0)) * a.HV + hv) * kDim;
            bf16 *db = dst + ((size_t)(t0 + (lb ? rb : 0)) * a.HV + hv) * kDim;
    #pragma unroll
            for (int c = 0; c < 4; ++c) {
                float r1[16], r2[16];
                epi::tmem_ld16x256_x4(t_row + 32 * c, r1);
                if constexpr (kForward) epi::tmem_ld16x256_x4(t_row + 128 + 32 * c, r2);
                tmem_ld_wait();
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int v = 32 * c + 8 * k + cq;
                    float x0, x1, y0, y1;
                    if constexpr (kForward) {
                        x0 = ca * r1[4 * k] + r2[4 * k];
                        x1 = ca * r1[4 * k + 1] + r2[4 * k + 1];
                        y0 = cb * r1[4 * k + 2] + r2[4 * k + 2];
                        y1 = cb * r1[4 * k + 3] + r2[4 * k + 3];
                    } else {
                        x0 = r1[4 * k]; x1 = r1[4 * k + 1]; y0 = r1[4 * k + 2]; y1 = r1[4 * k + 3];
                    }
                    if (L == 64) {  // staged for the TMA store
                        epi::put_pair(sm.stg + (c >> 1) * kBox, ra, v & 63, x0, x1);
                        epi::put_pair(sm.stg + (c >> 1) * kBox, rb, v & 63, y0, y1);
                    } else {
                        if (la && in_range(da + v - dst, 2, n_rows_hv(a), a.status))
                            *reinterpret_cast<uint32_t *>(da + v) = epi::pack_bf2(x0, x1);
                        if (lb && in_range(db + v - dst, 2, n_rows_hv(a), a.status))
                            *reinterpret_cast<uint32_t *>(db + v) = epi::pack_bf2(y0, y1);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);  // the unit's scalars, M operand and TMEM are free
        if (!ok) break;
        if (tid == 0 && L == 64) {
            tma_store_3d(&maps.out, 0, hv, t0, sm.stg);
            tma_store_3d(&maps.out, 64, hv, t0, sm.stg + kBox);
            tma_store_commit();
        }
        x = nx;
    }
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        if (issued > waited) mbar_wait(&sm.tma_bar, (issued - 1) & 1, kDrainLimitNs);  // drain (bounded)
    }
    if (tid == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, kTmemCols<kForward>);
}

template <bool kForward>
cudaError_t launch_out_mode(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    OutMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    const uint64_t hrows = (uint64_t)a.num_chunks * a.HV * 128;
    if (!encode_rows_bf16(&m.q, a.q, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.tv, kForward ? (const void *)a.vnew : (const void *)a.d_o, a.HV, a.T,
                          rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.out, kForward ? (const void *)a.o : (const void *)a.dvloc, a.HV, a.T,
                          rowb, rowb * a.HV, 64))
        return cudaErrorInvalidValue;
    if (kForward && !encode_rows_bf16(&m.h, a.hc, 1, hrows, rowb, rowb, 128))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(OutSmem<kForward>) + 1024;
    static_assert((kForward ? 2 : 3) * (sizeof(OutSmem<kForward>) + 2048) <= 233472, "CTAs per SM");
    cudaError_t e = cudaFuncSetAttribute(k_out_tc<kForward>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    const int nunits = a.num_chunks * a.HV;
    const int slots = (kForward ? 2 : 3) * sms;
    const int per = (nunits + slots - 1) / slots;
    TimerScope ts(a.timer, kForward ? GDN_KERNEL_OUT : GDN_KERNEL_DVLOC, s);
    k_out_tc<kForward><<<(nunits + per - 1) / per, kThr, smem, s>>>(a, m, per);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_out_tc(const ChunkArgs &a, cudaStream_t s) { return launch_out_mode<true>(a, s); }
cudaError_t launch_dvloc_tc(const ChunkArgs &a, cudaStream_t s) {
    return launch_out_mode<false>(a, s);
}

}  // namespace gdn
