// gdn_bstate_tc.cu -- backward (reverse) inter-chunk state scan on the tensor
// cores ("dhu" in "cake_gdn: deterministic chunked GDN training kernels",
// section 2; the reverse recurrence of the GDN context-parallel dh scan in
// "Qwen3.5-397B RL trainer on 128 v7x", maxtext #5799).
//
// One CTA of 128 threads per (sequence, value head) walks the chunks in
// reverse.  dS = dh^T (V x K) lives in TMEM as fp32 (lane v = row v), seeded
// with d(final state)^T.  Per chunk, with dh' the gradient of the state after
// the chunk (= the current dS^T):
//   1. thread v writes row v of dS as bf16 to shared memory (copied to
//      dh_c[chunk][hv], stored transposed [v][k], by one TMA store), then
//      dS <- e^{G_L} dS;
//   2. Pd = dS'_bf16 K^T                          (M=128 N=64 K=128)
//   3. dv_new^T[v][t] = dv_loc[t][v] + e^{G_L-G_t}/r_k,t Pd[v][t]  -> HBM (fp32)
//   4. dS += (c_t dO[t][v])^T Q - dv_new^T w,  c_t = e^{G_t} scale / r_q,t
//      (two M=128 N=128 K=64 products; Q and w are raw MN-major tiles)
// which is dh <- e^{G_L} dh' + Qtil^T dO - w^T dv_new and
// dv_new = dv_loc + Ktil dh'.  dh0 = dS^T at the sequence start.
// K, Q, w and dO tiles stream in by TMA two chunks ahead; waits are bounded.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
constexpr uint32_t kTileBytes = 64 * 128;
constexpr uint32_t kStageBytes = 10 * kTileBytes;  // K, Q, w, dO, dv_loc: two boxes each

struct BStateSmem {
    unsigned char a_ds[2 * 128 * 128];  // dS' bf16 [v][k]
    unsigned char a_do[128 * 128];      // c_t dO^T bf16 [v][t]
    unsigned char a_dv[128 * 128];      // -dv_new^T bf16 [v][t]
    unsigned char stage[2][kStageBytes];
    float kc[64];                       // e^{G_L - G_t} / r_k,t (0 past L)
    float qc[64];                       // e^{G_t} scale / r_q,t (0 past L)
    float gt[64], rkt[64], rqt[64];     // this chunk's G, r_k, r_q (prefetched)
    uint64_t tma_bar[2];
    uint64_t mma_bar;
    uint32_t tmem_base;
    int error;
};

struct BStateMaps {
    CUtensorMap k, q, w, dO, dl, dhc;
};

__device__ __forceinline__ void issue_stage(const BStateMaps &m, BStateSmem &sm, int st, int t0,
                                            int h, int hv) {
    unsigned char *b = sm.stage[st];
    uint64_t *bar = &sm.tma_bar[st];
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_3d(b + 0 * kTileBytes, &m.k, 0, h, t0, bar);
    tma_load_3d(b + 1 * kTileBytes, &m.k, 64, h, t0, bar);
    tma_load_3d(b + 2 * kTileBytes, &m.q, 0, h, t0, bar);
    tma_load_3d(b + 3 * kTileBytes, &m.q, 64, h, t0, bar);
    tma_load_3d(b + 4 * kTileBytes, &m.w, 0, hv, t0, bar);
    tma_load_3d(b + 5 * kTileBytes, &m.w, 64, hv, t0, bar);
    tma_load_3d(b + 6 * kTileBytes, &m.dO, 0, hv, t0, bar);
    tma_load_3d(b + 7 * kTileBytes, &m.dO, 64, hv, t0, bar);
    tma_load_3d(b + 8 * kTileBytes, &m.dl, 0, hv, t0, bar);
    tma_load_3d(b + 9 * kTileBytes, &m.dl, 64, hv, t0, bar);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThr, 1)
    k_bstate_tc(const ChunkArgs a, const __grid_constant__ BStateMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BStateSmem &sm = *reinterpret_cast<BStateSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int hv = blockIdx.x, n = a.seq_order[blockIdx.y];  // longest sequences first
    const int h = hv / (a.HV / a.H);
    const int v = tid;
    const int cb = a.seq_chunk_off[n];
    const int ce = min(a.seq_chunk_off[n + 1], a.num_chunks);
    const int nch = max(ce - cb, 0);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.tma_bar[0], 1);
        mbar_init(&sm.tma_bar[1], 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
        sm.error = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t_row = sm.tmem_base + ((uint32_t)(warp * 32) << 16);
    const uint32_t tS = t_row, tP = t_row + 128;

    if (tid == 0)
        for (int i = 0; i < 2 && i < nch; ++i) issue_stage(maps, sm, i, a.chunk_start[ce - 1 - i], h, hv);
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim;
    for (int kc = 0; kc < 4; ++kc) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            r[j] = a.d_ht ? a.d_ht[sbase + (size_t)(kc * 32 + j) * kDim + v] : 0.f;
        tmem_st32(tS + kc * 32, r);
    }
    tmem_st_wait();

    const uint32_t idP = idesc_bf16(128, 64, 0, 0);
    const uint32_t idS = idesc_bf16(128, 128, 0, 1);
    uint32_t mma_phase = 0;
    bool ok = true;
    // per-token scalars of the next chunk, loaded one chunk ahead
    float pg = 0.f, prk = 1.f, prq = 1.f;
    auto fetch = [&](int cc) {
        const int tt0 = a.chunk_start[cc], LL = a.chunk_len[cc];
        if (tid < LL) {
            const size_t t = (size_t)(tt0 + tid);
            pg = a.G[t * a.HV + hv];
            prk = a.rk[t * a.H + h];
            prq = a.rq[t * a.H + h];
        } else {
            pg = 0.f; prk = 1.f; prq = 1.f;
        }
    };
    if (tid < 64 && nch > 0) fetch(ce - 1);
    for (int i = 0; i < nch; ++i) {
        const int c = ce - 1 - i, st = i & 1;
        const int t0 = a.chunk_start[c], L = a.chunk_len[c];
        if (tid < 64) {
            sm.gt[tid] = pg;
            sm.rkt[tid] = prk;
            sm.rqt[tid] = prq;
            if (i + 1 < nch) fetch(c - 1);
        }
        __syncthreads();
        const float Gl = L > 0 ? sm.gt[L - 1] : 0.f;
        if (tid < 64) {
            float kk = 0.f, qq = 0.f;
            if (tid < L) {
                const float Gt = sm.gt[tid];
                kk = expf(Gl - Gt) / sm.rkt[tid];
                qq = expf(Gt) * a.scale / sm.rqt[tid];
            }
            sm.kc[tid] = kk;
            sm.qc[tid] = qq;
        }
        const float egl = expf(Gl);
        // 1. dS' -> bf16 operand (copied to dh_c by TMA below), then dS <- e^{G_L} dS'
        if (tid == 0) tma_store_wait_read();  // the previous chunk's dh_c store has read a_ds
        __syncthreads();
        for (int kc = 0; kc < 4; ++kc) {
            float r[32];
            tmem_ld32(tS + kc * 32, r);
            tmem_ld_wait();
            unsigned char *sub = sm.a_ds + (kc >> 1) * (128 * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int col = (kc & 1) * 32 + q * 8;
                *reinterpret_cast<uint4 *>(sub + sw128_off(v, col)) = make_uint4(
                    pack_bf2(r[q * 8 + 0], r[q * 8 + 1]), pack_bf2(r[q * 8 + 2], r[q * 8 + 3]),
                    pack_bf2(r[q * 8 + 4], r[q * 8 + 5]), pack_bf2(r[q * 8 + 6], r[q * 8 + 7]));
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= egl;
            tmem_st32(tS + kc * 32, r);
        }
        tmem_st_wait();
        if (!mbar_wait(&sm.tma_bar[st], (i >> 1) & 1)) sm.error = 1;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (sm.error) { ok = false; break; }
        // 2. Pd = dS' K^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t as = smem_u32(sm.a_ds), ks = smem_u32(sm.stage[st]);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tP, sdesc(as + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                         sdesc(ks + (s >> 2) * kTileBytes + (s & 3) * 32, 16, 1024), idP, s > 0);
            mma_commit(&sm.mma_bar);
            const int hrow = (c * a.HV + hv) * 128;  // dh_c^T rows of this chunk
            tma_store_3d(&maps.dhc, 0, 0, hrow, sm.a_ds);
            tma_store_3d(&maps.dhc, 64, 0, hrow, sm.a_ds + 128 * 128);
            tma_store_commit();
        }
        // meanwhile: A_DO[v][t] = qc_t dO[t][v]
        {
            const unsigned char *dos = sm.stage[st] + 6 * kTileBytes + (v >> 6) * kTileBytes;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = q * 8 + 2 * e;
                    const float d0 = bf2f(*reinterpret_cast<const bf16 *>(dos + sw128_off(t, v & 63)));
                    const float d1 = bf2f(*reinterpret_cast<const bf16 *>(dos + sw128_off(t + 1, v & 63)));
                    pk[e] = pack_bf2(d0 * sm.qc[t], d1 * sm.qc[t + 1]);
                }
                *reinterpret_cast<uint4 *>(sm.a_do + sw128_off(v, q * 8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) sm.error = 1;
        mma_phase ^= 1;
        tc_fence_after();
        // 3. dv_new^T = dv_loc^T + kc_t Pd  (dv_loc from the chunk's TMA tile)
        const unsigned char *dls = sm.stage[st] + 8 * kTileBytes + (v >> 6) * kTileBytes;
        for (int tc = 0; tc < 2; ++tc) {
            float p[32], dl[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                dl[j] = bf2f(*reinterpret_cast<const bf16 *>(dls + sw128_off(tc * 32 + j, v & 63)));
            tmem_ld32(tP + tc * 32, p);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x2[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int t = tc * 32 + q * 8 + 2 * e + z;
                        float dvn = 0.f;
                        if (t < L) {
                            const size_t o = ((size_t)(t0 + t) * a.HV + hv) * kDim + v;
                            dvn = dl[q * 8 + 2 * e + z] + sm.kc[t] * p[q * 8 + 2 * e + z];
                            a.dvnew[o] = f2bf(dvn);
                        }
                        x2[z] = -dvn;
                    }
                    pk[e] = pack_bf2(x2[0], x2[1]);
                }
                *reinterpret_cast<uint4 *>(sm.a_dv + sw128_off(v, tc * 32 + q * 8)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 4. dS += A_DO Q + A_DV w
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ado = smem_u32(sm.a_do), adv = smem_u32(sm.a_dv);
            const uint32_t qs = smem_u32(sm.stage[st] + 2 * kTileBytes);
            const uint32_t ws = smem_u32(sm.stage[st] + 4 * kTileBytes);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS, sdesc(ado + s * 32, 16, 1024), sdesc(qs + s * 2048, kTileBytes, 1024), idS, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS, sdesc(adv + s * 32, 16, 1024), sdesc(ws + s * 2048, kTileBytes, 1024), idS, true);
            mma_commit(&sm.mma_bar);
        }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) sm.error = 1;
        mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (sm.error) { ok = false; break; }
        if (tid == 0 && i + 2 < nch) issue_stage(maps, sm, st, a.chunk_start[c - 2], h, hv);
    }
    if (ok && a.dh0) {
        for (int kc = 0; kc < 4; ++kc) {
            float r[32];
            tmem_ld32(tS + kc * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) a.dh0[sbase + (size_t)(kc * 32 + j) * kDim + v] = r[j];
        }
    }
    if (tid == 0) tma_store_wait_all();
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        mbar_wait(&sm.tma_bar[0], 0, 1u << 20);
        mbar_wait(&sm.tma_bar[1], 0, 1u << 20);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(sm.tmem_base, 256);
}

}  // namespace

cudaError_t launch_bstate_tc(const ChunkArgs &a, cudaStream_t s) {
    BStateMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 128 * 2;
    if (a.T > 0 && (!encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
                    !encode_rows_bf16(&m.q, a.q, a.H, a.T, rowb, rowb * a.H, 64) ||
                    !encode_rows_bf16(&m.w, a.w, a.HV, a.T, rowb, rowb * a.HV, 64) ||
                    !encode_rows_bf16(&m.dO, a.d_o, a.HV, a.T, rowb, rowb * a.HV, 64) ||
                    !encode_rows_bf16(&m.dl, a.dvloc, a.HV, a.T, rowb, rowb * a.HV, 64) ||
                    !encode_rows_bf16(&m.dhc, a.dhc, 1, (uint64_t)a.num_chunks * a.HV * 128, rowb,
                                      rowb, 128)))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BStateSmem) + 1024;
    static_assert(sizeof(BStateSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k_bstate_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
    k_bstate_tc<<<dim3(a.HV, a.N), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
