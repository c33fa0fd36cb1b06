// gdn_bstate_tc.cu -- backward (reverse) inter-chunk state scan on the tensor
// cores ("dhu" in "cake_gdn: deterministic chunked GDN training kernels",
// section 2; the reverse recurrence of the GDN context-parallel dh scan in
// "Qwen3.5-397B RL trainer on 128 v7x", maxtext #5799).
//
// As in the forward scan, the value columns never mix, so one CTA of 128
// threads owns one (sequence, value head, value half) and walks the chunks in
// reverse.  dh[k][v'] (v' = 64 vb .. 64 vb + 63) lives in TMEM as fp32 (lane
// k, 64 columns), seeded with d(final state).  Per chunk, with dh' the gradient
// of the state after the chunk (= the current dh):
//   1. thread k writes row k of dh' as bf16 to shared memory (copied to
//      dh_c[chunk][hv][k][v'] by one TMA store), then dh <- e^{G_L} dh';
//   2. Pd[t][v'] = sum_k K[t][k] dh'[k][v']          (M=64 N=64 K=128)
//   3. thread t forms whole rows dv_new[t][v'] = dv_loc + e^{G_L-G_t}/r_k,t Pd
//      (to HBM, bf16) and the operands c_t dO[t][v'] and -dv_new[t][v'],
//      c_t = e^{G_t} scale / r_q,t;
//   4. dh += Q^T (c dO) - w^T dv_new                  (two M=128 N=64 K=64
//      products; Q and w are raw tiles read MN-major)
// which is dh <- e^{G_L} dh' + Qtil^T dO - w^T dv_new and dv_new = dv_loc +
// Ktil dh'.  dh0 = dh at the sequence start.  The tiles come in two single-
// buffered groups so that two CTAs share an SM: X (K, this half of dO and of
// dv_loc) is reloaded for the next chunk as soon as step 3 has read it, Y (Q, w)
// as soon as step 4 has finished.  Waits are bounded.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
constexpr uint32_t kBox = 64 * 128;       // one 64-row x 128-byte SW128 box
constexpr uint32_t kXBytes = 4 * kBox;    // K (2 boxes), dO half, dv_loc half
constexpr uint32_t kYBytes = 4 * kBox;    // Q (2 boxes), w (2 boxes)

struct BStateSmem {
    unsigned char a_ds[128 * 128];      // dh' bf16 [k][v']
    unsigned char a_do[64 * 128];       // c_t dO bf16 [t][v']
    unsigned char a_dv[64 * 128];       // -dv_new bf16 [t][v']
    unsigned char x[kXBytes];
    unsigned char y[kYBytes];
    float kc[64];                       // e^{G_L - G_t} / r_k,t (0 past L)
    float qc[64];                       // e^{G_t} scale / r_q,t (0 past L)
    float gt[64], rkt[64], rqt[64];     // this chunk's G, r_k, r_q (prefetched)
    uint64_t x_bar, y_bar, mma_bar;
    uint32_t tmem_base;
    int error;
};

struct BStateMaps {
    CUtensorMap k, q, w, dO, dl, dhc;
};

__device__ __forceinline__ void issue_x(const BStateMaps &m, BStateSmem &sm, int t0, int h, int hv,
                                        int vb) {
    mbar_arrive_expect_tx(&sm.x_bar, kXBytes);
    tma_load_3d(sm.x + 0 * kBox, &m.k, 0, h, t0, &sm.x_bar);
    tma_load_3d(sm.x + 1 * kBox, &m.k, 64, h, t0, &sm.x_bar);
    tma_load_3d(sm.x + 2 * kBox, &m.dO, 64 * vb, hv, t0, &sm.x_bar);
    tma_load_3d(sm.x + 3 * kBox, &m.dl, 64 * vb, hv, t0, &sm.x_bar);
}

__device__ __forceinline__ void issue_y(const BStateMaps &m, BStateSmem &sm, int t0, int h, int hv) {
    mbar_arrive_expect_tx(&sm.y_bar, kYBytes);
    tma_load_3d(sm.y + 0 * kBox, &m.q, 0, h, t0, &sm.y_bar);
    tma_load_3d(sm.y + 1 * kBox, &m.q, 64, h, t0, &sm.y_bar);
    tma_load_3d(sm.y + 2 * kBox, &m.w, 0, hv, t0, &sm.y_bar);
    tma_load_3d(sm.y + 3 * kBox, &m.w, 64, hv, t0, &sm.y_bar);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThr, 2)
    k_bstate_tc(const ChunkArgs a, const __grid_constant__ BStateMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BStateSmem &sm = *reinterpret_cast<BStateSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hv = blockIdx.x >> 1, vb = blockIdx.x & 1;
    const int n = a.seq_order[blockIdx.y];  // longest sequences first
    const int h = hv / (a.HV / a.H);
    const int cb = a.seq_chunk_off[n];
    const int ce = min(a.seq_chunk_off[n + 1], a.num_chunks);
    const int nch = max(ce - cb, 0);
    const int kr = tid;                 // the state row this thread owns (step 1)
    const int tr = 16 * warp + lane;    // the token row it owns (lanes 0..15)
    const bool trow = lane < 16;

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.x_bar, 1);
        mbar_init(&sm.y_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
        sm.error = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t_row = sm.tmem_base + ((uint32_t)(warp * 32) << 16);
    const uint32_t tS = t_row, tP = t_row + 64;

    int x_issued = 0, y_issued = 0;  // loads issued (thread 0's count)
    if (tid == 0 && nch > 0) {
        issue_x(maps, sm, a.chunk_start[ce - 1], h, hv, vb);
        issue_y(maps, sm, a.chunk_start[ce - 1], h, hv);
        x_issued = y_issued = 1;
    }
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim + (size_t)kr * kDim + 64 * vb;
    for (int half = 0; half < 2; ++half) {
        float r[32];
        if (a.d_ht) {
            const float4 *src = reinterpret_cast<const float4 *>(a.d_ht + sbase + 32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = src[q];
                r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0.f;
        }
        tmem_st32(tS + 32 * half, r);
    }
    tmem_st_wait();

    const uint32_t idP = idesc_bf16(64, 64, 0, 1);    // Pd = K dh'          (dh' MN-major)
    const uint32_t idS = idesc_bf16(128, 64, 1, 1);   // dh += Q^T A + w^T B (all MN-major)
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
        const int c = ce - 1 - i;
        const uint32_t par = i & 1;
        const int t0 = a.chunk_start[c], L = a.chunk_len[c];
        if (tid < 64) {
            sm.gt[tid] = pg;
            sm.rkt[tid] = prk;
            sm.rqt[tid] = prq;
            if (i + 1 < nch) fetch(c - 1);
        }
        if (tid == 0) tma_store_wait_read();  // the previous chunk's dh_c store has read a_ds
        __syncthreads();
        const float Gl = L > 0 ? sm.gt[L - 1] : 0.f;
        if (tid < 64) {
            float kk = 0.f, qq = 0.f;
            if (tid < L) {
                const float Gt = sm.gt[tid];
                kk = __expf(fminf(Gl - Gt, 0.f)) / sm.rkt[tid];
                qq = __expf(Gt) * a.scale / sm.rqt[tid];
            }
            sm.kc[tid] = kk;
            sm.qc[tid] = qq;
        }
        const float egl = __expf(Gl);
        // 1. dh' -> bf16 operand row kr (copied to dh_c by TMA below), then dh <- e^{G_L} dh'
        {
            float r0[32], r1[32];
            tmem_ld32(tS, r0);
            tmem_ld32(tS + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4 *>(sm.a_ds + sw128_off(kr, 8 * q)) =
                    make_uint4(pack_bf2(r0[8 * q], r0[8 * q + 1]), pack_bf2(r0[8 * q + 2], r0[8 * q + 3]),
                               pack_bf2(r0[8 * q + 4], r0[8 * q + 5]), pack_bf2(r0[8 * q + 6], r0[8 * q + 7]));
                *reinterpret_cast<uint4 *>(sm.a_ds + sw128_off(kr, 32 + 8 * q)) =
                    make_uint4(pack_bf2(r1[8 * q], r1[8 * q + 1]), pack_bf2(r1[8 * q + 2], r1[8 * q + 3]),
                               pack_bf2(r1[8 * q + 4], r1[8 * q + 5]), pack_bf2(r1[8 * q + 6], r1[8 * q + 7]));
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                r0[j] *= egl;
                r1[j] *= egl;
            }
            tmem_st32(tS, r0);
            tmem_st32(tS + 32, r1);
        }
        tmem_st_wait();
        if (!mbar_wait(&sm.x_bar, par)) sm.error = 1;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (sm.error) { ok = false; break; }
        // 2. Pd = K dh'
        if (tid == 0) {
            tc_fence_after();
            const uint32_t as = smem_u32(sm.a_ds), ks = smem_u32(sm.x);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tP, sdesc(ks + (s >> 2) * kBox + (s & 3) * 32, 16, 1024),
                         sdesc(as + s * 2048, kBox, 1024), idP, s > 0);
            mma_commit(&sm.mma_bar);
            const int hrow = (c * a.HV + hv) * 128;  // dh_c rows (k) of this chunk
            tma_store_3d(&maps.dhc, 64 * vb, 0, hrow, sm.a_ds);
            tma_store_commit();
        }
        // meanwhile: row tr of c_t dO
        if (trow) {
            const float qc = sm.qc[tr];
            const unsigned char *dos = sm.x + 2 * kBox;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 dx = *reinterpret_cast<const uint4 *>(dos + sw128_off(tr, 8 * q));
                const __nv_bfloat162 *db = reinterpret_cast<const __nv_bfloat162 *>(&dx);
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(db[e]);
                    pk[e] = pack_bf2(f.x * qc, f.y * qc);
                }
                *reinterpret_cast<uint4 *>(sm.a_do + sw128_off(tr, 8 * q)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) sm.error = 1;
        mma_phase ^= 1;
        tc_fence_after();
        // 3. dv_new = dv_loc + kc_t Pd, row tr
        {
            float p0[32], p1[32];
            tmem_ld32(tP, p0);
            tmem_ld32(tP + 32, p1);
            tmem_ld_wait();
            if (trow) {
                const bool live = tr < L;
                const float kc = sm.kc[tr];
                const unsigned char *dls = sm.x + 3 * kBox;
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.dvnew + ((size_t)(t0 + (live ? tr : 0)) * a.HV + hv) * kDim + 64 * vb);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 lx = *reinterpret_cast<const uint4 *>(dls + sw128_off(tr, 8 * q));
                    const __nv_bfloat162 *lb = reinterpret_cast<const __nv_bfloat162 *>(&lx);
                    float dv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 lf = __bfloat1622float2(lb[e]);
                        const int j = 8 * q + 2 * e;
                        const float pa = j < 32 ? p0[j & 31] : p1[j & 31];
                        const float pb = j + 1 < 32 ? p0[(j + 1) & 31] : p1[(j + 1) & 31];
                        dv[2 * e] = live ? lf.x + kc * pa : 0.f;
                        dv[2 * e + 1] = live ? lf.y + kc * pb : 0.f;
                    }
                    if (live)
                        dst[q] = make_uint4(pack_bf2(dv[0], dv[1]), pack_bf2(dv[2], dv[3]),
                                            pack_bf2(dv[4], dv[5]), pack_bf2(dv[6], dv[7]));
                    *reinterpret_cast<uint4 *>(sm.a_dv + sw128_off(tr, 8 * q)) =
                        make_uint4(pack_bf2(-dv[0], -dv[1]), pack_bf2(-dv[2], -dv[3]),
                                   pack_bf2(-dv[4], -dv[5]), pack_bf2(-dv[6], -dv[7]));
                }
            }
        }
        if (!mbar_wait(&sm.y_bar, par)) sm.error = 1;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();  // X has been read by step 2 and 3
        if (sm.error) { ok = false; break; }
        // 4. dh += Q^T (c dO) - w^T dv_new; X is free for the next chunk
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ado = smem_u32(sm.a_do), adv = smem_u32(sm.a_dv);
            const uint32_t qs = smem_u32(sm.y), ws = smem_u32(sm.y + 2 * kBox);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS, sdesc(qs + s * 2048, kBox, 1024), sdesc(ado + s * 2048, kBox, 1024), idS, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS, sdesc(ws + s * 2048, kBox, 1024), sdesc(adv + s * 2048, kBox, 1024), idS, true);
            mma_commit(&sm.mma_bar);
            if (i + 1 < nch) {
                issue_x(maps, sm, a.chunk_start[c - 1], h, hv, vb);
                ++x_issued;
            }
        }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) sm.error = 1;
        mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (sm.error) { ok = false; break; }
        if (tid == 0 && i + 1 < nch) {  // Y is free once step 4 has finished
            issue_y(maps, sm, a.chunk_start[c - 1], h, hv);
            ++y_issued;
        }
    }
    if (ok && a.dh0) {
        for (int half = 0; half < 2; ++half) {
            float r[32];
            tmem_ld32(tS + 32 * half, r);
            tmem_ld_wait();
            float4 *dst = reinterpret_cast<float4 *>(a.dh0 + sbase + 32 * half);
#pragma unroll
            for (int q = 0; q < 8; ++q) dst[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        }
    }
    if (tid == 0) tma_store_wait_all();
    if (!ok && tid == 0) {
        // drain the loads still in flight (bounded) before leaving
        if (a.status) atomicOr(a.status, 2);
        if (x_issued > 0) mbar_wait(&sm.x_bar, (x_issued - 1) & 1, 1u << 20);
        if (y_issued > 0) mbar_wait(&sm.y_bar, (y_issued - 1) & 1, 1u << 20);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(sm.tmem_base, 128);
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
    static_assert(2 * (sizeof(BStateSmem) + 2048) <= 233472, "two CTAs per SM");
    cudaError_t e = cudaFuncSetAttribute(k_bstate_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
    k_bstate_tc<<<dim3(2 * a.HV, a.N), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
