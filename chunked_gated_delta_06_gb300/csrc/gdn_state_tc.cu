// gdn_state_tc.cu -- forward inter-chunk state scan on the tensor cores.
//
// One CTA of 128 threads per (sequence, value head) walks the sequence's
// chunks in order ("cake_gdn: deterministic chunked GDN training kernels",
// Summary: fp32 running state across chunks, per-chunk h stored in bf16).
// The running state is kept transposed, S = h^T (V x K), as an fp32
// accumulator in TMEM: lane v holds row v, columns 0..127 hold k.  Per chunk
// (L <= 64 tokens starting at t0, G the chunk-local cumsum of g, G_L its last
// value):
//   1. thread v reads row v of S, writes it as bf16 to shared memory (MMA
//      operand) and e^{G_L} S back to TMEM; one TMA store copies the bf16 tile
//      to h_c[chunk][hv] (stored transposed, [v][k]);
//   2. P = S_bf16 w^T                      (tcgen05, M=128 N=64 K=128)
//   3. v_new^T[v][t] = u[t][v] - P[v][t]  -> v_new in HBM (bf16), and the
//      operand A_V[v][t] = v_new^T[v][t] e^{G_L - G_t} / r_k,t (bf16, smem)
//   4. S += A_V K                           (tcgen05, M=128 N=128 K=64; K is the
//      raw key tile read as an MN-major operand)
// which is h <- e^{G_L} h + (diag(e^{G_L-G}) Khat)^T v_new with
// Khat = diag(1 / r_k) K.  w, u and K tiles stream in by TMA two chunks ahead.
// Every wait is bounded; a timeout sets status bit 2 and the CTA unwinds.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
constexpr uint32_t kTileBytes = 64 * 128;          // one 64 x 64 bf16 SW128 box
constexpr uint32_t kStageBytes = 6 * kTileBytes;   // w (2 boxes), K (2), u (2)

struct StateSmem {
    // 1024-byte aligned operand tiles first
    unsigned char a_s[2 * 128 * 128];   // S bf16 [v][k]: two k-halves of 128 x 128 B
    unsigned char a_v[128 * 128];       // A_V bf16 [v][t]: 128 x 128 B
    unsigned char stage[2][kStageBytes];
    float coef[2][64];                  // e^{G_L - G_t} / r_k,t, 0 past L
    float gt[64], rkt[64];              // this chunk's G and r_k (prefetched)
    uint64_t tma_bar[2];
    uint64_t mma_bar;
    uint32_t tmem_base;
    int error;
};

struct StateMaps {
    CUtensorMap w, k, u, hc;
};

__device__ __forceinline__ void issue_stage(const StateMaps &m, StateSmem &sm, int st, int t0, int h,
                                            int hv) {
    unsigned char *b = sm.stage[st];
    mbar_arrive_expect_tx(&sm.tma_bar[st], kStageBytes);
    tma_load_3d(b + 0 * kTileBytes, &m.w, 0, hv, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 1 * kTileBytes, &m.w, 64, hv, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 2 * kTileBytes, &m.k, 0, h, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 3 * kTileBytes, &m.k, 64, h, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 4 * kTileBytes, &m.u, 0, hv, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 5 * kTileBytes, &m.u, 64, hv, t0, &sm.tma_bar[st]);
}

__global__ void __launch_bounds__(kThr, 1)
    k_state_tc(const ChunkArgs a, const __grid_constant__ StateMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    StateSmem &sm = *reinterpret_cast<StateSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int hv = blockIdx.x, n = a.seq_order[blockIdx.y];  // longest sequences first
    const int h = hv / (a.HV / a.H);
    const int v = tid;  // the state row this thread owns
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
    const uint32_t tmem = sm.tmem_base;
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's lanes
    const uint32_t tS = t_row, tP = t_row + 128;

    if (tid == 0) {
        for (int i = 0; i < 2 && i < nch; ++i) issue_stage(maps, sm, i, a.chunk_start[cb + i], h, hv);
    }
    // S <- h0^T (row v = column v of h0[n][hv])
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim;
    for (int kc = 0; kc < 4; ++kc) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            r[j] = a.h0 ? a.h0[sbase + (size_t)(kc * 32 + j) * kDim + v] : 0.f;
        tmem_st32(tS + kc * 32, r);
    }
    tmem_st_wait();

    const uint32_t idP = idesc_bf16(128, 64, 0, 0);    // P = S w^T
    const uint32_t idS = idesc_bf16(128, 128, 0, 1);   // S += A_V K  (K MN-major)
    uint32_t mma_phase = 0;
    bool ok = true;
    // per-token scalars of the next chunk, loaded one chunk ahead
    float pg = 0.f, prk = 1.f;
    auto fetch = [&](int cc) {
        const int tt0 = a.chunk_start[cc], LL = a.chunk_len[cc];
        if (tid < LL) {
            const size_t t = (size_t)(tt0 + tid);
            pg = a.G[t * a.HV + hv];
            prk = a.rk[t * a.H + h];
        } else {
            pg = 0.f; prk = 1.f;
        }
    };
    if (tid < 64 && nch > 0) fetch(cb);
    for (int i = 0; i < nch && ok; ++i) {
        const int c = cb + i, st = i & 1;
        const int t0 = a.chunk_start[c], L = a.chunk_len[c];
        if (tid < 64) {
            sm.gt[tid] = pg;
            sm.rkt[tid] = prk;
            if (i + 1 < nch) fetch(c + 1);
        }
        __syncthreads();
        const float Gl = L > 0 ? sm.gt[L - 1] : 0.f;
        if (tid < 64) sm.coef[st][tid] = tid < L ? expf(Gl - sm.gt[tid]) / sm.rkt[tid] : 0.f;
        const float egl = expf(Gl);
        // 1. S -> bf16 operand (copied to h_c by TMA below), then S <- e^{G_L} S
        if (tid == 0) tma_store_wait_read();  // the previous chunk's h_c store has read a_s
        __syncthreads();
        for (int kc = 0; kc < 4; ++kc) {
            float r[32];
            tmem_ld32(tS + kc * 32, r);
            tmem_ld_wait();
            unsigned char *sub = sm.a_s + (kc >> 1) * (128 * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 4 chunks of 8 columns
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 two = __floats2bfloat162_rn(r[q * 8 + 2 * e], r[q * 8 + 2 * e + 1]);
                    pk[e] = *reinterpret_cast<uint32_t *>(&two);
                }
                const int col = (kc & 1) * 32 + q * 8;
                *reinterpret_cast<uint4 *>(sub + sw128_off(v, col)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= egl;
            tmem_st32(tS + kc * 32, r);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 2. P = S_bf16 w^T (every thread waits for the chunk's tiles: u is read below)
        if (!mbar_wait(&sm.tma_bar[st], (i >> 1) & 1)) sm.error = 1;
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            if (!sm.error) {
                const uint32_t as = smem_u32(sm.a_s), ws = smem_u32(sm.stage[st]);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16(tP, sdesc(as + (s >> 2) * 16384 + (s & 3) * 32, 16, 1024),
                             sdesc(ws + (s >> 2) * kTileBytes + (s & 3) * 32, 16, 1024), idP, s > 0);
                mma_commit(&sm.mma_bar);
                const int hrow = (c * a.HV + hv) * 128;  // h_c^T rows of this chunk
                tma_store_3d(&maps.hc, 0, 0, hrow, sm.a_s);
                tma_store_3d(&maps.hc, 64, 0, hrow, sm.a_s + 128 * 128);
                tma_store_commit();
            }
        }
        __syncthreads();
        if (sm.error) { ok = false; break; }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) { sm.error = 1; }
        mma_phase ^= 1;
        tc_fence_after();
        // 3. v_new^T = u^T - P
        const unsigned char *us = sm.stage[st] + 4 * kTileBytes + (v >> 6) * kTileBytes;
        unsigned char *avs = sm.a_v;
        for (int tc = 0; tc < 2; ++tc) {
            float p[32];
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
                        float vn = 0.f;
                        if (t < L) {
                            const float uu = bf2f(*reinterpret_cast<const bf16 *>(us + sw128_off(t, v & 63)));
                            vn = uu - p[q * 8 + 2 * e + z];
                            a.vnew[((size_t)(t0 + t) * a.HV + hv) * kDim + v] = f2bf(vn);
                        }
                        x2[z] = vn * sm.coef[st][t];
                    }
                    __nv_bfloat162 two = __floats2bfloat162_rn(x2[0], x2[1]);
                    pk[e] = *reinterpret_cast<uint32_t *>(&two);
                }
                *reinterpret_cast<uint4 *>(avs + sw128_off(v, tc * 32 + q * 8)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // 4. S += A_V K
        if (tid == 0) {
            tc_fence_after();
            const uint32_t av = smem_u32(sm.a_v), ks = smem_u32(sm.stage[st] + 2 * kTileBytes);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tS, sdesc(av + s * 32, 16, 1024), sdesc(ks + s * 2048, kTileBytes, 1024), idS,
                         true);
            mma_commit(&sm.mma_bar);
        }
        if (!mbar_wait(&sm.mma_bar, mma_phase)) sm.error = 1;
        mma_phase ^= 1;
        tc_fence_after();
        __syncthreads();
        if (sm.error) { ok = false; break; }
        if (tid == 0 && i + 2 < nch) issue_stage(maps, sm, st, a.chunk_start[c + 2], h, hv);
    }
    if (ok && a.ht) {
        for (int kc = 0; kc < 4; ++kc) {
            float r[32];
            tmem_ld32(tS + kc * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) a.ht[sbase + (size_t)(kc * 32 + j) * kDim + v] = r[j];
        }
    }
    if (tid == 0) tma_store_wait_all();
    if (!ok) {
        // drain outstanding TMA copies (bounded) before leaving
        if (tid == 0) {
            if (a.status) atomicOr(a.status, 2);
            mbar_wait(&sm.tma_bar[0], 0, 1u << 20);
            mbar_wait(&sm.tma_bar[1], 0, 1u << 20);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_state_tc(const ChunkArgs &a, cudaStream_t s) {
    StateMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 128 * 2;
    if (a.T > 0 && (!encode_rows_bf16(&m.w, a.w, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.u, a.u, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.hc, a.hc, 1, (uint64_t)a.num_chunks * a.HV * 128, rowb, rowb, 128)))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(StateSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(k_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_STATE, s);
    k_state_tc<<<dim3(a.HV, a.N), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
