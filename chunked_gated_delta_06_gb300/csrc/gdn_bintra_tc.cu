// gdn_bintra_tc.cu -- backward terms of a chunk that go through the per-chunk
// states h (chunk start) and dh' (gradient of the state after the chunk), on
// the tensor cores ("dqkwg" of "cake_gdn: deterministic chunked GDN training
// kernels", section 2).
//
// One CTA of 256 threads per (chunk, value head).  With h_c, dh_c [k][v]
// (bf16, from the forward and reverse scans) and dO, dv_new, v_new [t][v]:
//   Dq[t][k] = sum_v dO[t][v] h[k][v]         dqhat_t = e^{G_t} Dq[t]
//   Dw[t][k] = sum_v dv_new[t][v] h[k][v]     dW_t    = -Dw[t]
//   Dk[t][k] = sum_v v_new[t][v] dh'[k][v]    dkhat_t = e^{G_L - G_t} Dk[t]
// three M=64 N=128 K=128 tcgen05 products (A = the token tiles, K-major;
// B = h / dh' as [N=k][K=v], i.e. their [k][v] tiles read K-major; all loaded
// by TMA).  An M=64 result row t
// sits in TMEM lane 32 (t / 16) + t % 16; the two warpgroups each take 64 of
// its 128 columns.  It also forms the gate-gradient pieces of these terms:
//   dG_t  = qhat_t . dqhat_t - xi_t,  xi_t = khat_t . dkhat_t,
//   dG_L += sum_t xi_t + e^{G_L} <h, dh'>.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 256;
constexpr uint32_t kBox = 64 * 128;       // 64 rows x 128 B
constexpr uint32_t kBig = 128 * 128;      // 128 rows x 128 B

struct BaSmem {
    unsigned char h[2 * kBig];    // h_c [k][v]: two v-halves of 128 rows
    unsigned char dh[2 * kBig];   // dh_c [k][v]
    unsigned char dO[2 * kBox];   // [t][v]
    unsigned char dvn[2 * kBox];
    unsigned char vn[2 * kBox];
    unsigned char q[2 * kBox];    // [t][k]
    unsigned char k[2 * kBox];
    float pq[2][64], pk[2][64];   // per-warpgroup partial row dots
    float hdh[kThr / 32];
    float eg[64], egl_g[64];      // e^{G_t}, e^{G_L - G_t} (0 past L)
    float qsc[64], rki[64];       // scale / r_q, 1 / r_k
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

struct BaMaps {
    CUtensorMap h, dh, dO, dvn, vn, q, k;
};

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

__global__ void __launch_bounds__(kThr, 1) k_bintra_a_tc(const ChunkArgs a,
                                                         const __grid_constant__ BaMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BaSmem &sm = *reinterpret_cast<BaSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, hv = blockIdx.y;
    const int h = hv / (a.HV / a.H);
    const int t0 = a.chunk_start[c], L = a.chunk_len[c];
    if (L <= 0) return;
    const bool active = lane < 16;
    const int grp = warp >> 2;
    const int t = (warp & 3) * 16 + lane;  // the token row this lane owns (valid when active)

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
        const int row = (c * a.HV + hv) * 128;
        mbar_arrive_expect_tx(&sm.tma_bar, 4 * kBig + 10 * kBox);
        tma_load_3d(sm.h, &maps.h, 0, 0, row, &sm.tma_bar);
        tma_load_3d(sm.h + kBig, &maps.h, 64, 0, row, &sm.tma_bar);
        tma_load_3d(sm.dh, &maps.dh, 0, 0, row, &sm.tma_bar);
        tma_load_3d(sm.dh + kBig, &maps.dh, 64, 0, row, &sm.tma_bar);
        tma_load_3d(sm.dO, &maps.dO, 0, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.dO + kBox, &maps.dO, 64, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.dvn, &maps.dvn, 0, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.dvn + kBox, &maps.dvn, 64, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.vn, &maps.vn, 0, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.vn + kBox, &maps.vn, 64, hv, t0, &sm.tma_bar);
        tma_load_3d(sm.q, &maps.q, 0, h, t0, &sm.tma_bar);
        tma_load_3d(sm.q + kBox, &maps.q, 64, h, t0, &sm.tma_bar);
        tma_load_3d(sm.k, &maps.k, 0, h, t0, &sm.tma_bar);
        tma_load_3d(sm.k + kBox, &maps.k, 64, h, t0, &sm.tma_bar);
    }
    const float Gl = a.G[(size_t)(t0 + L - 1) * a.HV + hv];
    if (tid < 64) {
        const bool in = tid < L;
        const size_t r = (size_t)(t0 + tid) * a.H + h;
        const float Gt = in ? a.G[(size_t)(t0 + tid) * a.HV + hv] : 0.f;
        sm.eg[tid] = in ? __expf(Gt) : 0.f;
        sm.egl_g[tid] = in ? __expf(fminf(Gl - Gt, 0.f)) : 0.f;
        sm.qsc[tid] = in ? a.scale / a.rq[r] : 0.f;
        sm.rki[tid] = in ? 1.f / a.rk[r] : 0.f;
    }
    const bool got = __syncthreads_and(mbar_wait(&sm.tma_bar, 0));
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)((warp & 3) * 32) << 16);
    if (tid == 0 && got) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 128, 0, 0);
        const uint32_t hs = smem_u32(sm.h), dhs = smem_u32(sm.dh);
        const uint32_t os = smem_u32(sm.dO), ds = smem_u32(sm.dvn), vs = smem_u32(sm.vn);
        for (int s = 0; s < 8; ++s) {
            const uint32_t ao = (s >> 2) * kBox + (s & 3) * 32, bo = (s >> 2) * kBig + (s & 3) * 32;
            mma_bf16(tb + 0, sdesc(os + ao, 16, 1024), sdesc(hs + bo, 16, 1024), id, s > 0);
            mma_bf16(tb + 128, sdesc(ds + ao, 16, 1024), sdesc(hs + bo, 16, 1024), id, s > 0);
            mma_bf16(tb + 256, sdesc(vs + ao, 16, 1024), sdesc(dhs + bo, 16, 1024), id, s > 0);
        }
        mma_commit(&sm.mma_bar);
    }
    // <h, dh'> while the products run: thread tid takes half a row of h and dh'
    float hdh = 0.f;
    if (got) {
        const int kr = tid >> 1, half = tid & 1;
        const unsigned char *hr = sm.h + half * kBig, *dr = sm.dh + half * kBig;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            const uint32_t off = sw128_off(kr, q8 * 8);
            const uint4 x = *reinterpret_cast<const uint4 *>(hr + off);
            const uint4 y = *reinterpret_cast<const uint4 *>(dr + off);
            const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&x);
            const __nv_bfloat162 *yb = reinterpret_cast<const __nv_bfloat162 *>(&y);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xf = __bfloat1622float2(xb[e]), yf = __bfloat1622float2(yb[e]);
                hdh += xf.x * yf.x + xf.y * yf.y;
            }
        }
    }
    hdh = warp_sum(hdh);
    if (lane == 0) sm.hdh[warp] = hdh;
    const bool done = __syncthreads_and(got && mbar_wait(&sm.mma_bar, 0));
    tc_fence_after();
    if (done) {
        const bool live = active && t < L;
        const float eg = live ? sm.eg[t] : 0.f, el = live ? sm.egl_g[t] : 0.f;
        const size_t o = ((size_t)(t0 + (live ? t : 0)) * a.HV + hv) * kDim;
        float xq = 0.f, xk = 0.f;
        for (int cc = 2 * grp; cc < 2 * grp + 2; ++cc) {  // this warpgroup's 64 columns
            float dq[32], dw[32], dk[32];
            tmem_ld32(t_row + 0 + cc * 32, dq);
            tmem_ld32(t_row + 128 + cc * 32, dw);
            tmem_ld32(t_row + 256 + cc * 32, dk);
            tmem_ld_wait();
            if (live) {
                float4 *qp = reinterpret_cast<float4 *>(a.dqp + o + cc * 32);
                float4 *kp = reinterpret_cast<float4 *>(a.dkp + o + cc * 32);
                const unsigned char *qrow = sm.q + (cc >> 1) * kBox, *krow = sm.k + (cc >> 1) * kBox;
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {  // 8 columns per step
                    const int col = (cc & 1) * 32 + q8 * 8;
                    const uint4 qx = *reinterpret_cast<const uint4 *>(qrow + sw128_off(t, col));
                    const uint4 kx = *reinterpret_cast<const uint4 *>(krow + sw128_off(t, col));
                    const __nv_bfloat162 *qb = reinterpret_cast<const __nv_bfloat162 *>(&qx);
                    const __nv_bfloat162 *kb = reinterpret_cast<const __nv_bfloat162 *>(&kx);
                    float dqv[8], dkv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 qf = __bfloat1622float2(qb[e]), kf = __bfloat1622float2(kb[e]);
                        dqv[2 * e] = eg * dq[q8 * 8 + 2 * e];
                        dqv[2 * e + 1] = eg * dq[q8 * 8 + 2 * e + 1];
                        dkv[2 * e] = el * dk[q8 * 8 + 2 * e];
                        dkv[2 * e + 1] = el * dk[q8 * 8 + 2 * e + 1];
                        xq += qf.x * dqv[2 * e] + qf.y * dqv[2 * e + 1];
                        xk += kf.x * dkv[2 * e] + kf.y * dkv[2 * e + 1];
                    }
                    qp[q8 * 2] = make_float4(dqv[0], dqv[1], dqv[2], dqv[3]);
                    qp[q8 * 2 + 1] = make_float4(dqv[4], dqv[5], dqv[6], dqv[7]);
                    kp[q8 * 2] = make_float4(dkv[0], dkv[1], dkv[2], dkv[3]);
                    kp[q8 * 2 + 1] = make_float4(dkv[4], dkv[5], dkv[6], dkv[7]);
                }
                uint4 *wp = reinterpret_cast<uint4 *>(a.dW + o + cc * 32);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    wp[q8] = make_uint4(pack_bf2(-dw[q8 * 8], -dw[q8 * 8 + 1]), pack_bf2(-dw[q8 * 8 + 2], -dw[q8 * 8 + 3]),
                                        pack_bf2(-dw[q8 * 8 + 4], -dw[q8 * 8 + 5]), pack_bf2(-dw[q8 * 8 + 6], -dw[q8 * 8 + 7]));
            }
        }
        if (active) {
            sm.pq[grp][t] = xq;
            sm.pk[grp][t] = xk;
        }
    } else if (tid == 0 && a.status) {
        atomicOr(a.status, 2);
    }
    __syncthreads();
    if (done && warp == 0) {  // dG_t, and the G_L terms summed in a fixed order
        float dgz[2], sx = 0.f;
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int tt = 2 * lane + z;
            float dg = 0.f, xi = 0.f;
            if (tt < L) {
                xi = (sm.pk[0][tt] + sm.pk[1][tt]) * sm.rki[tt];
                dg = (sm.pq[0][tt] + sm.pq[1][tt]) * sm.qsc[tt] - xi;
            }
            sx += xi;
            dgz[z] = dg;
        }
        sx = warp_sum(sx);
        float hd = 0.f;
#pragma unroll
        for (int w = 0; w < kThr / 32; ++w) hd += sm.hdh[w];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int tt = 2 * lane + z;
            if (tt < L) {
                const float extra = (tt == L - 1) ? sx + __expf(Gl) * hd : 0.f;
                a.dGp[(size_t)(t0 + tt) * a.HV + hv] = dgz[z] + extra;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

cudaError_t launch_bintra_a_tc(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    BaMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    const uint64_t hrows = (uint64_t)a.num_chunks * a.HV * 128;
    // h_c / dh_c as rows of 128: dims {128, 1, rows}, boxes of 128 rows x 64
    if (!encode_rows_bf16(&m.h, a.hc, 1, hrows, rowb, rowb, 128) ||
        !encode_rows_bf16(&m.dh, a.dhc, 1, hrows, rowb, rowb, 128) ||
        !encode_rows_bf16(&m.dO, a.d_o, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dvn, a.dvnew, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.vn, a.vnew, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.q, a.q, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BaSmem) + 1024;
    static_assert(sizeof(BaSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k_bintra_a_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BINTRA_A, s);
    k_bintra_a_tc<<<dim3(a.num_chunks, a.HV), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
