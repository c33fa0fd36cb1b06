// gdn_bintra_tc.cu -- backward terms of a chunk that go through the per-chunk
// states h (chunk start) and dh' (gradient of the state after the chunk), on
// the tensor cores ("dqkwg" of "cake_gdn: deterministic chunked GDN training
// kernels", section 2).
//
// One CTA of 128 threads per (chunk, value head).  With h_c, dh_c [k][v]
// (bf16, from the forward and reverse scans) and dO, dv_new, v_new [t][v]:
//   Dq[k][t] = sum_v h[k][v] dO[t][v]         dqhat_t   = e^{G_t} Dq[:,t]
//   Dw[k][t] = sum_v h[k][v] dv_new[t][v]     dW_t      = -Dw[:,t]
//   Dk[k][t] = sum_v dh'[k][v] v_new[t][v]    dkhat_t   = e^{G_L - G_t} Dk[:,t]
// three M=128 N=64 K=128 tcgen05 products with A = h / dh' and B = the token
// tiles, all K-major and loaded by TMA.  Thread k owns row k of each result.
// It also forms the gate gradient pieces of these terms:
//   dG_t  = qhat_t . dqhat_t - xi_t,  xi_t = khat_t . dkhat_t,
//   dG_L += sum_t xi_t + e^{G_L} <h, dh'>.
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
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
    float red[4][2][64];          // per-warp partial column sums
    float part[kThr / 32];
    float eg[64], egl_g[64];      // e^{G_t}, e^{G_L - G_t} (0 past L)
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

struct BaMaps {
    CUtensorMap h, dh, dO, dvn, vn, q, k;
};

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
    const int kk = tid;  // row k of the results this thread owns

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
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
        tma_load_3d(sm.q, &maps.q, 0, h, t0, &sm.tma_bar);
        tma_load_3d(sm.q + kBox, &maps.q, 64, h, t0, &sm.tma_bar);
        tma_load_3d(sm.k, &maps.k, 0, h, t0, &sm.tma_bar);
        tma_load_3d(sm.k + kBox, &maps.k, 64, h, t0, &sm.tma_bar);
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
    }
    const float Gl = a.G[(size_t)(t0 + L - 1) * a.HV + hv];
    if (tid < 64) {
        float e1 = 0.f, e2 = 0.f;
        if (tid < L) {
            const float Gt = a.G[(size_t)(t0 + tid) * a.HV + hv];
            e1 = expf(Gt);
            e2 = expf(Gl - Gt);
        }
        sm.eg[tid] = e1;
        sm.egl_g[tid] = e2;
    }
    const bool got = __syncthreads_and(mbar_wait(&sm.tma_bar, 0));
    const uint32_t t_row = sm.tmem_base + ((uint32_t)(warp * 32) << 16);
    if (tid == 0 && got) {
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 64, 0, 0);
        const uint32_t hs = smem_u32(sm.h), dhs = smem_u32(sm.dh);
        const uint32_t os = smem_u32(sm.dO), ds = smem_u32(sm.dvn), vs = smem_u32(sm.vn);
        for (int s = 0; s < 8; ++s) {
            const uint32_t ao = (s >> 2) * kBig + (s & 3) * 32, bo = (s >> 2) * kBox + (s & 3) * 32;
            mma_bf16(sm.tmem_base + 0, sdesc(hs + ao, 16, 1024), sdesc(os + bo, 16, 1024), id, s > 0);
            mma_bf16(sm.tmem_base + 64, sdesc(hs + ao, 16, 1024), sdesc(ds + bo, 16, 1024), id, s > 0);
            mma_bf16(sm.tmem_base + 128, sdesc(dhs + ao, 16, 1024), sdesc(vs + bo, 16, 1024), id, s > 0);
        }
        mma_commit(&sm.mma_bar);
    }
    // <h, dh'> row k while the products run
    float hdh = 0.f;
    if (got) {
        for (int vv = 0; vv < 128; ++vv) {
            const uint32_t off = (vv >> 6) * kBig + sw128_off(kk, vv & 63);
            hdh += bf2f(*reinterpret_cast<const bf16 *>(sm.h + off)) *
                   bf2f(*reinterpret_cast<const bf16 *>(sm.dh + off));
        }
    }
    const bool done = __syncthreads_and(got && mbar_wait(&sm.mma_bar, 0));
    tc_fence_after();
    if (!done) {
        if (tid == 0 && a.status) atomicOr(a.status, 2);
    } else {
        for (int half = 0; half < 2; ++half) {
            float rq_[32], rw_[32], rk_[32];
            tmem_ld32(t_row + 0 + half * 32, rq_);
            tmem_ld32(t_row + 64 + half * 32, rw_);
            tmem_ld32(t_row + 128 + half * 32, rk_);
            tmem_ld_wait();
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const int t = half * 32 + j;
                float xq = 0.f, xk = 0.f;
                if (t < L) {
                    const size_t o = ((size_t)(t0 + t) * a.HV + hv) * kDim + kk;
                    const uint32_t so = (kk >> 6) * kBox + sw128_off(t, kk & 63);
                    const float dq = sm.eg[t] * rq_[j];
                    const float dk = sm.egl_g[t] * rk_[j];
                    a.dqp[o] = dq;
                    a.dW[o] = f2bf(-rw_[j]);
                    a.dkp[o] = dk;
                    xq = bf2f(*reinterpret_cast<const bf16 *>(sm.q + so)) * dq;
                    xk = bf2f(*reinterpret_cast<const bf16 *>(sm.k + so)) * dk;
                }
                xq = warp_sum(xq);
                xk = warp_sum(xk);
                if (lane == 0) {
                    sm.red[warp][0][t] = xq;
                    sm.red[warp][1][t] = xk;
                }
            }
        }
    }
    hdh = warp_sum(hdh);
    if (lane == 0) sm.part[warp] = hdh;
    __syncthreads();
    if (done && tid < 64) {
        const int t = tid;
        float dg = 0.f, xi = 0.f;
        if (t < L) {
            const size_t r = (size_t)(t0 + t) * a.H + h;
            const float sq = sm.red[0][0][t] + sm.red[1][0][t] + sm.red[2][0][t] + sm.red[3][0][t];
            const float sk = sm.red[0][1][t] + sm.red[1][1][t] + sm.red[2][1][t] + sm.red[3][1][t];
            xi = sk / a.rk[r];
            dg = a.scale * sq / a.rq[r] - xi;
        }
        sm.red[0][1][t] = xi;  // reuse: xi_t for the sum below
        if (t < L) a.dGp[(size_t)(t0 + t) * a.HV + hv] = dg;
    }
    __syncthreads();
    if (done && tid == 0) {
        float sx = 0.f;
        for (int t = 0; t < L; ++t) sx += sm.red[0][1][t];
        const float hd = sm.part[0] + sm.part[1] + sm.part[2] + sm.part[3];
        a.dGp[(size_t)(t0 + L - 1) * a.HV + hv] += sx + expf(Gl) * hd;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(sm.tmem_base, 256);
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
    cudaError_t e = cudaFuncSetAttribute(k_bintra_a_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BINTRA_A, s);
    k_bintra_a_tc<<<dim3(a.num_chunks, a.HV), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
