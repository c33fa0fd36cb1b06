// gdn_intra_tc.cu -- WY pass of a chunk on the tensor cores ("WY pass" of
// "cake_gdn: deterministic chunked GDN training kernels", section 2; the
// chunk form of the GDN context-parallel scans in "Qwen3.5-397B RL trainer on
// 128 v7x", maxtext #5799).
//
// Persistent CTAs of 128 threads walking runs of (chunk, value head) units, sized
// so that four share an SM (about 55 KB of shared memory, the w / u operands
// taking the bytes of the fp32 inverse once it is in registers, and 128 TMEM
// columns each): the pass is a chain of short dependent steps, and co-resident CTAs hide
// one another's latencies, while each CTA loads its next unit under its epilogue.  With Khat = diag(1 / r_k) K and Gamma_ij = exp(G_i - G_j):
//   KK = K K^T                                   (tcgen05, M=64 N=64 K=128)
// The M=64 KK result is read as 16x256b fragments (two rows, eight columns per lane).
//   A  = strict_tril(diag(beta) KKhat (.) Gamma) (CUDA cores, fp32)
//   T  = (I + A)^-1                              (in place over A: 16x16 diagonal
//        blocks by substitution and T21 = -T22 (A21 T11) at block size 16 in
//        fp32 on the CUDA cores; the block-32 step on the tensor cores, every
//        operand split into bf16 hi + lo parts, fp32 accumulation)
//   w^T = K^T (T diag(beta e^G / r_k))^T,  u^T = V^T (T diag(beta))^T
//                                                (tcgen05, M=128 N=64 K=64; the K
//                                                 and V tiles are read MN-major, so
//                                                 row d of w^T / u^T is TMEM lane d)
// Each unit also writes the record of per-token scalars that the two state scans
// apply (ScRec: e^{G_L - G_t} / r_k,t, e^{G_t} scale / r_q,t, e^{G_L}).
// w^T, u^T and T (kept for the backward) go to HBM in bf16, w^T and u^T per chunk
// as [C][HV][128][64]: thread d holds row d of both (the chunk's 64 tokens) and
// stages it in the bytes of T (swizzled as the tile map expects); one TMA store per
// tile copies the 128 rows out.  Columns past L come out zero
// (beta is zero there, so those rows of T diag(c) are), and the scans that read
// the tiles rely on that.
#include <stddef.h>
#include <string.h>

#include "gdn_epi.cuh"
#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 128;
constexpr uint32_t kHalf = 64 * 128;   // 64 rows x 128 bytes (one SW128 column half)
constexpr uint32_t kTile = 2 * kHalf;  // 64 rows x 128 bf16
constexpr int kS = 68;                 // fp32 row stride of the A / T array (16-byte rows)
constexpr int kXs = 36;                // fp32 row stride of the X scratch

struct IntraSmem {
    unsigned char k[kTile];     // K rows [t][d] (TMA, SW128, two 64-column halves)
    unsigned char v[kTile];     // V rows [t][d]
    float M[64 * kS];           // A (strictly lower, zeros elsewhere), then T in place; once
                                // every thread holds its slice of T, the same bytes hold the
                                // w / u operands (op_w, op_u below)
    float X[32 * kXs];          // A21 T11 of the current merge level
    float G[64], beta[64], wc[64], rki[64];
    uint64_t ld_bar, v_bar, mma_bar;   // K (ld_bar), V (v_bar), products
    uint32_t tmem_base;
};

struct IntraMaps {
    CUtensorMap k, v;
    CUtensorMap w, u;   // outputs: [C][HV][128] rows of 64 tokens, 128-row boxes
};

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// The two 32x32 diagonal blocks of T = (I + A)^-1, in place over M (64 x 64 fp32, row
// stride kS).  On entry M holds A strictly below the diagonal and zeros on and above
// it; on exit its diagonal blocks hold T11 and T22 (zeros above the diagonal, so the
// products below may run over full block ranges) and rows 32.. columns 0..31 still
// hold A21.  All 128 threads call it; X is scratch.
__device__ __forceinline__ void tri_inverse(float *M, float *X, int tid) {
    // 16x16 diagonal blocks: thread (b, c) forward-substitutes column c of block b.
    // t[m] stays 0 for m < c, so the fixed-range sums need no masks; a row of the
    // block comes in as four 16-byte loads.
    float t[16];
    if (tid < 64) {
        const int base = (tid >> 4) * 16, c = tid & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float arow[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(&M[(base + r) * kS + base + 4 * q]);
                arow[4 * q] = v.x; arow[4 * q + 1] = v.y; arow[4 * q + 2] = v.z; arow[4 * q + 3] = v.w;
            }
            float x = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) x -= arow[m] * t[m];
            t[r] = x;
        }
    }
    __syncthreads();  // every read of the diagonal blocks' A is done
    if (tid < 64) {
        const int base = (tid >> 4) * 16, c = tid & 15;
#pragma unroll
        for (int r = 0; r < 16; ++r) M[(base + r) * kS + base + c] = t[r];
    }
    __syncthreads();
    // block size 16: pairs p = 0, 1 (rows 32p+16.., columns 32p..); 2x2 outputs a
    // thread; the A rows come four elements at a time, the right factor in pairs
    {
        const int p = tid >> 6, tt = tid & 63;
        const int r0 = 32 * p + 16, c0 = 32 * p;
        const int rr = 2 * (tt >> 3), cc = 2 * (tt & 7);
        float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&M[(r0 + rr) * kS + c0 + 4 * m4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&M[(r0 + rr + 1) * kS + c0 + 4 * m4]);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 b = *reinterpret_cast<const float2 *>(&M[(c0 + 4 * m4 + e) * kS + c0 + cc]);
                x00 += av0[e] * b.x;
                x01 += av0[e] * b.y;
                x10 += av1[e] * b.x;
                x11 += av1[e] * b.y;
            }
        }
        *reinterpret_cast<float2 *>(&X[(16 * p + rr) * kXs + cc]) = make_float2(x00, x01);
        *reinterpret_cast<float2 *>(&X[(16 * p + rr + 1) * kXs + cc]) = make_float2(x10, x11);
        __syncthreads();
        float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&M[(r0 + rr) * kS + r0 + 4 * m4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&M[(r0 + rr + 1) * kS + r0 + 4 * m4]);
            const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 b = *reinterpret_cast<const float2 *>(&X[(16 * p + 4 * m4 + e) * kXs + cc]);
                y00 += av0[e] * b.x;
                y01 += av0[e] * b.y;
                y10 += av1[e] * b.x;
                y11 += av1[e] * b.y;
            }
        }
        *reinterpret_cast<float2 *>(&M[(r0 + rr) * kS + c0 + cc]) = make_float2(-y00, -y01);
        *reinterpret_cast<float2 *>(&M[(r0 + rr + 1) * kS + c0 + cc]) = make_float2(-y10, -y11);
        __syncthreads();
    }
}

struct IntraUnit {
    int c, hv, h, t0, L;
};

__device__ __forceinline__ IntraUnit intra_unit(const ChunkArgs &a, int u) {
    IntraUnit x;
    x.c = u / a.HV;
    x.hv = u - x.c * a.HV;
    x.h = x.hv / (a.HV / a.H);
    const bool in = in_range(x.c, 1, a.num_chunks, a.status);
    x.t0 = in ? a.chunk_start[x.c] : 0;
    x.L = in ? a.chunk_len[x.c] : 0;
    return x;
}

// Unit u + 1 after unit x = u; the chunk table is read only when the chunk changes.
__device__ __forceinline__ IntraUnit intra_next(const ChunkArgs &a, const IntraUnit &x) {
    if (x.hv + 1 < a.HV) {
        IntraUnit y = x;
        y.hv = x.hv + 1;
        y.h = y.hv / (a.HV / a.H);
        return y;
    }
    return intra_unit(a, (x.c + 1) * a.HV);
}

__device__ __forceinline__ void issue_k(const IntraMaps &m, IntraSmem &sm, const IntraUnit &x) {
    mbar_arrive_expect_tx(&sm.ld_bar, kTile);
    tma_load_3d(sm.k, &m.k, 0, x.h, x.t0, &sm.ld_bar);
    tma_load_3d(sm.k + kHalf, &m.k, 64, x.h, x.t0, &sm.ld_bar);
}
// V is loaded once the block-32 step of the inverse (whose operands use its bytes) is
// done; the L2 prefetch at the unit's start makes that load a short one.
__device__ __forceinline__ void issue_v(const IntraMaps &m, IntraSmem &sm, const IntraUnit &x) {
    mbar_arrive_expect_tx(&sm.v_bar, kTile);
    tma_load_3d(sm.v, &m.v, 0, x.hv, x.t0, &sm.v_bar);
    tma_load_3d(sm.v + kHalf, &m.v, 64, x.hv, x.t0, &sm.v_bar);
}

// Eight fp32 values as bf16 hi (rounded) and lo (the rounded remainder) parts, 16
// bytes each, at (row, col) of two SW128 tiles (col a multiple of 8).
__device__ __forceinline__ void split8(const float *src, unsigned char *hi, uint32_t hrow,
                                       unsigned char *lo, uint32_t lrow, int col) {
    const float4 a = *reinterpret_cast<const float4 *>(src), b = *reinterpret_cast<const float4 *>(src + 4);
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * z], x[2 * z + 1]);
        const float2 hf = __bfloat1622float2(h2);
        ph[z] = *reinterpret_cast<const uint32_t *>(&h2);
        pl[z] = pack_bf2(x[2 * z] - hf.x, x[2 * z + 1] - hf.y);
    }
    *reinterpret_cast<uint4 *>(hi + sw128_off(hrow, col)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4 *>(lo + sw128_off(lrow, col)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
}

// Persistent: CTA b walks the units [b per, (b + 1) per) (unit u = chunk u / HV, value
// head u % HV), four CTAs per SM; the next unit's K and V tiles load as soon as the
// w / u products have read this unit's, and its per-token scalars a unit ahead.
__global__ void __launch_bounds__(kThr, 4) k_intra_tc(const ChunkArgs a,
                                                      const __grid_constant__ IntraMaps maps, int per) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    IntraSmem &sm = smem_struct<IntraSmem>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nunits = a.num_chunks * a.HV;
    const int ub = blockIdx.x * per, ue = min(nunits, ub + per);
    if (ub >= ue) return;
    if (tid == 0) tma_prefetch_maps(maps);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    IntraUnit x = intra_unit(a, ub);
    if (tid == 0) {
        mbar_init(&sm.ld_bar, 1);
        mbar_init(&sm.v_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
        issue_k(maps, sm, x);
    }
    // per-token scalars of thread tid < 64, fetched one unit ahead
    float pG = 0.f, pR = 1.f, pQ = 1.f;
    uint32_t pB = 0;   // raw beta bits, converted when published
    bool pin = false;
    auto fetch = [&](const IntraUnit &y) {
        pin = tid < 64 && tid < y.L;
        if (pin) {
            const size_t gi = (size_t)(y.t0 + tid) * a.HV + y.hv;
            const size_t ri = (size_t)(y.t0 + tid) * a.H + y.h;
            if (kChecked && !(in_range(gi, 1, n_tok_hv(a), a.status) && in_range(ri, 1, n_tok_h(a), a.status)))
                pin = false;
            else {
                pG = a.G[gi];
                pB = load_beta_raw(a, gi);
                pR = a.rk[ri];
                pQ = a.rq[ri];
            }
        }
    };
    fetch(x);
    tc_fence_before();
    __syncthreads();  // the barriers are initialised before anyone waits on them
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)(warp * 32) << 16);
    int issued = 1, waited = 0, v_issued = 0, v_waited = 0;
    uint32_t mphase = 0;
    bool ok = true;
    for (int u = ub; u < ue; ++u) {
        const bool has_next = u + 1 < ue;
        const int c = x.c, hv = x.hv, t0 = x.t0, L = x.L;
        if (tid < 64) {  // tokens past L get G = 0, beta = 0 and 1 / r_k = 1
            const float ri = pin ? 1.f / pR : 1.f, bb = pin ? beta_from_raw(a, pB) : 0.f;
            const float gg = pin ? pG : 0.f;
            sm.G[tid] = gg;
            sm.beta[tid] = bb;
            sm.rki[tid] = ri;
            sm.wc[tid] = bb * __expf(gg) * ri;
        }
        ok = __syncthreads_and(ok && mbar_wait(&sm.ld_bar, waited & 1));
        ++waited;
        if (!ok) break;
        tc_fence_after();
        // KK = K K^T into columns 0..63 (M=64: row m at lane 32 (m / 16) + m % 16), issued
        // by lane 0 of warp 3 while warps 0 and 1 write the scalar record and fetch the
        // next unit's scalars (an issuing thread stalls while the tensor pipe's queue is full)
        if (tid == 96 && ok) {
            const uint32_t ks = smem_u32(sm.k);
            const uint32_t id = idesc_bf16(64, 64, 0, 0);
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
                mma_bf16(tb, sdesc(ks + off, 16, 1024), sdesc(ks + off, 16, 1024), id, s > 0);
            }
            mma_commit(&sm.mma_bar);
            tma_prefetch_3d(&maps.v, 0, hv, t0);   // V, loaded after the inverse
            tma_prefetch_3d(&maps.v, 64, hv, t0);
        }
        if (tid < 64) {  // the unit's scalar record for the state scans (before the fetch below)
            const float Gl = L > 0 ? sm.G[L - 1] : 0.f;
            if (in_range(((size_t)c * a.HV + hv) * kScRec, kScRec, (long long)a.num_chunks * a.HV * kScRec,
                         a.status)) {
                ScRec *rec = reinterpret_cast<ScRec *>(a.sc) + (size_t)c * a.HV + hv;
                rec->kc[tid] = pin ? __expf(fminf(Gl - pG, 0.f)) / pR : 0.f;
                rec->qc[tid] = pin ? __expf(pG) * a.scale / pQ : 0.f;
                if (tid == 0) rec->egl = __expf(Gl);
            }
        }
        // the next unit (its table entries are a dependent load: after the MMA issue)
        const IntraUnit nx = has_next ? intra_next(a, x) : x;
        if (has_next) fetch(nx);
        if (tid == 0) tma_store_wait_read();  // the last unit's u^T rows have left M
        ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, mphase));
        mphase ^= 1;
        tc_fence_after();
        if (ok) {  // A from 16x256b fragments of KK: rows ra, ra + 8 of the warp's block, columns
                   // 32 c + 8k + cq + {0, 1}; zeros on and above the diagonal
            const int ra = 16 * warp + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
            const float Ga = sm.G[ra], Gb = sm.G[rb];
            const float aa = sm.beta[ra] * sm.rki[ra], ab = sm.beta[rb] * sm.rki[rb];
    #pragma unroll
            for (int c = 0; c < 2; ++c) {
                float kk[16];
                epi::tmem_ld16x256_x4(t_row + 32 * c, kk);
                tmem_ld_wait();
    #pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int j = 32 * c + 8 * k + cq;
                    const float r0 = sm.rki[j], r1 = sm.rki[j + 1];
                    const float g0 = sm.G[j], g1 = sm.G[j + 1];
                    const float e0 = (j < ra ? aa : 0.f) * kk[4 * k] * r0 * __expf(fminf(Ga - g0, 0.f));
                    const float e1 = (j + 1 < ra ? aa : 0.f) * kk[4 * k + 1] * r1 * __expf(fminf(Ga - g1, 0.f));
                    const float f0 = (j < rb ? ab : 0.f) * kk[4 * k + 2] * r0 * __expf(fminf(Gb - g0, 0.f));
                    const float f1 = (j + 1 < rb ? ab : 0.f) * kk[4 * k + 3] * r1 * __expf(fminf(Gb - g1, 0.f));
                    *reinterpret_cast<float2 *>(sm.M + ra * kS + j) = make_float2(e0, e1);
                    *reinterpret_cast<float2 *>(sm.M + rb * kS + j) = make_float2(f0, f1);
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // KK has been read: its TMEM columns are free
        tri_inverse(sm.M, sm.X, tid);
        // Block-32 step: T21 = -T22 (A21 T11), two M=64 N=64 K=32 products on bf16 hi / lo
        // parts with fp32 accumulation.  The A operand holds the hi part of data row r at
        // row 16 (r / 8) + r % 8 and its lo part 8 rows below, so that the 16x256b
        // fragment of a lane holds both (rows ra, ra + 8) and their sum is the product
        // row.  Operand space: the V tile (loaded afterwards); TMEM columns 0 / 64.
        {
            unsigned char *opA = sm.v, *opBh = sm.v + 2 * 4096, *opBl = sm.v + 3 * 4096;
            const int r = tid >> 2, k8 = 8 * (tid & 3);          // data row, first of 8 columns
            const uint32_t mh = 16 * (r >> 3) + (r & 7);         // its hi row in opA
            split8(sm.M + (32 + r) * kS + k8, opA, mh, opA, mh + 8, k8);   // A21 (K-major)
            split8(sm.M + r * kS + k8, opBh, r, opBl, r, k8);              // T11 [k][j] (MN-major)
            const uint32_t id = idesc_bf16(64, 64, 0, 1);
            const int xr = 8 * warp + (lane >> 2), cq = 2 * (lane & 3);    // fragment data row / column
            auto merge_product = [&](uint32_t col) {
                fence_proxy_async_smem();
                tc_fence_before();
                __syncthreads();
                if (tid == 0 && ok) {
                    tc_fence_after();
                    const uint32_t as = smem_u32(opA), bh = smem_u32(opBh), bl = smem_u32(opBl);
#pragma unroll
                    for (int s = 0; s < 2; ++s)
                        mma_bf16(tb + col, sdesc(as + s * 32, 16, 1024), sdesc(bh + s * 2048, 4096, 1024), id, s > 0);
#pragma unroll
                    for (int s = 0; s < 2; ++s)
                        mma_bf16(tb + col, sdesc(as + s * 32, 16, 1024), sdesc(bl + s * 2048, 4096, 1024), id, true);
                    mma_commit(&sm.mma_bar);
                }
                ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, mphase));
                mphase ^= 1;
                tc_fence_after();
            };
            merge_product(0);   // A21 T11
            {  // X = A21 T11 (hi + lo rows) as the hi / lo B operands; T22 split into opA
                float d[16];
                epi::tmem_ld16x256_x4(t_row, d);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float x0 = d[4 * k] + d[4 * k + 2], x1 = d[4 * k + 1] + d[4 * k + 3];
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                    const float2 hf = __bfloat1622float2(h2);
                    *reinterpret_cast<__nv_bfloat162 *>(opBh + sw128_off(xr, 8 * k + cq)) = h2;
                    *reinterpret_cast<uint32_t *>(opBl + sw128_off(xr, 8 * k + cq)) = pack_bf2(x0 - hf.x, x1 - hf.y);
                }
                split8(sm.M + (32 + r) * kS + 32 + k8, opA, mh, opA, mh + 8, k8);   // T22
            }
            merge_product(64);  // T22 (A21 T11)
            {
                float d[16];
                epi::tmem_ld16x256_x4(t_row + 64, d);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<float2 *>(sm.M + (32 + xr) * kS + 8 * k + cq) =
                        make_float2(-(d[4 * k] + d[4 * k + 2]), -(d[4 * k + 1] + d[4 * k + 3]));
            }
            tc_fence_before();
            __syncthreads();   // T is complete in M; the V tile's bytes are free
            if (tid == 0 && ok) issue_v(maps, sm, x);
            if (ok) ++v_issued;
        }
        {  // operands T diag(c) as bf16 rows, and T to HBM: thread -> row tid / 2, 32 columns
            const int i = tid >> 1, j0 = 32 * (tid & 1);
            const float *Mi = sm.M + i * kS + j0;
            const size_t toff = (((size_t)c * a.HV + hv) * 64 + i) * 64 + j0;
            const bool t_in = in_range(toff, 32, (long long)a.num_chunks * a.HV * 64 * 64, a.status);
            uint4 *Tdst = reinterpret_cast<uint4 *>(a.Tm + toff);
            float tv[32];
    #pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = *reinterpret_cast<const float4 *>(Mi + 4 * q);
                tv[4 * q] = x.x; tv[4 * q + 1] = x.y; tv[4 * q + 2] = x.z; tv[4 * q + 3] = x.w;
            }
            __syncthreads();  // T is in registers: its bytes become the operands
            unsigned char *op_w = reinterpret_cast<unsigned char *>(sm.M), *op_u = op_w + kHalf;
    #pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float *t8 = tv + 8 * q;
                if (t_in) Tdst[q] = make_uint4(pack_bf2(t8[0], t8[1]), pack_bf2(t8[2], t8[3]), pack_bf2(t8[4], t8[5]),
                                               pack_bf2(t8[6], t8[7]));
                const int jb = j0 + 8 * q;
                float wc[8], bt[8];  // the column scales of the eight columns, 16 bytes at a time
                *reinterpret_cast<float4 *>(wc) = *reinterpret_cast<const float4 *>(&sm.wc[jb]);
                *reinterpret_cast<float4 *>(wc + 4) = *reinterpret_cast<const float4 *>(&sm.wc[jb + 4]);
                *reinterpret_cast<float4 *>(bt) = *reinterpret_cast<const float4 *>(&sm.beta[jb]);
                *reinterpret_cast<float4 *>(bt + 4) = *reinterpret_cast<const float4 *>(&sm.beta[jb + 4]);
                uint32_t pw[4], pu[4];
    #pragma unroll
                for (int z = 0; z < 4; ++z) {
                    pw[z] = pack_bf2(t8[2 * z] * wc[2 * z], t8[2 * z + 1] * wc[2 * z + 1]);
                    pu[z] = pack_bf2(t8[2 * z] * bt[2 * z], t8[2 * z + 1] * bt[2 * z + 1]);
                }
                *reinterpret_cast<uint4 *>(op_w + sw128_off(i, jb)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                *reinterpret_cast<uint4 *>(op_u + sw128_off(i, jb)) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok && mbar_wait(&sm.v_bar, v_waited & 1));
        ++v_waited;
        if (tid == 0 && ok) {  // w^T -> columns 0..63, u^T -> 64..127 (lane d, column i)
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64, 1, 0);
            const uint32_t ks = smem_u32(sm.k), vs = smem_u32(sm.v);
            const uint32_t ws = smem_u32(sm.M), us = ws + kHalf;  // op_w, op_u
            for (int s = 0; s < 4; ++s) {
                mma_bf16(tb, sdesc(ks + s * 2048, kHalf, 1024), sdesc(ws + s * 32, 16, 1024), id, s > 0);
                mma_bf16(tb + 64, sdesc(vs + s * 2048, kHalf, 1024), sdesc(us + s * 32, 16, 1024), id, s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        ok = __syncthreads_and(ok && mbar_wait(&sm.mma_bar, mphase));
        mphase ^= 1;
        tc_fence_after();
        if (tid == 0 && ok && has_next) issue_k(maps, sm, nx);  // K has been read
        if (ok && has_next) ++issued;
        if (ok) {  // w^T, then u^T: thread d stages row d (64 tokens) in M, one TMA store each
            unsigned char *stg = reinterpret_cast<unsigned char *>(sm.M);
            const int row = (c * a.HV + hv) * kDim;
            for (int part = 0; part < 2; ++part) {
                float x[2][32];
                tmem_ld32(t_row + 64 * part, x[0]);
                tmem_ld32(t_row + 64 * part + 32, x[1]);
                tmem_ld_wait();
                if (part == 1) {  // the w^T store has read the staged rows
                    if (tid == 0) tma_store_wait_read();
                    __syncthreads();
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float *y = x[q >> 2] + 8 * (q & 3);
                    *reinterpret_cast<uint4 *>(stg + sw128_off(tid, 8 * q)) =
                        make_uint4(pack_bf2(y[0], y[1]), pack_bf2(y[2], y[3]), pack_bf2(y[4], y[5]),
                                   pack_bf2(y[6], y[7]));
                }
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tma_store_3d(part == 0 ? &maps.w : &maps.u, 0, 0, row, stg);
                    tma_store_commit();
                }
            }
        }
        tc_fence_before();
        ok = __syncthreads_and(ok);  // the unit's scalars, operands and TMEM are free
        if (!ok) break;
        x = nx;
    }
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        if (issued > waited) mbar_wait(&sm.ld_bar, (issued - 1) & 1, kDrainLimitNs);  // drain (bounded)
        if (v_issued > v_waited) mbar_wait(&sm.v_bar, (v_issued - 1) & 1, kDrainLimitNs);
    }
    if (tid == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 128);
}

}  // namespace

cudaError_t launch_intra_tc(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    IntraMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    const uint64_t wrows = (uint64_t)a.num_chunks * a.HV * kDim;
    if (!encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.v, a.v, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.w, a.w, 1, wrows, 128, 128, 128, kChunk) ||
        !encode_rows_bf16(&m.u, a.u, 1, wrows, 128, 128, 128, kChunk))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(IntraSmem) + 1024;
    static_assert(4 * (sizeof(IntraSmem) + 2048) <= 233472, "four CTAs per SM");
    static_assert(offsetof(IntraSmem, M) % 1024 == 0 && sizeof(IntraSmem::M) >= 2 * kHalf,
                  "the w / u operands fit, 1024-aligned, in the bytes of T");
    cudaError_t e = cudaFuncSetAttribute(k_intra_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    const int nunits = a.num_chunks * a.HV;
    const int per = (nunits + 4 * sms - 1) / (4 * sms);
    TimerScope ts(a.timer, GDN_KERNEL_INTRA, s);
    k_intra_tc<<<(nunits + per - 1) / per, kThr, smem, s>>>(a, m, per);
    return cudaGetLastError();
}

}  // namespace gdn
