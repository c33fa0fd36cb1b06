// gdn_bintra_b_tc.cu -- WY pullback of a chunk on the tensor cores ("WY
// pullback" of "cake_gdn: deterministic chunked GDN training kernels",
// section 2).
//
// Persistent CTAs of 256 threads, two per SM (about 100 KB of shared memory and
// 256 TMEM columns each), each walking a run of (chunk, value head) units.  With Khat = diag(1/r_k) K,
// Gamma_ij = exp(G_i - G_j), the WY inverse T (saved in bf16 by the forward) and dW =
// -dv_new h^T (from the h / dh' kernel):
//   phase 1 (M=64 N=64 K=128, rows = tokens):  KK = K K^T, D1 = dW K^T, D2 = dv_new V^T
//     dT_ij = beta_j (e^{G_j} D1_ij / r_k,j + D2_ij)          (j < i)
//   phase 1b/1c (K = 64): X = dT T^T,  dA = -T^T X          (strictly lower)
//     B = dA (.) beta_i Gamma,   P2 = dA (.) KKhat Gamma
//   phase 2 (M=128 N=64 K=64, rows = features d, columns = tokens m):
//     (B Khat + B^T Khat)^T,  dWt^T = (T^T dW)^T,  dUt^T = (T^T dv_new)^T
//     dkhat_m += (B Khat + B^T Khat)_m + beta_m e^{G_m} dWt_m,  dv_m = beta_m dUt_m
// The M=64 results are read as 16x256b fragments (two rows and eight columns per
// lane, all 32 lanes busy).  The row dots khat_m . dWt_m = sum_i T_im D1_im / r_k,m
// and v_m . dUt_m = sum_i T_im D2_im that dbeta and dG need are column sums of
// T (.) D1 and T (.) D2 read off phase 1, taken with warp butterflies, as are the
// column sums of beta_i P2:
//   dbeta_m = sum_j P2_mj + e^{G_m}/r_k,m sum_i T_im D1_im + sum_i T_im D2_im
//   dG_m   += beta_m sum_j P2_mj - sum_i beta_i P2_im + beta_m e^{G_m}/r_k,m sum_i T_im D1_im
// and dg is the reverse cumulative sum of dG (which arrives holding the h / dh'
// and Q K^T terms).  A CTA walks whole groups of the r = HV / H value heads of one
// key head and sums their dkhat terms in fp32 in spare TMEM columns (value heads in
// order).  After the group's last value head it finishes dk for the key head: the
// sums (staged as bf16 rows in shared memory) plus the h / dh' and Q K^T terms that
// k_bintra_a_tc left (bf16 [T, H, 128]) give dkhat_t, and the L2-norm backward
//   dk_t = (dkhat_t - k_t (k_t . dkhat_t) / r_k,t^2) / r_k,t
// runs token-major, half a warp per token.
#include <stddef.h>
#include <string.h>

#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_epi.cuh"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;
using epi::pack_bf2;
using epi::colsum_frag;
using epi::colsum_frag_col;
using epi::get_pair;
using epi::put_pair;
using epi::quad_sum;
using epi::tmem_ld16x256_x4;

constexpr int kThr = 256;   // two warpgroups share the 128 TMEM lanes
// The products are issued by lane 0 of warp 7: an issuing thread stalls while the
// tensor pipe's queue is full, and warps 0 and 1 have per-token work (the next
// unit's scalars, dbeta and dG) that runs beside the products.
constexpr int kIssuer = 224;
constexpr uint32_t kHalf = 64 * 128;      // 64 rows x 128 B
constexpr uint32_t kTile = 2 * kHalf;     // 64 rows x 128 bf16: two 8 KB halves

// TMEM columns (256 allocated).  X reuses D2's columns and T^T X D1's (both read
// before), so that columns 192 .. 255 hold, for the whole kernel, the key head's
// dkhat sums (lane d = feature, column 192 + token).
constexpr uint32_t cKK = 0, cD1 = 64, cD2 = 128, cX = 128, cA = 64;   // phase 1
constexpr uint32_t cDK = 0, cWT = 64, cUT = 128;                       // phase 2
constexpr uint32_t cACC = 192;                                         // dkhat sums

struct BwSmem {
    unsigned char k[kTile], v[kTile], dw[kTile], dvn[kTile];
    unsigned char op_t[kHalf];     // T_ij [i][j]: K-major B of X, MN-major A of T^T X, MN-major B of phase 2
    unsigned char op_dx[kHalf];    // dT rows (K-major A of X = dT T^T), then X rows (MN-major B of T^T X)
    unsigned char op_b[kHalf];     // B_tj / r_k,j  [t][j]  K-major B
    unsigned char op_bt[kHalf];    // B_it / r_k,i  [i][t]  MN-major B
    float G[64], beta[64], rki[64], eg[64], dG[64], db[64];
    float rs[2][64];               // per-warpgroup partial row sums of P2
    float cy[4][64], cz[4][64], cp[4][64];  // per-row-block column sums
    // (op_b and op_bt, adjacent, also hold a last value head's summed dkhat rows: bf16
    // [t][128], 256-byte rows, once phase 2 has read them)
    uint64_t a_bar, v_bar, mma_bar;
    uint32_t tmem_base;
};

static_assert(offsetof(BwSmem, op_bt) == offsetof(BwSmem, op_b) + kHalf, "op_b, op_bt: one 16 KB tile");

struct BwMaps {
    CUtensorMap k, v, dw, dvn, t;
    CUtensorMap dkp;   // the h / dh' dkhat terms [T][H][128]: L2 prefetch for the dk pass
};

struct BwUnit {
    int c, hv, h, t0, L;
};

__device__ __forceinline__ BwUnit bw_unit(const ChunkArgs &a, int u) {
    BwUnit x;
    x.c = u / a.HV;
    x.hv = u - x.c * a.HV;
    x.h = x.hv / (a.HV / a.H);
    const bool in = in_range(x.c, 1, a.num_chunks, a.status);
    x.t0 = in ? a.chunk_start[x.c] : 0;
    x.L = in ? a.chunk_len[x.c] : 0;
    return x;
}
// Unit u + 1 after unit x = u: the chunk table is read only when the chunk changes
// (once every HV units), so the lookup rarely waits on a load.
__device__ __forceinline__ BwUnit bw_next(const ChunkArgs &a, const BwUnit &x) {
    if (x.hv + 1 < a.HV) {
        BwUnit y = x;
        y.hv = x.hv + 1;
        y.h = y.hv / (a.HV / a.H);
        return y;
    }
    return bw_unit(a, (x.c + 1) * a.HV);
}

// group A: K, dW, dv_new and T (free once phase 2 has run); group V: V (free after phase 1)
__device__ __forceinline__ void issue_a(const BwMaps &m, BwSmem &sm, const ChunkArgs &a, const BwUnit &x) {
    mbar_arrive_expect_tx(&sm.a_bar, 3 * kTile + kHalf);
    tma_load_3d(sm.op_t, &m.t, 0, 0, (x.c * a.HV + x.hv) * 64, &sm.a_bar);  // T rows (bf16)
    tma_load_3d(sm.k, &m.k, 0, x.h, x.t0, &sm.a_bar);
    tma_load_3d(sm.k + kHalf, &m.k, 64, x.h, x.t0, &sm.a_bar);
    tma_load_3d(sm.dw, &m.dw, 0, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dw + kHalf, &m.dw, 64, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dvn, &m.dvn, 0, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dvn + kHalf, &m.dvn, 64, x.hv, x.t0, &sm.a_bar);
}

__device__ __forceinline__ void issue_v(const BwMaps &m, BwSmem &sm, const BwUnit &x) {
    mbar_arrive_expect_tx(&sm.v_bar, kTile);
    tma_load_3d(sm.v, &m.v, 0, x.hv, x.t0, &sm.v_bar);
    tma_load_3d(sm.v + kHalf, &m.v, 64, x.hv, x.t0, &sm.v_bar);
}

// Persistent: CTA b walks the units [b per, (b + 1) per) (unit u = chunk u / HV, value
// head u % HV), two CTAs per SM.  The next unit's V loads as soon as phase 1 has read
// this one's, its K, dW, dv_new and T as soon as phase 2 has, and its per-token scalars
// a unit ahead, so the loads run under the epilogues.
__global__ void __launch_bounds__(kThr, 2) k_bintra_b_tc(const ChunkArgs a,
                                                         const __grid_constant__ BwMaps maps, int per) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BwSmem &sm = smem_struct<BwSmem>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nunits = a.num_chunks * a.HV;
    const int ub = blockIdx.x * per, ue = min(nunits, ub + per);
    if (ub >= ue) return;
    const int grp = warp >> 2;                // warpgroup: which half of the columns
    const int sub = warp & 3;                 // TMEM lane quarter
    if (tid == 0) tma_prefetch_maps(maps);

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.a_bar, 1);
        mbar_init(&sm.v_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    BwUnit x = bw_unit(a, ub);
    if (tid == 0) {
        issue_a(maps, sm, a, x);
        issue_v(maps, sm, x);
    }
    int a_issued = 1, v_issued = 1, waited = 0;  // same on every thread
    // per-token scalars of thread tid < 64, fetched one unit ahead
    float pG = 0.f, pR = 1.f, pD = 0.f;
    uint32_t pB = 0;   // raw beta bits, converted when published
    bool pin = false;
    auto fetch = [&](const BwUnit &y) {
        pin = tid < 64 && tid < y.L &&
              in_range((size_t)(y.t0 + tid) * a.HV + y.hv, 1, n_tok_hv(a), a.status);
        if (pin) {
            const size_t gi = (size_t)(y.t0 + tid) * a.HV + y.hv;
            pG = a.G[gi];
            pB = load_beta_raw(a, gi);
            pR = a.rk[(size_t)(y.t0 + tid) * a.H + y.h];
            pD = a.dGp[gi];
        }
    };
    fetch(x);
    // dk of a key head (after its last value head): half a warp per token, eight features
    // a lane, four tokens a warp.  Every global load of the pass (k and the h / dh' dkhat
    // terms, L2-warm from the prefetch at the unit's start) goes out before any is used;
    // the staged WY sums (op_b / op_bt) are added, the L2-norm backward applied and dk
    // stored.
    const int l16 = lane & 15;
    auto dk_pass = [&](int ut0, int uh, int uL) {
        const size_t base = ((size_t)ut0 * a.H + uh) * kDim + 8 * l16;
        uint4 lks[4], l1s[4];
        uint32_t live = 0;
    #pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * warp + 2 * i + (lane >> 4);
            const size_t row = base + (size_t)m * a.H * kDim;
            lks[i] = make_uint4(0u, 0u, 0u, 0u);
            l1s[i] = lks[i];
            if (m < uL && in_range(row, 8, n_rows_h(a), a.status)) {
                live |= 1u << i;
                lks[i] = __ldg(reinterpret_cast<const uint4 *>(a.k + row));
                l1s[i] = __ldg(reinterpret_cast<const uint4 *>(a.dkpart + row));
            }
        }
        const bf16 *stg = reinterpret_cast<const bf16 *>(sm.op_b);
    #pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * warp + 2 * i + (lane >> 4);
            const uint4 lk = lks[i], l1 = l1s[i];
            const uint4 l2 = *reinterpret_cast<const uint4 *>(stg + m * kDim + 8 * l16);
            const uint32_t wk[4] = {lk.x, lk.y, lk.z, lk.w}, w1[4] = {l1.x, l1.y, l1.z, l1.w},
                           w2[4] = {l2.x, l2.y, l2.z, l2.w};
            float xk[8], dd[8];
    #pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
                const float2 kk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wk[u2]));
                const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w1[u2]));
                const float2 p2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w2[u2]));
                xk[2 * u2] = kk.x; xk[2 * u2 + 1] = kk.y;
                dd[2 * u2] = p1.x + p2.x; dd[2 * u2 + 1] = p1.y + p2.y;
            }
            float dot = 0.f;
    #pragma unroll
            for (int u2 = 0; u2 < 8; ++u2) dot += xk[u2] * dd[u2];
    #pragma unroll
            for (int o = 8; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);  // the token's 16 lanes
            const float ri = sm.rki[m], cdot = dot * ri * ri;
            if ((live >> i) & 1u) {
                uint32_t pk[4];
    #pragma unroll
                for (int u2 = 0; u2 < 4; ++u2)
                    pk[u2] = pack_bf2((dd[2 * u2] - xk[2 * u2] * cdot) * ri, (dd[2 * u2 + 1] - xk[2 * u2 + 1] * cdot) * ri);
                *reinterpret_cast<uint4 *>(a.dk + base + (size_t)m * a.H * kDim) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
    };
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)(sub * 32) << 16);
    uint32_t phase = 0;
    bool ok = true;
    for (int u = ub; u < ue; ++u) {
        const bool has_next = u + 1 < ue;
        const int c = x.c, hv = x.hv, t0 = x.t0, L = x.L;
        if (tid < 64) {  // tokens past L get zeros and 1 / r_k = 1
            sm.G[tid] = pin ? pG : 0.f;
            sm.beta[tid] = pin ? beta_from_raw(a, pB) : 0.f;
            sm.rki[tid] = pin ? 1.f / pR : 1.f;
            sm.eg[tid] = pin ? __expf(pG) : 0.f;
            sm.dG[tid] = pin ? pD : 0.f;
        }
        {
            const bool got = mbar_wait(&sm.a_bar, waited & 1) && mbar_wait(&sm.v_bar, waited & 1);
            ok = __syncthreads_and(ok && got);
            ++waited;
            if (!ok) break;
        }
        auto commit_wait = [&](bool &okr) {
            okr = __syncthreads_and(okr && mbar_wait(&sm.mma_bar, phase));
            phase ^= 1;
            tc_fence_after();
        };
        // ---- phase 1: KK, D1, D2 (64 x 64, contraction 128)
        if (tid == kIssuer && ok) {
            if (hv % (a.HV / a.H) == a.HV / a.H - 1) {  // a last value head: warm L2 for its dk pass
                tma_prefetch_3d(&maps.dkp, 0, x.h, t0);
                tma_prefetch_3d(&maps.dkp, 64, x.h, t0);
            }
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 64, 0, 0);
            const uint32_t A[3] = {smem_u32(sm.k), smem_u32(sm.dw), smem_u32(sm.dvn)};
            const uint32_t B[3] = {smem_u32(sm.k), smem_u32(sm.k), smem_u32(sm.v)};
            const uint32_t col[3] = {cKK, cD1, cD2};
    #pragma unroll
            for (int p = 0; p < 3; ++p)
    #pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * kHalf + (s & 3) * 32;
                    mma_bf16(tb + col[p], sdesc(A[p] + off, 16, 1024), sdesc(B[p] + off, 16, 1024), id, s > 0);
                }
            mma_commit(&sm.mma_bar);
        }
        // the next unit (its table entries are a dependent load: after the MMA issue)
        const BwUnit nx = has_next ? bw_next(a, x) : x;
        if (has_next) fetch(nx);
        commit_wait(ok);
        if (tid == 0 && ok && has_next) issue_v(maps, sm, nx);  // V has been read by phase 1
        if (ok && has_next) ++v_issued;
        // M=64 epilogues read 16x256b fragments: lane t of warp (grp, sub) holds rows
        // ra = 16 sub + t/4 and rb = ra + 8, columns j0 + 8k + 2 (t % 4) + {0, 1}.
        const int j0 = 32 * grp;                  // this warpgroup's columns
        const int ra = sub * 16 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
        const bool la = ra < L, lb = rb < L;
        const int ccol = j0 + colsum_frag_col(lane);  // the column whose sums this lane keeps
        if (ok) {  // dT rows (bf16 operand) and the column sums of T (.) D1, T (.) s
            float d1[16], d2[16];
            tmem_ld16x256_x4(t_row + cD1 + j0, d1);
            tmem_ld16x256_x4(t_row + cD2 + j0, d2);
            tmem_ld_wait();
            float z[8], y[8];
    #pragma unroll
            for (int k = 0; k < 4; ++k) {
    #pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int j = j0 + 8 * k + cq + p;
                    const float f1 = sm.eg[j] * sm.rki[j], bj = sm.beta[j];
                    const float sa = f1 * d1[4 * k + p] + d2[4 * k + p];
                    const float sb = f1 * d1[4 * k + 2 + p] + d2[4 * k + 2 + p];
                    const float2 ta = get_pair(sm.op_t, ra, j0 + 8 * k + cq);   // T is zero above the diagonal
                    const float2 tb2 = get_pair(sm.op_t, rb, j0 + 8 * k + cq);
                    const float tva = la ? (p ? ta.y : ta.x) : 0.f, tvb = lb ? (p ? tb2.y : tb2.x) : 0.f;
                    z[2 * k + p] = tva * d1[4 * k + p] + tvb * d1[4 * k + 2 + p];
                    y[2 * k + p] = tva * sa + tvb * sb;
                    d2[4 * k + p] = (la && j < ra) ? bj * sa : 0.f;        // dT, in place
                    d2[4 * k + 2 + p] = (lb && j < rb) ? bj * sb : 0.f;
                }
                put_pair(sm.op_dx, ra, j0 + 8 * k + cq, d2[4 * k], d2[4 * k + 1]);
                put_pair(sm.op_dx, rb, j0 + 8 * k + cq, d2[4 * k + 2], d2[4 * k + 3]);
            }
            sm.cz[sub][ccol] = colsum_frag(z, lane);
            sm.cy[sub][ccol] = colsum_frag(y, lane);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- phase 1b: X = dT T^T  (A = dT rows, B = T rows as [N][K])
        if (tid == kIssuer && ok) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 64, 0, 0);
    #pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tb + cX, sdesc(smem_u32(sm.op_dx) + s * 32, 16, 1024),
                         sdesc(smem_u32(sm.op_t) + s * 32, 16, 1024), id, s > 0);
            mma_commit(&sm.mma_bar);
        }
        commit_wait(ok);
        if (ok) {  // X rows -> bf16 over the dT rows (the product that read them is done)
            float x[16];
            tmem_ld16x256_x4(t_row + cX + j0, x);
            tmem_ld_wait();
    #pragma unroll
            for (int k = 0; k < 4; ++k) {
                put_pair(sm.op_dx, ra, j0 + 8 * k + cq, x[4 * k], x[4 * k + 1]);
                put_pair(sm.op_dx, rb, j0 + 8 * k + cq, x[4 * k + 2], x[4 * k + 3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- phase 1c: T^T X  (A = T rows read MN-major, B = X rows read MN-major)
        if (tid == kIssuer && ok) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(64, 64, 1, 1);
    #pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tb + cA, sdesc(smem_u32(sm.op_t) + s * 2048, kHalf, 1024),
                         sdesc(smem_u32(sm.op_dx) + s * 2048, kHalf, 1024), id, s > 0);
            mma_commit(&sm.mma_bar);
        }
        commit_wait(ok);
        if (ok) {  // dA = -(T^T X): B and its operands, P2 row sums, column sums of beta_i P2
            float ta[16], kk[16];
            tmem_ld16x256_x4(t_row + cA + j0, ta);
            tmem_ld16x256_x4(t_row + cKK + j0, kk);
            tmem_ld_wait();
            const float Ga = sm.G[ra], Gb = sm.G[rb];
            const float ba = sm.beta[ra], bb = sm.beta[rb];
            const float rka = sm.rki[ra], rkb = sm.rki[rb];
            float rsa = 0.f, rsb = 0.f, pb[8];
    #pragma unroll
            for (int k = 0; k < 4; ++k) {
                float b1[4], b2[4];
    #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = j0 + 8 * k + cq + (e & 1);
                    const bool up = e & 2;                       // row rb
                    const int r = up ? rb : ra;
                    const float msk = ((up ? lb : la) && j < r) ? 1.f : 0.f;
                    const float dag = -ta[4 * k + e] * msk * __expf(fminf((up ? Gb : Ga) - sm.G[j], 0.f));
                    const float rkj = sm.rki[j], br = up ? bb : ba, rkr = up ? rkb : rka;
                    const float p2 = dag * kk[4 * k + e] * rkr * rkj;
                    if (up) rsb += p2; else rsa += p2;
                    b1[e] = dag * br * rkj;   // B_rj / r_k,j
                    b2[e] = dag * br * rkr;   // B_rj / r_k,r
                    kk[4 * k + e] = br * p2;  // beta_r P2_rj
                }
                pb[2 * k] = kk[4 * k] + kk[4 * k + 2];
                pb[2 * k + 1] = kk[4 * k + 1] + kk[4 * k + 3];
                put_pair(sm.op_b, ra, j0 + 8 * k + cq, b1[0], b1[1]);
                put_pair(sm.op_b, rb, j0 + 8 * k + cq, b1[2], b1[3]);
                put_pair(sm.op_bt, ra, j0 + 8 * k + cq, b2[0], b2[1]);
                put_pair(sm.op_bt, rb, j0 + 8 * k + cq, b2[2], b2[3]);
            }
            sm.cp[sub][ccol] = colsum_frag(pb, lane);
            rsa = quad_sum(rsa);
            rsb = quad_sum(rsb);
            if ((lane & 3) == 0) {
                sm.rs[grp][ra] = rsa;
                sm.rs[grp][rb] = rsb;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- phase 2 (M=128: row d of each product is TMEM lane d, column m is a token)
        if (tid == kIssuer && ok) {
            tc_fence_after();
            const uint32_t kA = smem_u32(sm.k), wA = smem_u32(sm.dw), vA = smem_u32(sm.dvn);
            const uint32_t tB = smem_u32(sm.op_t), bB = smem_u32(sm.op_b), btB = smem_u32(sm.op_bt);
            const uint32_t id_mk = idesc_bf16(128, 64, 1, 0);  // A MN-major, B K-major
            const uint32_t id_mm = idesc_bf16(128, 64, 1, 1);  // A MN-major, B MN-major
    #pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t aK = sdesc(kA + s * 2048, kHalf, 1024);
                mma_bf16(tb + cDK, aK, sdesc(bB + s * 32, 16, 1024), id_mk, s > 0);
                mma_bf16(tb + cDK, aK, sdesc(btB + s * 2048, kHalf, 1024), id_mm, true);
                mma_bf16(tb + cWT, sdesc(wA + s * 2048, kHalf, 1024), sdesc(tB + s * 2048, kHalf, 1024), id_mm,
                         s > 0);
                mma_bf16(tb + cUT, sdesc(vA + s * 2048, kHalf, 1024), sdesc(tB + s * 2048, kHalf, 1024), id_mm,
                         s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        // meanwhile: dbeta and this kernel's dG terms per token m (fixed order)
        if (ok && tid < 64) {
            const int m = tid;
            const float r2 = sm.rs[0][m] + sm.rs[1][m];
            const float cy = ((sm.cy[0][m] + sm.cy[1][m]) + sm.cy[2][m]) + sm.cy[3][m];
            const float cz = ((sm.cz[0][m] + sm.cz[1][m]) + sm.cz[2][m]) + sm.cz[3][m];
            const float cp = ((sm.cp[0][m] + sm.cp[1][m]) + sm.cp[2][m]) + sm.cp[3][m];
            const float bm = sm.beta[m];
            sm.db[m] = r2 + cy;
            sm.dG[m] += bm * r2 - cp + bm * sm.eg[m] * sm.rki[m] * cz;
        }
        commit_wait(ok);
        if (tid == 0 && ok && has_next) issue_a(maps, sm, a, nx);  // K, dW, dv_new, T read by phase 2
        if (ok && has_next) ++a_issued;
        const int r = a.HV / a.H;
        const bool first = hv % r == 0, last = hv % r == r - 1;  // of the key head's value heads
        if (ok) {  // thread d holds element d of the token rows m in [32 grp, 32 grp + 32);
                   // lanes 2i and 2i + 1 swap halves so that each stores bf16 pairs (d even,
                   // d + 1) of alternate tokens: even lanes tokens 2j, odd lanes 2j + 1.
                   // The dkhat terms are added to the key head's sums (fp32, value heads
                   // in order); dv is this value head's own.
            const int d = sub * 32 + lane, odd = lane & 1;
            const size_t ts = (size_t)a.HV * kDim;
            const size_t base = ((size_t)t0 * a.HV + hv) * kDim + (d & ~1) + (size_t)odd * ts;
    #pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // 16 token columns at a time
                const int m0 = j0 + 16 * hh;
                float dk[16], wt[16], ut[16], acc[16];
                tmem_ld16(t_row + cDK + m0, dk);
                tmem_ld16(t_row + cWT + m0, wt);
                tmem_ld16(t_row + cUT + m0, ut);
                if (!first) tmem_ld16(t_row + cACC + m0, acc);
                tmem_ld_wait();
    #pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int me = m0 + 2 * jj;  // the even token of the pair
                    const float b0 = sm.beta[me], b1 = sm.beta[me + 1];
                    const float k0 = dk[2 * jj] + b0 * sm.eg[me] * wt[2 * jj];
                    const float k1 = dk[2 * jj + 1] + b1 * sm.eg[me + 1] * wt[2 * jj + 1];
                    acc[2 * jj] = (first ? 0.f : acc[2 * jj]) + k0;
                    acc[2 * jj + 1] = (first ? 0.f : acc[2 * jj + 1]) + k1;
                    const float v0 = b0 * ut[2 * jj], v1 = b1 * ut[2 * jj + 1];
                    const float rv = __shfl_xor_sync(0xffffffffu, odd ? v0 : v1, 1);
                    if (me + odd < L && in_range(base + (size_t)me * ts, 2, n_rows_hv(a), a.status)) {
                        const size_t o = base + (size_t)me * ts;
                        *reinterpret_cast<uint32_t *>(a.dv + o) = odd ? pack_bf2(rv, v1) : pack_bf2(v0, rv);
                    }
                    if (last) {  // the key head's summed terms, staged as bf16 rows [t][d]
                        bf16 *stg = reinterpret_cast<bf16 *>(sm.op_b);
                        stg[me * kDim + d] = __float2bfloat16_rn(acc[2 * jj]);
                        stg[(me + 1) * kDim + d] = __float2bfloat16_rn(acc[2 * jj + 1]);
                    }
                }
                if (!last) tmem_st16(t_row + cACC + m0, acc);
            }
            tmem_st_wait();
        } else if (tid == 0 && a.status) {
            atomicOr(a.status, 2);
        }
        __syncthreads();
        if (ok && last) dk_pass(t0, x.h, L);
        if (ok && warp == 0) {  // dg = reverse cumulative sum of dG (warp scan), dbeta
            float dgv[2];
    #pragma unroll
            for (int z = 0; z < 2; ++z) {
                const int m = 2 * lane + z;
                dgv[z] = m < L ? sm.dG[m] : 0.f;
            }
            const float pair = dgv[0] + dgv[1];
            float suf = pair;
    #pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane + off < 32) suf += y;
            }
            const float after = suf - pair;  // sum over elements 2*lane+2 ...
            float pa = 0.f, pd = 0.f;        // fused gating: sums of dg g and of da over the chunk
    #pragma unroll
            for (int z = 0; z < 2; ++z) {
                const int m = 2 * lane + z;
                if (m < L && in_range((size_t)(t0 + m) * a.HV + hv, 1, n_tok_hv(a), a.status)) {
                    const size_t gi = (size_t)(t0 + m) * a.HV + hv;
                    const float dgm = (z == 0 ? dgv[0] + dgv[1] : dgv[1]) + after;
                    store_dbeta(a, gi, sm.db[m], sm.beta[m]);
                    if (a.beta_mode == 2) {  // da = dg (-e^{A_log}) softplus'(a + dt_bias)
                        const float x = bf2f(a.ga[gi]) + a.dt_bias[hv], nea = -expf(a.A_log[hv]);
                        const float da = dgm * nea * gate_softplus_slope(x);
                        a.da[gi] = f2bf(da);
                        pa += dgm * (nea * gate_softplus(x));
                        pd += da;
                    } else {
                        a.dg[gi] = dgm;
                    }
                }
            }
            if (a.beta_mode == 2) {
                pa = warp_sum(pa);
                pd = warp_sum(pd);
                if (lane == 0 && in_range((size_t)c * a.HV + hv, 1, (long long)a.num_chunks * a.HV, a.status))
                    reinterpret_cast<float2 *>(a.gpart)[(size_t)c * a.HV + hv] = make_float2(pa, pd);
            }
        }
        tc_fence_before();
        ok = __syncthreads_and(ok);  // the unit's scalars, operand tiles and TMEM are free
        if (!ok) break;
        x = nx;
    }
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        // drain the loads still in flight (bounded) before leaving
        if (a_issued > waited) mbar_wait(&sm.a_bar, (a_issued - 1) & 1, kDrainLimitNs);
        if (v_issued > waited) mbar_wait(&sm.v_bar, (v_issued - 1) & 1, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
}

}  // namespace

cudaError_t launch_bintra_b_tc(const ChunkArgs &a, cudaStream_t s) {
    if (a.num_chunks == 0) return cudaSuccess;
    BwMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 256;
    if (!encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.v, a.v, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dw, a.dW, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dvn, a.dvnew, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.t, a.Tm, 1, (uint64_t)a.num_chunks * a.HV * 64, 128, 128, 64, 64) ||
        !encode_rows_bf16(&m.dkp, a.dkpart, a.H, a.T, rowb, rowb * a.H, 64))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BwSmem) + 1024;
    static_assert(2 * (sizeof(BwSmem) + 2048) <= 233472, "two CTAs per SM");
    cudaError_t e = cudaFuncSetAttribute(k_bintra_b_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = sm_count(&sms)) != cudaSuccess) return e;
    // whole groups of the r value heads of a key head per CTA (their dk sums)
    const int r = a.HV / a.H;
    const int nunits = a.num_chunks * a.HV, ngroups = nunits / r;
    const int slots = 2 * sms;
    const int per = (ngroups + slots - 1) / slots * r;
    TimerScope ts(a.timer, GDN_KERNEL_BINTRA_B, s);
    k_bintra_b_tc<<<(nunits + per - 1) / per, kThr, smem, s>>>(a, m, per);
    return cudaGetLastError();
}

}  // namespace gdn
