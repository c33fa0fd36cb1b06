// gdn_bintra_tc.cu -- backward terms of a chunk that go through the per-chunk
// states h (chunk start) and dh' (gradient of the state after the chunk) and
// through the intra-chunk attention matrix, on the tensor cores ("dqkwg" of
// "cake_gdn: deterministic chunked GDN training kernels", section 2).
//
// Persistent: one CTA of 512 threads per SM walks a contiguous run of (chunk,
// value head) units.  Its two halves of two warpgroups split every epilogue by
// side: the first takes the Q K^T / dM terms and the dq terms, the second dW and
// the dk terms.  The next unit's h, dh', dO, dv_new and v_new tiles load as soon
// as batch 1 has consumed the current ones; q and k (only when the key head
// changes) load into a second buffer at the start of the unit before, so the loads
// run under the epilogues.  With h_c, dh_c [k][v] (bf16,
// from the forward and reverse scans), dO, dv_new, v_new [t][v], Qhat =
// diag(scale / r_q) Q, Khat = diag(1 / r_k) K and Gamma_ij = exp(G_i - G_j):
//   batch 1 (M=64, rows = tokens, contraction 128):
//     Dq = dO h^T,  Dw = dv_new h^T,  Dk = v_new dh'^T     (N = 128)
//     QK = Q K^T,   dM = dO v_new^T                         (N = 64)
//   dW = -Dw (to HBM, for the WY pullback);
//   M_ij = QK_ij scale / (r_q,i r_k,j) Gamma_ij,  dMG = dM (.) Gamma,  P1 = dM (.) M
//   (j <= i);
//   batch 2 (M=64, contraction 64): dMG Khat and dMG^T Qhat;
//   dqhat_t = e^{G_t} Dq_t + (dMG Khat)_t
//   dkhat_t = e^{G_L - G_t} Dk_t + (dMG^T Qhat)_t           (the rest comes from the WY
//                                                              pullback)
// A CTA walks whole groups of the r = HV / H value heads of one key head, which
// share q and k, and sums dqhat and dkhat over them in registers (fp32, value heads
// in order).  After the group's last value head it writes the key head's dq with the
// L2-norm backward applied, dq = (scale dqhat - nq (nq . scale dqhat)) / r_q with
// nq = q / r_q, and the summed dkhat terms (bf16 [T, H, 128]) that the WY pullback
// completes;
//   dG_t    = qhat_t . e^{G_t} Dq_t - xi_t + sum_j P1_tj - sum_i P1_it,
//   xi_t = khat_t . e^{G_L - G_t} Dk_t,   dG_L += sum_t xi_t + e^{G_L} <h, dh'>.
// h / dh' are read as [N=k][K=v], i.e. their [k][v] tiles K-major; all tiles
// come by TMA.  An M=64 result row t sits in TMEM lane 32 (t / 16) + t % 16; the
// two warpgroups split the columns.  Column sums are warp butterflies.
#include <stddef.h>
#include <string.h>

#include "gdn_epi.cuh"
#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;
using epi::colsum16;
using epi::pack_bf2;
using epi::colsum_frag;
using epi::colsum_frag_col;
using epi::get_pair;
using epi::put_pair;
using epi::quad_sum;
using epi::tmem_ld16x256_x4;

constexpr int kThr = 512;   // two halves of two warpgroups: the dq side and the dk side
constexpr uint32_t kBox = 64 * 128;       // 64 rows x 128 B
constexpr uint32_t kBig = 128 * 128;      // 128 rows x 128 B
constexpr uint32_t kHV = kBig + kBox;     // one v-half of h_c and of v_new

// TMEM columns (512 allocated)
// Dq and dM share their A operand (dO) and come out of one N = 192 product: B is a
// v-half of h_c followed by the same v-half of v_new
constexpr uint32_t cDQ = 0, cDM = 128, cQK = 192, cDW = 256, cDK = 384;   // batch 1
constexpr uint32_t cQI = 128, cKI = 256;                                   // batch 2
// Every product here is M = 64, which fills lanes 0..15 of each 32-lane quarter; the
// key head's dqhat / dkhat sums live in lanes 16..31 of the Dq / Dk columns, in the
// 16x256b fragment layout of the epilogue (the MMAs never write those lanes).
constexpr uint32_t kAccLanes = 16u << 16;
// The next unit's group-A tiles are issued by lane 0 of warp 8, on the dk side, whose
// part of the epilogue that follows is the lighter one (an issuing thread can stall).
constexpr int kLoader = 256;

struct BaSmem {
    unsigned char hvn[2 * kHV];   // per v-half: h_c [k][v] (128 rows), then v_new [t][v] (64 rows)
    unsigned char dh[2 * kBig];   // dh_c [k][v]
    unsigned char dO[2 * kBox];   // [t][v]
    unsigned char dvn[2 * kBox];
    unsigned char q[2][2 * kBox];  // [t][k], two buffers (the next key head loads into the other)
    unsigned char k[2][2 * kBox];
    unsigned char op_dmg[kBox];   // dMG_tj / r_k,j        [t][j]  K-major A of dMG Khat
    unsigned char op_dmgt[kBox];  // dMG_it scale / r_q,i  [i][t]  MN-major A of dMG^T Qhat
                                  // (after batch 2, with op_dmg: the dqhat rows of a full chunk)
    unsigned char stg[2 * kBox];  // rows of a full chunk staged for TMA stores: dW, then dkhat
    float pq[2][64], pk[2][64];   // per-warpgroup partial row dots
    float pn[2][64];              // per-warpgroup partial row dots q . (summed dqhat)
    float iq[2][64];              // 1 / r_q (0 past L); [2]: this unit's and the next one's
    float rp[2][64];              // per-warpgroup partial row sums of P1
    float cp[4][64];              // per-row-block column sums of P1
    float hdh[2][4];              // per-warp partial <h, dh'> (warps 8..11), by unit parity
    float G[2][64], eg[64], egl_g[64];  // G, e^{G_t}, e^{G_L - G_t} (0 past L)
    float qsc[2][64], rki[2][64];       // scale / r_q, 1 / r_k
    uint64_t a_bar, b_bar[2], mma_bar;   // group A (h, dh, dO, dv_new, v_new), group B (q, k) per buffer
    uint32_t tmem_base;
};

// Every TMA / SW128 tile starts on a 1024-byte boundary of the (1024-aligned) struct.
static_assert(offsetof(BaSmem, dh) % 1024 == 0 && offsetof(BaSmem, dO) % 1024 == 0 &&
                  offsetof(BaSmem, dvn) % 1024 == 0 && kHV % 1024 == 0 &&
                  offsetof(BaSmem, q) % 1024 == 0 && offsetof(BaSmem, k) % 1024 == 0 &&
                  offsetof(BaSmem, op_dmg) % 1024 == 0 && offsetof(BaSmem, op_dmgt) % 1024 == 0 &&
                  offsetof(BaSmem, stg) % 1024 == 0,
              "SW128 tiles on 1024-byte boundaries");

struct BaMaps {
    CUtensorMap h, dh, dO, dvn, vn, q, k;
    CUtensorMap dw, dq, dkp;    // outputs, stored by TMA from a full chunk's staged rows
};

struct Unit {
    int c, hv, h, t0, L;
};

__device__ __forceinline__ Unit unit_of(const ChunkArgs &a, int u) {
    Unit x;
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
__device__ __forceinline__ Unit next_unit(const ChunkArgs &a, const Unit &x) {
    if (x.hv + 1 < a.HV) {
        Unit y = x;
        y.hv = x.hv + 1;
        y.h = y.hv / (a.HV / a.H);
        return y;
    }
    return unit_of(a, (x.c + 1) * a.HV);
}

__device__ __forceinline__ void issue_a(const BaMaps &m, BaSmem &sm, const ChunkArgs &a, const Unit &x) {
    const int row = (x.c * a.HV + x.hv) * 128;
    mbar_arrive_expect_tx(&sm.a_bar, 4 * kBig + 6 * kBox);
    tma_load_3d(sm.hvn, &m.h, 0, 0, row, &sm.a_bar);
    tma_load_3d(sm.hvn + kHV, &m.h, 64, 0, row, &sm.a_bar);
    tma_load_3d(sm.dh, &m.dh, 0, 0, row, &sm.a_bar);
    tma_load_3d(sm.dh + kBig, &m.dh, 64, 0, row, &sm.a_bar);
    tma_load_3d(sm.dO, &m.dO, 0, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dO + kBox, &m.dO, 64, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dvn, &m.dvn, 0, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.dvn + kBox, &m.dvn, 64, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.hvn + kBig, &m.vn, 0, x.hv, x.t0, &sm.a_bar);
    tma_load_3d(sm.hvn + kHV + kBig, &m.vn, 64, x.hv, x.t0, &sm.a_bar);
}

__device__ __forceinline__ void issue_b(const BaMaps &m, BaSmem &sm, const Unit &x, int bf) {
    mbar_arrive_expect_tx(&sm.b_bar[bf], 4 * kBox);
    tma_load_3d(sm.q[bf], &m.q, 0, x.h, x.t0, &sm.b_bar[bf]);
    tma_load_3d(sm.q[bf] + kBox, &m.q, 64, x.h, x.t0, &sm.b_bar[bf]);
    tma_load_3d(sm.k[bf], &m.k, 0, x.h, x.t0, &sm.b_bar[bf]);
    tma_load_3d(sm.k[bf] + kBox, &m.k, 64, x.h, x.t0, &sm.b_bar[bf]);
}


__global__ void __launch_bounds__(kThr, 1) k_bintra_a_tc(const ChunkArgs a,
                                                         const __grid_constant__ BaMaps maps, int per) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BaSmem &sm = smem_struct<BaSmem>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nunits = a.num_chunks * a.HV;
    const int ub = blockIdx.x * per, ue = min(nunits, ub + per);
    if (ub >= ue) return;
    const int side = warp >> 3;        // 0: (a) and the dq terms; 1: (b) and the dk terms
    const int grp = (warp >> 2) & 1;   // warpgroup within the side: which column half
    const int sub = warp & 3;          // TMEM lane quarter

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.a_bar, 1);
        mbar_init(&sm.b_bar[0], 1);
        mbar_init(&sm.b_bar[1], 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = sm.tmem_base;
    const uint32_t t_row = tb + ((uint32_t)(sub * 32) << 16);
    Unit x = unit_of(a, ub);
    if (tid == 0) {
        issue_a(maps, sm, a, x);
        issue_b(maps, sm, x, 0);
    }
    int a_issued = 1, a_waited = 0;           // same on every thread
    uint32_t bpar = 0, bpend = 1;  // per q / k buffer (bit i): parity of its next wait, a load in flight
    int bcur = 0;         // the q / k buffer of the current unit
    bool need_b = true;   // the current unit waits for a q / k load
    // Warp 0 issues the products and does nothing else while they run (its issuing
    // thread stalls for as long as the tensor pipe is full); meanwhile warp 1 finishes
    // the unit before's dG, warps 2 and 3 own the per-token scalars (token ft = tid - 64),
    // fetched one unit ahead, and warps 8..11 take the <h, dh'> dot.
    const int ft = tid - 64;
    const bool scal = ft >= 0 && ft < 64;
    float pG = 0.f, pRq = 1.f, pRk = 1.f;
    auto fetch = [&](const Unit &y) {
        if (scal && ft < y.L && in_range((size_t)(y.t0 + ft) * a.HV + y.hv, 1, n_tok_hv(a), a.status)) {
            const size_t r = (size_t)(y.t0 + ft) * a.H + y.h;
            pG = a.G[(size_t)(y.t0 + ft) * a.HV + y.hv];
            pRq = a.rq[r];
            pRk = a.rk[r];
        } else {
            pG = 0.f; pRq = 1.f; pRk = 1.f;
        }
    };
    fetch(x);
    bool ok = true;
    uint32_t phase = 0;
    // a unit's scalars go into buffer buf at the end of the unit before (the first
    // unit's here), off the unit's own chain: the divides run while nothing waits on them
    auto publish = [&](int Ly, int buf) {
        if (scal) {
            const bool in = ft < Ly;
            sm.G[buf][ft] = pG;
            sm.qsc[buf][ft] = in ? a.scale / pRq : 0.f;
            sm.rki[buf][ft] = in ? 1.f / pRk : 0.f;
            sm.iq[buf][ft] = in ? 1.f / pRq : 0.f;
        }
    };
    publish(x.L, 0);
    // A unit's dG runs on warp 1 during the next unit's first product batch (warp 1 is
    // idle there: warp 0 issues the products, warps 2 and 3 fetch scalars, warps 8..11
    // take the <h, dh'> dot).
    struct Pend {
        bool on;
        int t0, hv, L, buf;
    };
    Pend pend = {false, 0, 0, 0, 0};
    auto finish_dg = [&](const Pend &p) {  // dG_t, and the G_L terms summed in a fixed order
        const float *pRki = sm.rki[p.buf], *pQsc = sm.qsc[p.buf];
        const float Gl = p.L > 0 ? sm.G[p.buf][p.L - 1] : 0.f;
        float dgz[2], sx = 0.f;
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int tt = 2 * lane + z;
            float dg = 0.f, xi = 0.f;
            if (tt < p.L) {
                xi = (sm.pk[0][tt] + sm.pk[1][tt]) * pRki[tt];
                const float cps = ((sm.cp[0][tt] + sm.cp[1][tt]) + sm.cp[2][tt]) + sm.cp[3][tt];
                dg = (sm.pq[0][tt] + sm.pq[1][tt]) * pQsc[tt] - xi + (sm.rp[0][tt] + sm.rp[1][tt]) - cps;
            }
            sx += xi;
            dgz[z] = dg;
        }
        sx = warp_sum(sx);
        float hd = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) hd += sm.hdh[p.buf][w];
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int tt = 2 * lane + z;
            if (tt < p.L && in_range((size_t)(p.t0 + tt) * a.HV + p.hv, 1, n_tok_hv(a), a.status)) {
                const float extra = (tt == p.L - 1) ? sx + __expf(Gl) * hd : 0.f;
                a.dGp[(size_t)(p.t0 + tt) * a.HV + p.hv] = dgz[z] + extra;
            }
        }
    };
    for (int u = ub; u < ue; ++u) {
        const bool has_next = u + 1 < ue;
        const int L = x.L;
        const int cur = (u - ub) & 1;
        const float *sG = sm.G[cur], *sQsc = sm.qsc[cur], *sRki = sm.rki[cur], *sIq = sm.iq[cur];
        bool got = mbar_wait(&sm.a_bar, a_waited & 1);
        if (need_b) got = mbar_wait(&sm.b_bar[bcur], (bpar >> bcur) & 1) && got;
        got = __syncthreads_and(got);
        ++a_waited;
        if (need_b) {
            bpar ^= 1u << bcur;
            bpend &= ~(1u << bcur);
        }
        if (!got) { ok = false; break; }
        const float Gl = L > 0 ? sG[L - 1] : 0.f;
        if (scal) {
            const bool in = ft < L;
            const float Gt = sG[ft];
            sm.eg[ft] = in ? __expf(Gt) : 0.f;
            sm.egl_g[ft] = in ? __expf(fminf(Gl - Gt, 0.f)) : 0.f;
        }
        if (tid == 0) {  // batch 1
            tc_fence_after();
            const uint32_t id192 = idesc_bf16(64, 192, 0, 0), id128 = idesc_bf16(64, 128, 0, 0),
                           id64 = idesc_bf16(64, 64, 0, 0);
            const uint32_t hs = smem_u32(sm.hvn), dhs = smem_u32(sm.dh);
            const uint32_t os = smem_u32(sm.dO), ds = smem_u32(sm.dvn);
            const uint32_t qs = smem_u32(sm.q[bcur]), ks = smem_u32(sm.k[bcur]);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t ao = (s >> 2) * kBox + (s & 3) * 32, bo = (s >> 2) * kBig + (s & 3) * 32;
                const uint32_t ho = (s >> 2) * kHV + (s & 3) * 32;  // h_c, then v_new at + kBig
                mma_bf16(tb + cDQ, sdesc(os + ao, 16, 1024), sdesc(hs + ho, 16, 1024), id192, s > 0);
                mma_bf16(tb + cDW, sdesc(ds + ao, 16, 1024), sdesc(hs + ho, 16, 1024), id128, s > 0);
                mma_bf16(tb + cDK, sdesc(hs + kBig + ho, 16, 1024), sdesc(dhs + bo, 16, 1024), id128, s > 0);
                mma_bf16(tb + cQK, sdesc(qs + ao, 16, 1024), sdesc(ks + ao, 16, 1024), id64, s > 0);
            }
            mma_commit(&sm.mma_bar);
        }
        // the next unit (its table entries are a dependent load: after the MMA issue)
        const Unit nx = has_next ? next_unit(a, x) : x;
        if (has_next) fetch(nx);
        // a new key head for the next unit: its q / k load into the other buffer now (that
        // buffer's last reader, an earlier unit, has finished)
        const bool need_next_b = has_next && (nx.c != x.c || nx.h != x.h);
        if (need_next_b) {
            if (tid == 0) issue_b(maps, sm, nx, bcur ^ 1);
            bpend |= 1u << (bcur ^ 1);
        }
        // <h, dh'> while the products run: thread tid - 256 of warps 8..11 takes a row
        // of h and dh'
        if (warp >= 8 && warp < 12) {
            const int kr = tid - 256;
            float hdh = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint32_t off = sw128_off(kr, q8 * 8);
                    const uint4 xx = *reinterpret_cast<const uint4 *>(sm.hvn + half * kHV + off);
                    const uint4 yy = *reinterpret_cast<const uint4 *>(sm.dh + half * kBig + off);
                    const __nv_bfloat162 *xb = reinterpret_cast<const __nv_bfloat162 *>(&xx);
                    const __nv_bfloat162 *yb = reinterpret_cast<const __nv_bfloat162 *>(&yy);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 xf = __bfloat1622float2(xb[e]), yf = __bfloat1622float2(yb[e]);
                        hdh += xf.x * yf.x + xf.y * yf.y;
                    }
                }
            hdh = warp_sum(hdh);
            if (lane == 0) sm.hdh[cur][warp - 8] = hdh;
        }
        if (pend.on && warp == 1) finish_dg(pend);  // the unit before's, while the products run
        if (tid == 0) tma_store_wait_read();  // the last unit's staged rows have been read
        bool done = __syncthreads_and(mbar_wait(&sm.mma_bar, phase));
        phase ^= 1;
        tc_fence_after();
        if (!done) { ok = false; break; }
        // group A has been consumed (batch 1 and the dot): load the next unit's
        if (has_next) {
            if (tid == kLoader) issue_a(maps, sm, a, nx);
            ++a_issued;
        }
        const int ra = sub * 16 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);  // fragment rows / column
        const bool la = ra < L, lb = rb < L;
        if (side == 0) {
            // (a) QK, dM -> P1 (row and column sums) and the two dMG operand rows, read
            // as 16x256b fragments: rows ra, rb = ra + 8, columns j0 + 8k + cq + {0, 1}
            const int j0 = 32 * grp;
            float qk[16], dm[16];
            tmem_ld16x256_x4(t_row + cQK + j0, qk);
            tmem_ld16x256_x4(t_row + cDM + j0, dm);
            tmem_ld_wait();
            const float Ga = sG[ra], Gb = sG[rb], qsa = sQsc[ra], qsb = sQsc[rb];
            float rsa = 0.f, rsb = 0.f, pc[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {  // in place: dm <- dMG, qk <- P1
                    const int j = j0 + 8 * k + cq + (e & 1);
                    const bool up = e & 2;
                    const int r = up ? rb : ra;
                    const float msk = ((up ? lb : la) && j <= r) ? 1.f : 0.f;
                    dm[4 * k + e] *= msk * __expf(fminf((up ? Gb : Ga) - sG[j], 0.f));
                    qk[4 * k + e] = dm[4 * k + e] * qk[4 * k + e] * (up ? qsb : qsa) * sRki[j];
                    if (up) rsb += qk[4 * k + e]; else rsa += qk[4 * k + e];
                }
                pc[2 * k] = qk[4 * k] + qk[4 * k + 2];
                pc[2 * k + 1] = qk[4 * k + 1] + qk[4 * k + 3];
                const int j = j0 + 8 * k + cq;
                const float r0 = sRki[j], r1 = sRki[j + 1];
                put_pair(sm.op_dmg, ra, j, dm[4 * k] * r0, dm[4 * k + 1] * r1);
                put_pair(sm.op_dmg, rb, j, dm[4 * k + 2] * r0, dm[4 * k + 3] * r1);
                put_pair(sm.op_dmgt, ra, j, dm[4 * k] * qsa, dm[4 * k + 1] * qsa);
                put_pair(sm.op_dmgt, rb, j, dm[4 * k + 2] * qsb, dm[4 * k + 3] * qsb);
            }
            sm.cp[sub][j0 + colsum_frag_col(lane)] = colsum_frag(pc, lane);
            rsa = quad_sum(rsa);
            rsb = quad_sum(rsb);
            if ((lane & 3) == 0) {
                sm.rp[grp][ra] = rsa;
                sm.rp[grp][rb] = rsb;
            }
        } else {
            // (b) dW = -Dw rows on 16x256b fragments: rows ra, rb, this warpgroup's 64
            // columns 64 grp + 32 cc + 8k + cq + {0, 1}; a full chunk's rows are staged
            // (this warpgroup's 64-column half of stg) for one TMA store
            const size_t oa = ((size_t)(x.t0 + (la ? ra : 0)) * a.HV + x.hv) * kDim;
            const size_t ob = ((size_t)(x.t0 + (lb ? rb : 0)) * a.HV + x.hv) * kDim;
            float dw[2][16];
            tmem_ld16x256_x4(t_row + cDW + 64 * grp, dw[0]);
            tmem_ld16x256_x4(t_row + cDW + 64 * grp + 32, dw[1]);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int cl = 32 * cc + 8 * k + cq, col = 64 * grp + cl;
                    if (L == 64) {
                        put_pair(sm.stg + grp * kBox, ra, cl, -dw[cc][4 * k], -dw[cc][4 * k + 1]);
                        put_pair(sm.stg + grp * kBox, rb, cl, -dw[cc][4 * k + 2], -dw[cc][4 * k + 3]);
                    } else {
                        if (la && in_range(oa + col, 2, n_rows_hv(a), a.status))
                            *reinterpret_cast<uint32_t *>(a.dW + oa + col) = pack_bf2(-dw[cc][4 * k], -dw[cc][4 * k + 1]);
                        if (lb && in_range(ob + col, 2, n_rows_hv(a), a.status))
                            *reinterpret_cast<uint32_t *>(a.dW + ob + col) = pack_bf2(-dw[cc][4 * k + 2], -dw[cc][4 * k + 3]);
                    }
                }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {  // batch 2: dMG Khat -> cQI, dMG^T Qhat -> cKI (over the Dw columns)
            tc_fence_after();
            const uint32_t id_km = idesc_bf16(64, 128, 0, 1);  // A K-major, B MN-major
            const uint32_t id_mm = idesc_bf16(64, 128, 1, 1);  // A MN-major, B MN-major
            const uint32_t ks = smem_u32(sm.k[bcur]), qs = smem_u32(sm.q[bcur]);
            const uint32_t g1 = smem_u32(sm.op_dmg), g2 = smem_u32(sm.op_dmgt);
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                mma_bf16(tb + cQI, sdesc(g1 + s * 32, 16, 1024), sdesc(ks + s * 2048, kBox, 1024), id_km, s > 0);
                mma_bf16(tb + cKI, sdesc(g2 + s * 2048, kBox, 1024), sdesc(qs + s * 2048, kBox, 1024), id_mm, s > 0);
            }
            mma_commit(&sm.mma_bar);
            if (L == 64) {  // the staged dW rows
                tma_store_3d(&maps.dw, 0, x.hv, x.t0, sm.stg);
                tma_store_3d(&maps.dw, 64, x.hv, x.t0, sm.stg + kBox);
                tma_store_commit();
            }
        }
        done = __syncthreads_and(mbar_wait(&sm.mma_bar, phase));
        phase ^= 1;
        tc_fence_after();
        if (!done) { ok = false; break; }
        if (tid == 0) tma_store_wait_read();  // stg is rewritten below
        __syncthreads();
        const int r = a.HV / a.H;
        const bool first = x.hv % r == 0, last = x.hv % r == r - 1;  // of the key head's value heads
        {  // dqhat, dkhat rows (this warpgroup's 64 columns) added to the key head's sums,
           // and the inter-term row dots, on 16x256b fragments (rows ra, rb; columns
           // c0 + 8k + cq + {0, 1})
            const float ega = la ? sm.eg[ra] : 0.f, egb = lb ? sm.eg[rb] : 0.f;
            const float ela = la ? sm.egl_g[ra] : 0.f, elb = lb ? sm.egl_g[rb] : 0.f;
            float pna = 0.f, pnb = 0.f;
            {
                const int m = side;  // 0: dq with q; 1: dk with k
                const uint32_t cA = m ? cDK : cDQ, cB = m ? cKI : cQI;
                const unsigned char *tile = m ? sm.k[bcur] : sm.q[bcur];
                const float fa = m ? ela : ega, fb = m ? elb : egb;
                float xa = 0.f, xb = 0.f;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int c0 = 32 * (2 * grp + h2);
                    float dd[16], ii[16], acc[16];
                    tmem_ld16x256_x4(t_row + cA + c0, dd);
                    tmem_ld16x256_x4(t_row + cB + c0, ii);
                    if (!first) tmem_ld16x256_x4(t_row + kAccLanes + cA + c0, acc);
                    tmem_ld_wait();
                    const unsigned char *half = tile + (c0 >> 6) * kBox;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int col = (c0 & 63) + 8 * k + cq;  // within the 64-column half
                        const float2 qa = get_pair(half, ra, col), qb = get_pair(half, rb, col);
                        const float a0 = fa * dd[4 * k], a1 = fa * dd[4 * k + 1];
                        const float b0 = fb * dd[4 * k + 2], b1 = fb * dd[4 * k + 3];
                        xa += qa.x * a0 + qa.y * a1;
                        xb += qb.x * b0 + qb.y * b1;
                        const float v[4] = {a0 + ii[4 * k], a1 + ii[4 * k + 1], b0 + ii[4 * k + 2],
                                            b1 + ii[4 * k + 3]};
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[4 * k + e] = (first ? 0.f : acc[4 * k + e]) + v[e];
                        if (m == 0 && last) {
                            pna += qa.x * acc[4 * k] + qa.y * acc[4 * k + 1];
                            pnb += qb.x * acc[4 * k + 2] + qb.y * acc[4 * k + 3];
                        }
                    }
                    epi::tmem_st16x256_x4(t_row + kAccLanes + cA + c0, acc);
                }
                xa = quad_sum(xa); xb = quad_sum(xb);
                tmem_st_wait();
                if ((lane & 3) == 0) {
                    float (*dst)[64] = m ? sm.pk : sm.pq;
                    dst[grp][ra] = xa; dst[grp][rb] = xb;
                }
            }
            if (side == 0 && last) {
                pna = quad_sum(pna); pnb = quad_sum(pnb);
                if ((lane & 3) == 0) { sm.pn[grp][ra] = pna; sm.pn[grp][rb] = pnb; }
            }
        }
        __syncthreads();  // q / k tiles, TMEM and the row sums are all read or written
        if (last) {  // the key head's dq (L2-norm backward applied) and summed dkhat terms:
                     // full chunks staged for TMA stores, ragged ones stored directly
            const float sa = la ? sQsc[ra] : 0.f, sb = lb ? sQsc[rb] : 0.f;
            const float ia = la ? sIq[ra] : 0.f, ib = lb ? sIq[rb] : 0.f;
            const float Pa = (sm.pn[0][ra] + sm.pn[1][ra]) * ia * ia;
            const float Pb = (sm.pn[0][rb] + sm.pn[1][rb]) * ib * ib;
            const size_t oa = ((size_t)(x.t0 + (la ? ra : 0)) * a.H + x.h) * kDim;
            const size_t ob = ((size_t)(x.t0 + (lb ? rb : 0)) * a.H + x.h) * kDim;
            // side 0: dq (staged in op_dmg); side 1: the summed dkhat terms (staged in stg)
            bf16 *gout = side ? a.dkpart : a.dq;
            unsigned char *st = side ? sm.stg : sm.op_dmg;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c0 = 32 * (2 * grp + h2);
                const unsigned char *half = sm.q[bcur] + (c0 >> 6) * kBox;
                float av[16];
                tmem_ld16x256_x4(t_row + kAccLanes + (side ? cDK : cDQ) + c0, av);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int col = (c0 & 63) + 8 * k + cq, gcol = c0 + 8 * k + cq;
                    float v0 = av[4 * k], v1 = av[4 * k + 1], v2 = av[4 * k + 2], v3 = av[4 * k + 3];
                    if (side == 0) {
                        const float2 qa = get_pair(half, ra, col), qb = get_pair(half, rb, col);
                        v0 = sa * (v0 - qa.x * Pa); v1 = sa * (v1 - qa.y * Pa);
                        v2 = sb * (v2 - qb.x * Pb); v3 = sb * (v3 - qb.y * Pb);
                    }
                    if (L == 64) {
                        put_pair(st + (c0 >> 6) * kBox, ra, col, v0, v1);
                        put_pair(st + (c0 >> 6) * kBox, rb, col, v2, v3);
                    } else {
                        if (la && in_range(oa + gcol, 2, n_rows_h(a), a.status))
                            *reinterpret_cast<uint32_t *>(gout + oa + gcol) = pack_bf2(v0, v1);
                        if (lb && in_range(ob + gcol, 2, n_rows_h(a), a.status))
                            *reinterpret_cast<uint32_t *>(gout + ob + gcol) = pack_bf2(v2, v3);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0 && L == 64) {  // the staged dq and dkhat rows of key head h
                tma_store_3d(&maps.dq, 0, x.h, x.t0, sm.op_dmg);
                tma_store_3d(&maps.dq, 64, x.h, x.t0, sm.op_dmg + kBox);
                tma_store_3d(&maps.dkp, 0, x.h, x.t0, sm.stg);
                tma_store_3d(&maps.dkp, 64, x.h, x.t0, sm.stg + kBox);
                tma_store_commit();
            }
        }
        tc_fence_before();
        pend = {true, x.t0, x.hv, L, cur};
        if (has_next) publish(nx.L, cur ^ 1);
        __syncthreads();  // the per-unit scalars are free for the next unit
        if (need_next_b) bcur ^= 1;
        need_b = need_next_b;
        x = nx;
    }
    if (ok && pend.on && warp == 1) finish_dg(pend);  // the last unit's
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        // drain the loads still in flight (bounded) before leaving
        if (a_issued > a_waited) mbar_wait(&sm.a_bar, a_waited & 1, kDrainLimitNs);
        for (int bf = 0; bf < 2; ++bf)
            if ((bpend >> bf) & 1) mbar_wait(&sm.b_bar[bf], (bpar >> bf) & 1, kDrainLimitNs);
    }
    if (tid == 0) tma_store_wait_all();
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
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.dw, a.dW, a.HV, a.T, rowb, rowb * a.HV, 64) ||
        !encode_rows_bf16(&m.dq, a.dq, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.dkp, a.dkpart, a.H, a.T, rowb, rowb * a.H, 64))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BaSmem) + 1024;
    static_assert(sizeof(BaSmem) + 1024 <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(k_bintra_a_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // whole groups of the r value heads of a key head per CTA (their dq / dk sums)
    const int r = a.HV / a.H;
    const int nunits = a.num_chunks * a.HV, ngroups = nunits / r;
    const int grid = ngroups < sms ? ngroups : sms;
    const int per = (ngroups + grid - 1) / grid * r;
    TimerScope ts(a.timer, GDN_KERNEL_BINTRA_A, s);
    k_bintra_a_tc<<<(nunits + per - 1) / per, kThr, smem, s>>>(a, m, per);  // 16 warps
    return cudaGetLastError();
}

}  // namespace gdn
