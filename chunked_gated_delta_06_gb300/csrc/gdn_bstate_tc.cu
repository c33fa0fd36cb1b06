// gdn_bstate_tc.cu -- backward (reverse) inter-chunk state scan on the tensor
// cores ("dhu" in "cake_gdn: deterministic chunked GDN training kernels",
// section 2; the reverse recurrence of the GDN context-parallel dh scan in
// "Qwen3.5-397B RL trainer on 128 v7x", maxtext #5799).
//
// As in the forward scan, the value columns never mix, so one CTA (two
// warpgroups that split the columns of every pass) owns one (sequence, value
// head, value half) and walks the chunks in reverse.  dh[k][v'] (v' = 64 vb .. 64 vb + 63) lives in TMEM as fp32 (lane
// k, 64 columns), seeded with d(final state).  Per chunk, with dh' the gradient
// of the state after the chunk (= the current dh):
//   1. thread k writes row k of dh' as bf16 to shared memory (copied to
//      dh_c[chunk][hv][k][v'] by one TMA store), then dh <- e^{G_L} dh';
//   2. Pd[t][v'] = sum_k K[t][k] dh'[k][v']          (M=64 N=64 K=128)
//   3. on 16x256b fragments of Pd (two token rows and eight columns per lane):
//      dv_new[t][v'] = dv_loc + e^{G_L-G_t}/r_k,t Pd (bf16) and the operands
//      c_t dO[t][v'] and dv_new[t][v'], c_t = e^{G_t} scale / r_q,t; a full chunk's
//      dv_new goes to HBM by one TMA store of that operand tile;
//   4. dh += Q^T (c dO) - w^T dv_new                  (two M=128 N=64 K=64
//      products; Q is the raw tile read MN-major, w^T the chunk's [k][t] tile
//      read K-major, and the minus sign is the descriptor's negate-B bit)
// which is dh <- e^{G_L} dh' + Qtil^T dO - w^T dv_new and dv_new = dv_loc +
// Ktil dh'.  dh0 = dh at the sequence start.  The tiles are single-buffered so
// that two CTAs share an SM, and each group is reloaded for the next chunk as
// soon as it is free: K after step 2, the halves of dO and dv_loc after step 3,
// Q and w after step 4; every tile of the chunk after that is prefetched into L2
// a step ahead.  The chunk's scalar record (kc_t = e^{G_L - G_t} / r_k,t, qc_t =
// e^{G_t} scale / r_q,t and e^{G_L}, written by the WY pass) comes with K, into one of two
// buffers by the parity of the step; a chunk costs two block barriers.
// Waits are bounded.  Long sequences with few heads can be scanned segment-
// parallel (the plan of the forward scan; see k_bstate_tc).
#include <string.h>

#include "gdn_epi.cuh"
#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 256;
// Step 2's product and the h_c store are issued by lane 0 of warp 7 (which also waits
// for that store), so that warp 0 is not held up in the c_t dO work beside the
// product: an issuing thread stalls while the tensor pipe's queue is full.
constexpr int kPdIssuer = 224;
constexpr uint32_t kBox = 64 * 128;       // one 64-row x 128-byte SW128 box
constexpr uint32_t kXBytes = 4 * kBox;    // K (2 boxes), dO half, dv_loc half
constexpr uint32_t kYBytes = 4 * kBox;    // Q (2 boxes), w^T (128 rows: 2 boxes)

struct BStateSmem {
    unsigned char a_ds[128 * 128];      // dh' bf16 [k][v']
    unsigned char a_do[64 * 128];       // c_t dO bf16 [t][v']
    unsigned char a_dv[64 * 128];       // -dv_new bf16 [t][v']
    unsigned char x[kXBytes];
    unsigned char y[kYBytes];
    ScRec sc[2];                        // the scalar records of this and the next step
    uint64_t xk_bar, xd_bar, y_bar, mma_bar;   // X = K (xk) + dO, dv_loc halves (xd); Y = Q, w
    uint32_t tmem_base;
};

struct BStateMaps {
    CUtensorMap k, q, w, dO, dl, dhc;
    CUtensorMap dvn;   // dv_new [T][HV][128]: a full chunk's rows of this value half, stored by TMA
};

// K of chunk c (tokens from t0) and its scalar record, into record buffer rb
__device__ __forceinline__ void issue_xk(const BStateMaps &m, BStateSmem &sm, const ChunkArgs &a, int c, int t0,
                                         int h, int hv, int rb) {
    mbar_arrive_expect_tx(&sm.xk_bar, 2 * kBox + (uint32_t)sizeof(ScRec));
    bulk_load(&sm.sc[rb], a.sc + ((size_t)c * a.HV + hv) * kScRec, sizeof(ScRec), &sm.xk_bar);
    tma_load_3d(sm.x + 0 * kBox, &m.k, 0, h, t0, &sm.xk_bar);
    tma_load_3d(sm.x + 1 * kBox, &m.k, 64, h, t0, &sm.xk_bar);
}

__device__ __forceinline__ void issue_xd(const BStateMaps &m, BStateSmem &sm, int t0, int hv, int vb) {
    mbar_arrive_expect_tx(&sm.xd_bar, 2 * kBox);
    tma_load_3d(sm.x + 2 * kBox, &m.dO, 64 * vb, hv, t0, &sm.xd_bar);
    tma_load_3d(sm.x + 3 * kBox, &m.dl, 64 * vb, hv, t0, &sm.xd_bar);
}

// L2 prefetch of every tile of chunk c (tokens from t0; loaded a step later);
// transition columns read no dO / dv_loc
__device__ __forceinline__ void prefetch_chunk(const BStateMaps &m, const ChunkArgs &a, int c, int t0, int h,
                                               int hv, int vb, bool with_d) {
    tma_prefetch_3d(&m.k, 0, h, t0);
    tma_prefetch_3d(&m.k, 64, h, t0);
    if (with_d) {
        tma_prefetch_3d(&m.dO, 64 * vb, hv, t0);
        tma_prefetch_3d(&m.dl, 64 * vb, hv, t0);
    }
    tma_prefetch_3d(&m.q, 0, h, t0);
    tma_prefetch_3d(&m.q, 64, h, t0);
    tma_prefetch_3d(&m.w, 0, 0, (c * a.HV + hv) * kDim);
}

__device__ __forceinline__ void issue_y(const BStateMaps &m, BStateSmem &sm, const ChunkArgs &a, int c, int t0,
                                        int h, int hv) {
    mbar_arrive_expect_tx(&sm.y_bar, kYBytes);
    tma_load_3d(sm.y + 0 * kBox, &m.q, 0, h, t0, &sm.y_bar);
    tma_load_3d(sm.y + 1 * kBox, &m.q, 64, h, t0, &sm.y_bar);
    tma_load_3d(sm.y + 2 * kBox, &m.w, 0, 0, (c * a.HV + hv) * kDim, &sm.y_bar);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// pass 0: every sequence in one piece.  Segment-parallel reverse scan (the forward
// scan's segments of a.seg_len chunks, walked from the last): pass 1 scans the last
// segment from d(final state) (all outputs, end state to seg_end) beside the
// pre-scans of segments S-2 .. 1, which start from dh = 0 with the transition
// columns [dh | Psi] (Psi from the identity, dO = dv_loc = 0 there) and store only
// their end state; k_seg_stitch turns those into the start states (the gradient
// after each segment's last chunk) of segments S-2 .. 0; pass 2 re-scans them.
// Segment records are indexed by rho = S - 1 - segment.
template <int pass>
__global__ void __launch_bounds__(kThr, 2)
    k_bstate_tc(const ChunkArgs a, const __grid_constant__ BStateMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BStateSmem &sm = smem_struct<BStateSmem>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) tma_prefetch_maps(maps);
    const int ncol = pass == 1 ? 4 : 2;            // column blocks of 64 per value head
    const int hv = blockIdx.x / ncol, cbk = blockIdx.x % ncol;
    const bool phi = pass == 1 && cbk >= 2;        // transition columns (pass 1 only)
    const int vb = cbk & 1;
    const int nsy = pass ? a.seg_max - 1 : 1;
    if (!in_range(blockIdx.y / nsy, 1, a.N, a.status)) return;
    const int n = a.seq_order[blockIdx.y / nsy];   // longest sequences first
    if (!in_range(n, 2, a.N + 1, a.status)) return;
    const int h = hv / (a.HV / a.H);
    const int cb = a.seq_chunk_off[n];
    const int ce = min(a.seq_chunk_off[n + 1], a.num_chunks);
    if (ce > cb && !in_range(cb, ce - cb, a.num_chunks, a.status)) return;
    const int nseq = max(ce - cb, 0);
    const int S = pass ? max(1, (nseq + a.seg_len - 1) / a.seg_len) : 1;
    const int rho = pass == 2 ? blockIdx.y % nsy + 1 : (pass ? blockIdx.y % nsy : 0);
    if (pass == 1 && !(S == 1 ? (rho == 0 && !phi) : (rho == 0 ? !phi : rho <= S - 2))) return;
    if (pass == 2 && !(S >= 2 && rho <= S - 1)) return;
    const bool from_input = rho == 0;              // d(final state) (else zero or seg_start)
    const bool pre = pass == 1 && rho >= 1;        // pre-scan: no per-chunk outputs
    const bool to_final = pass == 0 || (pass == 1 && S == 1) || (pass == 2 && rho == S - 1);
    const int sgm = S - 1 - rho;                   // the segment, in chunk order
    const int jend = pass ? min(nseq, (sgm + 1) * a.seg_len) : nseq;  // one past its last chunk
    const int nch = pass ? max(0, jend - sgm * a.seg_len) : nseq;
    const int grp = warp >> 2, sub = warp & 3;
    const int kr = sub * 32 + lane;     // state row (TMEM lane) of step 1
    const int c0 = 32 * grp;            // this warpgroup's 32 of the 64 columns
    // the sequence's chunks are consecutive 64-token blocks of [ts0, ts1); the
    // i-th step of the reverse walk handles block jend - 1 - i
    const int ts0 = nseq > 0 ? a.chunk_start[cb] : 0;
    const int ts1 = nseq > 0 ? a.chunk_start[ce - 1] + a.chunk_len[ce - 1] : 0;
    auto step_t0 = [&](int i) { return ts0 + 64 * (jend - 1 - i); };
    auto step_len = [&](int i) { return min(64, ts1 - step_t0(i)); };
    auto step_c = [&](int i) { return cb + jend - 1 - i; };  // its chunk

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.xk_bar, 1);
        mbar_init(&sm.xd_bar, 1);
        mbar_init(&sm.y_bar, 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t t_row = tbase + ((uint32_t)(sub * 32) << 16);
    const uint32_t tS = t_row + c0, tP = t_row + 64 + c0;   // this warpgroup's columns

    int xk_issued = 0, xd_issued = 0, y_issued = 0;  // load counts (thread 0's are complete)
    if (tid == 0 && nch > 0) {
        issue_xk(maps, sm, a, step_c(0), step_t0(0), h, hv, 0);
        if (!phi) issue_xd(maps, sm, step_t0(0), hv, vb);
        issue_y(maps, sm, a, step_c(0), step_t0(0), h, hv);
        if (nch > 1) prefetch_chunk(maps, a, step_c(1), step_t0(1), h, hv, vb, !phi);
        xk_issued = y_issued = 1;
        xd_issued = phi ? 0 : 1;
    }
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim + (size_t)kr * kDim + 64 * vb + c0;
    // segment buffers: seg_end[n][rho][hv][k][256] (dh | Psi), seg_start[n][rho-1][hv][k][128]
    float *send = pass == 1 ? a.seg_end + (((size_t)n * (a.seg_max - 1) + rho) * a.HV + hv) * kDim * 2 * kDim +
                                  (size_t)kr * (2 * kDim) + (phi ? kDim : 0) + 64 * vb + c0
                            : nullptr;
    {
        float r[32];
        if (pre) {  // dh from zero; Psi from the identity (row k, column k' = 64 vb + c0 + j)
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = (phi && kr == 64 * vb + c0 + j) ? 1.f : 0.f;
        } else if (!from_input) {
            const size_t off = (((size_t)n * (a.seg_max - 1) + rho - 1) * a.HV + hv) * kDim * kDim +
                               (size_t)kr * kDim + 64 * vb + c0;
            const float4 *src = reinterpret_cast<const float4 *>(a.seg_start + off);
            const bool in = in_range(off, 32, (long long)a.N * (a.seg_max - 1) * a.HV * kDim * kDim, a.status);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = in ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
        } else if (a.d_ht && in_range(sbase, 32, n_states(a), a.status)) {
            const float4 *src = reinterpret_cast<const float4 *>(a.d_ht + sbase);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = src[q];
                r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0.f;
        }
        tmem_st32(tS, r);
        tmem_st_wait();
    }
    __syncthreads();
    const uint32_t idP = idesc_bf16(64, 64, 0, 1);    // Pd = K dh'          (dh' MN-major)
    const uint32_t idS = idesc_bf16(128, 64, 1, 1);   // dh += Q^T A       (both MN-major)
    // dh -= w^T dv_new: w^T K-major, dv_new MN-major and negated by the descriptor's
    // negate-B bit (bit 14), so that the operand tile holds +dv_new and is also the
    // source of dv_new's TMA store
    const uint32_t idW = idesc_bf16(128, 64, 0, 1) | (1u << 14);
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
        const int c = step_c(i);
        const uint32_t par = i & 1;
        const int t0 = step_t0(i), L = step_len(i);
        const ScRec &rec = sm.sc[par];
        // K and the scalar record (e^{G_L} is needed right below)
        const bool gk = mbar_wait(&sm.xk_bar, par);
        const float egl = rec.egl;
        // 1. dh' -> bf16 operand (copied to dh_c by TMA below), then dh <- e^{G_L} dh'
        {
            float r[32];
            tmem_ld32(tS, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(sm.a_ds + sw128_off(kr, c0 + 8 * q)) =
                    make_uint4(pack_bf2(r[8 * q], r[8 * q + 1]), pack_bf2(r[8 * q + 2], r[8 * q + 3]),
                               pack_bf2(r[8 * q + 4], r[8 * q + 5]), pack_bf2(r[8 * q + 6], r[8 * q + 7]));
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= egl;
            tmem_st32(tS, r);
            tmem_st_wait();
        }
        if (tid == 0) tma_store_wait_read();  // the last step's dv_new store has read a_dv
        fence_proxy_async_smem();
        tc_fence_before();
        const bool gx = gk && (phi || mbar_wait(&sm.xd_bar, par));
        ok = __syncthreads_and(ok && gx);
        if (!ok) break;
        // 2. Pd = K dh'
        if (tid == kPdIssuer) {
            tc_fence_after();
            const uint32_t as = smem_u32(sm.a_ds), ks = smem_u32(sm.x);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tbase + 64, sdesc(ks + (s >> 2) * kBox + (s & 3) * 32, 16, 1024),
                         sdesc(as + s * 2048, kBox, 1024), idP, s > 0);
            mma_commit(&sm.mma_bar);
            if (!pre) {
                tma_store_3d(&maps.dhc, 64 * vb, 0, (c * a.HV + hv) * 128, sm.a_ds);  // dh_c rows (k)
                tma_store_commit();
            }
        }
        // meanwhile: c_t dO on the fragment positions used below (rows ra, ra + 8,
        // columns c0 + 8k + cq + {0, 1}); transition columns have no dO term
        const int ra = sub * 16 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
        if (!phi) {
            const float qa = rec.qc[ra], qb = rec.qc[rb];
            const unsigned char *dos = sm.x + 2 * kBox;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int col = c0 + 8 * k + cq;
                const float2 fa = epi::get_pair(dos, ra, col), fb = epi::get_pair(dos, rb, col);
                epi::put_pair(sm.a_do, ra, col, fa.x * qa, fa.y * qa);
                epi::put_pair(sm.a_do, rb, col, fb.x * qb, fb.y * qb);
            }
        }
        ok = mbar_wait(&sm.mma_bar, phase) && ok;
        phase ^= 1;
        tc_fence_after();
        if (tid == 0 && ok && i + 1 < nch) {  // K has been read by step 2
            issue_xk(maps, sm, a, step_c(i + 1), step_t0(i + 1), h, hv, par ^ 1);
            ++xk_issued;
        }
        // 3. dv_new = dv_loc + kc_t Pd on 16x256b fragments
        {
            float p[16];
            epi::tmem_ld16x256_x4(tP, p);
            tmem_ld_wait();
            const bool la = ra < L, lb = rb < L;
            const float ka = rec.kc[ra], kb = rec.kc[rb];
            // dv_new goes to a_dv (the operand of step 4, and for a full chunk the source
            // of one TMA store); a ragged chunk's rows are stored directly
            const unsigned char *dls = sm.x + 3 * kBox;
            bf16 *da = a.dvnew + ((size_t)(t0 + (la ? ra : 0)) * a.HV + hv) * kDim + 64 * vb;
            bf16 *db = a.dvnew + ((size_t)(t0 + (lb ? rb : 0)) * a.HV + hv) * kDim + 64 * vb;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int col = c0 + 8 * k + cq;
                const float2 la2 = phi ? make_float2(0.f, 0.f) : epi::get_pair(dls, ra, col);
                const float2 lb2 = phi ? make_float2(0.f, 0.f) : epi::get_pair(dls, rb, col);
                const float va0 = la ? la2.x + ka * p[4 * k] : 0.f, va1 = la ? la2.y + ka * p[4 * k + 1] : 0.f;
                const float vb0 = lb ? lb2.x + kb * p[4 * k + 2] : 0.f, vb1 = lb ? lb2.y + kb * p[4 * k + 3] : 0.f;
                if (!pre && L < 64) {
                    if (la && in_range(da + col - a.dvnew, 2, n_rows_hv(a), a.status))
                        *reinterpret_cast<uint32_t *>(da + col) = pack_bf2(va0, va1);
                    if (lb && in_range(db + col - a.dvnew, 2, n_rows_hv(a), a.status))
                        *reinterpret_cast<uint32_t *>(db + col) = pack_bf2(vb0, vb1);
                }
                epi::put_pair(sm.a_dv, ra, col, va0, va1);
                epi::put_pair(sm.a_dv, rb, col, vb0, vb1);
            }
        }
        if (tid == kPdIssuer) tma_store_wait_read();  // dh_c has been read out of a_ds
        const bool gy = mbar_wait(&sm.y_bar, par);
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok && gy);  // the dO / dv_loc halves have been read
        if (!ok) break;
        // 4. dh += Q^T (c dO) - w^T dv_new
        if (tid == 0) {
            tc_fence_after();
            const uint32_t ado = smem_u32(sm.a_do), adv = smem_u32(sm.a_dv);
            const uint32_t qs = smem_u32(sm.y), ws = smem_u32(sm.y + 2 * kBox);
            if (!phi)
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tbase, sdesc(qs + s * 2048, kBox, 1024), sdesc(ado + s * 2048, kBox, 1024), idS, true);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tbase, sdesc(ws + s * 32, 16, 1024), sdesc(adv + s * 2048, kBox, 1024), idW, true);
            mma_commit(&sm.mma_bar);
            if (!pre && L == 64) {  // this value half's dv_new rows, from the operand tile
                tma_store_3d(&maps.dvn, 64 * vb, hv, t0, sm.a_dv);
                tma_store_commit();
            }
        }
        // the next chunk's dO / dv_loc halves (read by step 3) and the L2 prefetch a step
        // further, from warp 1 while thread 0 issues step 4: one thread issuing all of it
        // reached step 4's wait late
        if (i + 1 < nch && !phi) {
            if (tid == 32) issue_xd(maps, sm, step_t0(i + 1), hv, vb);
            ++xd_issued;
        }
        if (tid == 32 && i + 2 < nch) prefetch_chunk(maps, a, step_c(i + 2), step_t0(i + 2), h, hv, vb, !phi);
        ok = mbar_wait(&sm.mma_bar, phase) && ok;
        phase ^= 1;
        tc_fence_after();
        if (tid == 0 && ok && i + 1 < nch) {  // Q and w are free once step 4 has finished
            issue_y(maps, sm, a, step_c(i + 1), step_t0(i + 1), h, hv);
            ++y_issued;
        }
    }
    ok = __syncthreads_and(ok);
    if (ok && to_final && a.dh0 && in_range(sbase, 32, n_states(a), a.status)) {
        float r[32];
        tmem_ld32(tS, r);
        tmem_ld_wait();
        float4 *dst = reinterpret_cast<float4 *>(a.dh0 + sbase);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
    if (ok && pass == 1 && !to_final &&
        in_range(send - a.seg_end, 32, (long long)a.N * (a.seg_max - 1) * a.HV * kDim * 2 * kDim, a.status)) {
        // a segment's end state (dh columns, and Psi in a pre-scan)
        float r[32];
        tmem_ld32(tS, r);
        tmem_ld_wait();
        float4 *dst = reinterpret_cast<float4 *>(send);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
    if (tid == 0 || tid == kPdIssuer) tma_store_wait_all();
    if (!ok && tid == 0) {
        if (a.status) atomicOr(a.status, 2);
        // drain the loads still in flight (bounded) before leaving
        if (xk_issued > 0) mbar_wait(&sm.xk_bar, (xk_issued - 1) & 1, kDrainLimitNs);
        if (xd_issued > 0) mbar_wait(&sm.xd_bar, (xd_issued - 1) & 1, kDrainLimitNs);
        if (y_issued > 0) mbar_wait(&sm.y_bar, (y_issued - 1) & 1, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 128);
}

}  // namespace

cudaError_t launch_bstate_tc(const ChunkArgs &a, cudaStream_t s) {
    BStateMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 128 * 2;
    if (a.T > 0 && (!encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
                    !encode_rows_bf16(&m.q, a.q, a.H, a.T, rowb, rowb * a.H, 64) ||
                    !encode_rows_bf16(&m.w, a.w, 1, (uint64_t)a.num_chunks * a.HV * kDim, 128, 128, 128,
                                      kChunk) ||
                    !encode_rows_bf16(&m.dO, a.d_o, a.HV, a.T, rowb, rowb * a.HV, 64) ||
                    !encode_rows_bf16(&m.dl, a.dvloc, a.HV, a.T, rowb, rowb * a.HV, 64) ||
                    !encode_rows_bf16(&m.dhc, a.dhc, 1, (uint64_t)a.num_chunks * a.HV * 128, rowb,
                                      rowb, 128) ||
                    !encode_rows_bf16(&m.dvn, a.dvnew, a.HV, a.T, rowb, rowb * a.HV, 64)))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(BStateSmem) + 1024;
    static_assert(2 * (sizeof(BStateSmem) + 2048) <= 233472, "two CTAs per SM");
    cudaError_t e = cudaSuccess;
    for (const void *f : {(const void *)k_bstate_tc<0>, (const void *)k_bstate_tc<1>, (const void *)k_bstate_tc<2>})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
    if (a.seg_len == 0) {
        TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
        k_bstate_tc<0><<<dim3(2 * a.HV, a.N), kThr, smem, s>>>(a, m);
        return cudaGetLastError();
    }
    const unsigned ny = (unsigned)a.N * (unsigned)(a.seg_max - 1);
    {
        TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
        k_bstate_tc<1><<<dim3(4 * a.HV, ny), kThr, smem, s>>>(a, m);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_seg_stitch(a, s)) != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_BSTATE, s);
    k_bstate_tc<2><<<dim3(2 * a.HV, ny), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
