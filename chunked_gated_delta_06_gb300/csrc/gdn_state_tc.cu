// gdn_state_tc.cu -- forward inter-chunk state scan on the tensor cores.
//
// The chunks of one sequence are walked in order ("cake_gdn: deterministic
// chunked GDN training kernels", Summary: fp32 running state across chunks,
// per-chunk h stored in bf16).  The value columns of the state never mix
// (v_new[:, v] and h[:, v] depend only on column v), so one CTA owns one
// (sequence, value head, value half): h[k][v'] for the 64 columns v' = 64 vb ..
// 64 vb + 63, as an fp32 accumulator in TMEM (lane k, 64 columns); its 256
// threads are two warpgroups that split the columns of every pass.
// Per chunk (L <= 64 tokens from t0, G the chunk-local cumsum of g, G_L its last
// value):
//   1. thread k writes row k of h as bf16 to shared memory (MMA operand; one TMA
//      store copies it to h_c[chunk][hv][k][v']), and e^{G_L} h back to TMEM;
//   2. P[t][v'] = sum_k w[t][k] h[k][v']          (tcgen05, M=64 N=64 K=128; w
//      comes as the chunk's w^T tile [k][t] and is read MN-major)
//   3. the result is read as 16x256b fragments (two token rows and eight columns
//      per lane); v_new[t][v'] = u - P goes to HBM (bf16), and
//      A_V[t][v'] = v_new e^{G_L - G_t} / r_k,t to shared memory (bf16);
//   4. h[k][v'] += sum_t K[t][k] A_V[t][v']        (tcgen05, M=128 N=64 K=64; the
//      raw key tile is read MN-major)
// which is h <- e^{G_L} h + (diag(e^{G_L-G}) Khat)^T v_new with Khat =
// diag(1 / r_k) K.  w^T, K, this half of u^T and the chunk's scalar record
// (e^{G_L - G_t} / r_k,t and e^{G_L}, written by the WY pass) stream in two chunks ahead,
// and a chunk costs two block barriers.  Two CTAs
// share an SM.  Every wait is bounded; a timeout sets status bit 2 and the CTA
// unwinds.  In paged-prefill mode the initial state comes from, and the final
// state goes back to, a slot of the decode state pool [slots, HV, V, K] (the
// layout "Replace Qwen3.5 FLA paths with Attention Gym" keeps shared between
// prefill and decode), read and written transposed in place.
#include <string.h>

#include "gdn_epi.cuh"
#include "gdn_kernels.h"
#include "gdn_tma.h"
#include "gdn_umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThr = 256;
constexpr uint32_t kBox = 64 * 128;             // one 64-row x 128-byte SW128 box
constexpr uint32_t kStageBytes = 5 * kBox;      // w^T (128 rows: 2 boxes), K (2), u^T half (1)

struct StateSmem {
    // 1024-byte aligned operand tiles first
    unsigned char a_s[128 * 128];       // h bf16 [k][v']: 128 rows x 128 B
    unsigned char a_v[64 * 128];        // A_V bf16 [t][v']: 64 rows x 128 B
    unsigned char stage[2][kStageBytes];
    ScRec sc[2];                        // the stages' scalar records (kc = coef_t, egl)
    uint64_t tma_bar[2];
    uint64_t mma_bar;
    uint32_t tmem_base;
};

struct StateMaps {
    CUtensorMap w, k, u, hc;
    CUtensorMap vn;   // v_new [T][HV][128]: a full chunk's rows of this value half, stored by TMA
};

// Chunk c (tokens from t0): its w^T tile [k][t] (128 rows), K, and (unless the columns
// are a transition's, whose u is zero) this half of its u^T tile [v'][t] (64 rows)
__device__ __forceinline__ void issue_stage(const StateMaps &m, StateSmem &sm, const ChunkArgs &a, int st,
                                            int c, int t0, int h, int hv, int vb, bool with_u) {
    unsigned char *b = sm.stage[st];
    const int row = (c * a.HV + hv) * kDim;
    mbar_arrive_expect_tx(&sm.tma_bar[st], (with_u ? kStageBytes : kStageBytes - kBox) + (uint32_t)sizeof(ScRec));
    bulk_load(&sm.sc[st], a.sc + ((size_t)c * a.HV + hv) * kScRec, sizeof(ScRec), &sm.tma_bar[st]);
    tma_load_3d(b + 0 * kBox, &m.w, 0, 0, row, &sm.tma_bar[st]);
    tma_load_3d(b + 2 * kBox, &m.k, 0, h, t0, &sm.tma_bar[st]);
    tma_load_3d(b + 3 * kBox, &m.k, 64, h, t0, &sm.tma_bar[st]);
    if (with_u) tma_load_3d(b + 4 * kBox, &m.u, 0, 0, row + 64 * vb, &sm.tma_bar[st]);
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// pass 0: every sequence in one piece.  Segment-parallel scan (sequences cut into
// segments of a.seg_len chunks, S segments): pass 1 runs segment 0 from the
// initial state (all outputs, end state to seg_end) beside the pre-scans of
// segments 1 .. S-2, which start from h = 0 with the transition columns
// [h | Phi] (Phi from the identity, u = 0 there) and store only their end state;
// k_seg_stitch turns those into the start states of segments 1 .. S-1; pass 2
// re-scans those segments from them with every output.
template <int pass>
__global__ void __launch_bounds__(kThr, 2)
    k_state_tc(const ChunkArgs a, const __grid_constant__ StateMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    StateSmem &sm = smem_struct<StateSmem>(smem_raw);
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
    const int nseq = max(ce - cb, 0);              // chunks of the sequence
    const int S = pass ? max(1, (nseq + a.seg_len - 1) / a.seg_len) : 1;
    const int sg = pass == 2 ? blockIdx.y % nsy + 1 : (pass ? blockIdx.y % nsy : 0);
    if (pass == 1 && !(S == 1 ? (sg == 0 && !phi) : (sg == 0 ? !phi : sg <= S - 2))) return;
    if (pass == 2 && !(S >= 2 && sg <= S - 1)) return;
    const bool from_input = sg == 0;               // h0 / pool slot (else zero or seg_start)
    const bool pre = pass == 1 && sg >= 1;         // pre-scan: no per-chunk outputs
    const bool to_final = pass == 0 || (pass == 1 && S == 1) || (pass == 2 && sg == S - 1);
    const int jb = pass ? sg * a.seg_len : 0;      // first chunk of the segment
    const int nch = pass ? max(0, min(a.seg_len, nseq - jb)) : nseq;
    const int grp = warp >> 2, sub = warp & 3;
    const int kr = sub * 32 + lane;     // state row (TMEM lane) of the state pass
    const int c0 = 32 * grp;            // this warpgroup's 32 of the 64 columns
    // the sequence's chunks are consecutive 64-token blocks of [ts0, ts1)
    const int ts0 = nseq > 0 ? a.chunk_start[cb] : 0;
    const int ts1 = nseq > 0 ? a.chunk_start[ce - 1] + a.chunk_len[ce - 1] : 0;
    auto chunk_t0 = [&](int j) { return ts0 + 64 * (jb + j); };
    auto chunk_len = [&](int j) { return min(64, ts1 - chunk_t0(j)); };

    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 128);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sm.tma_bar[0], 1);
        mbar_init(&sm.tma_bar[1], 1);
        mbar_init(&sm.mma_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;
    const uint32_t t_row = tbase + ((uint32_t)(sub * 32) << 16);  // this warp's lanes
    const uint32_t tH = t_row + c0, tP = t_row + 64 + c0;          // this warpgroup's columns

    if (tid == 0)
        for (int i = 0; i < 2 && i < nch; ++i) issue_stage(maps, sm, a, i, cb + jb + i, chunk_t0(i), h, hv, vb, !phi);
    // h <- h0[n][hv][k][v'] (row kr, this warpgroup's 32 columns), or in paged mode
    // the transpose of pool slot S[v'][k] (lanes are consecutive k: coalesced per v')
    const size_t sbase = ((size_t)n * a.HV + hv) * kDim * kDim + (size_t)kr * kDim + 64 * vb + c0;
    int slot = 0;
    bool resume = false;
    if (a.pool) {
        slot = a.pool_idx[n];
        if (slot >= a.num_slots) {
            if (a.pool_status && tid == 0) *a.pool_status = 1;
            slot = 0;
        }
        if (slot < 0) slot = 0;
        resume = slot > 0 && (!a.pool_resume || a.pool_resume[n] != 0);
    }
    float *pslot = a.pool ? a.pool + (((size_t)slot * a.HV + hv) * kDim + 64 * vb + c0) * kDim + kr
                          : nullptr;  // S[v'][kr] of this thread's first column
    auto pool_in = [&](const float *ps) {  // the 32 columns of S[.][kr] this thread reads / writes
        return in_range(ps - a.pool, 31 * kDim + 1, (long long)a.num_slots * a.HV * kDim * kDim, a.status);
    };
    // segment buffers: seg_end[n][s][hv][k][256] (h | Phi), seg_start[n][s-1][hv][k][128]
    const size_t seg_row = (size_t)kr * (2 * kDim) + (phi ? kDim : 0) + 64 * vb + c0;
    float *send = pass == 1 ? a.seg_end + (((size_t)n * (a.seg_max - 1) + sg) * a.HV + hv) * kDim * 2 * kDim +
                                  seg_row
                            : nullptr;
    {
        float r[32];
        if (pre) {  // h from zero; Phi from the identity (row k, column k' = 64 vb + c0 + j)
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = (phi && kr == 64 * vb + c0 + j) ? 1.f : 0.f;
        } else if (!from_input) {
            const size_t off = (((size_t)n * (a.seg_max - 1) + sg - 1) * a.HV + hv) * kDim * kDim +
                               (size_t)kr * kDim + 64 * vb + c0;
            const float4 *src = reinterpret_cast<const float4 *>(a.seg_start + off);
            const bool in = in_range(off, 32, (long long)a.N * (a.seg_max - 1) * a.HV * kDim * kDim, a.status);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = in ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
        } else if (a.pool) {
            const bool in = !resume || pool_in(pslot);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = resume && in ? pslot[(size_t)j * kDim] : 0.f;
        } else if (a.h0 && in_range(sbase, 32, n_states(a), a.status)) {
            const float4 *src = reinterpret_cast<const float4 *>(a.h0 + sbase);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = src[q];
                r[4 * q] = x.x; r[4 * q + 1] = x.y; r[4 * q + 2] = x.z; r[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0.f;
        }
        tmem_st32(tH, r);
        tmem_st_wait();
    }
    __syncthreads();
    const uint32_t idP = idesc_bf16(64, 64, 1, 1);    // P = w h       (w^T and h MN-major)
    const uint32_t idS = idesc_bf16(128, 64, 1, 1);   // h += K^T A_V  (both MN-major)
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
        const int c = cb + jb + i, st = i & 1;
        const int t0 = chunk_t0(i), L = chunk_len(i);
        // the chunk's tiles and scalar record (e^{G_L} is needed right below)
        const bool got = mbar_wait(&sm.tma_bar[st], (i >> 1) & 1);
        const float egl = sm.sc[st].egl;
        // 1. h -> bf16 operand (copied to h_c by TMA below), then h <- e^{G_L} h
        {
            float r[32];
            tmem_ld32(tH, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(sm.a_s + sw128_off(kr, c0 + 8 * q)) =
                    make_uint4(pack_bf2(r[8 * q], r[8 * q + 1]), pack_bf2(r[8 * q + 2], r[8 * q + 3]),
                               pack_bf2(r[8 * q + 4], r[8 * q + 5]), pack_bf2(r[8 * q + 6], r[8 * q + 7]));
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] *= egl;
            tmem_st32(tH, r);
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok && got);
        if (!ok) break;
        // 2. P = w h
        if (tid == 0) {
            tc_fence_after();
            const uint32_t as = smem_u32(sm.a_s), ws = smem_u32(sm.stage[st]);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16(tbase + 64, sdesc(ws + s * 2048, kBox, 1024), sdesc(as + s * 2048, kBox, 1024), idP,
                         s > 0);
            mma_commit(&sm.mma_bar);
            if (!pre) {
                tma_store_3d(&maps.hc, 64 * vb, 0, (c * a.HV + hv) * 128, sm.a_s);  // h_c rows (k)
                tma_store_commit();
            }
        }
        ok = mbar_wait(&sm.mma_bar, phase) && ok;
        phase ^= 1;
        tc_fence_after();
        // 3. v_new = u - P on 16x256b fragments: rows ra, ra + 8, this warpgroup's
        //    columns c0 + 8k + cq + {0, 1}
        {
            float p[16];
            epi::tmem_ld16x256_x4(tP, p);
            tmem_ld_wait();
            const int ra = sub * 16 + (lane >> 2), rb = ra + 8, cq = 2 * (lane & 3);
            const bool la = ra < L, lb = rb < L;
            const float cfa = sm.sc[st].kc[ra], cfb = sm.sc[st].kc[rb];
            const unsigned char *us = sm.stage[st] + 4 * kBox;   // u^T [v'][t]
            auto u2 = [&](int t, int v) {  // u[t][v], u[t][v + 1]
                const bf16 *e0 = reinterpret_cast<const bf16 *>(us + sw128_off(v, t));
                const bf16 *e1 = reinterpret_cast<const bf16 *>(us + sw128_off(v + 1, t));
                return make_float2(__bfloat162float(*e0), __bfloat162float(*e1));
            };
            bf16 *da = a.vnew + ((size_t)(t0 + (la ? ra : 0)) * a.HV + hv) * kDim + 64 * vb;
            bf16 *db = a.vnew + ((size_t)(t0 + (lb ? rb : 0)) * a.HV + hv) * kDim + 64 * vb;
            // a full chunk's v_new rows are staged over this stage's w^T tile (read by the
            // product above) for one TMA store; a ragged chunk's rows are stored directly
            unsigned char *vstg = sm.stage[st];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int col = c0 + 8 * k + cq;
                const float2 ua = phi ? make_float2(0.f, 0.f) : u2(ra, col);
                const float2 ub = phi ? make_float2(0.f, 0.f) : u2(rb, col);
                const float va0 = la ? ua.x - p[4 * k] : 0.f, va1 = la ? ua.y - p[4 * k + 1] : 0.f;
                const float vb0 = lb ? ub.x - p[4 * k + 2] : 0.f, vb1 = lb ? ub.y - p[4 * k + 3] : 0.f;
                if (!pre && L == 64) {
                    epi::put_pair(vstg, ra, col, va0, va1);
                    epi::put_pair(vstg, rb, col, vb0, vb1);
                } else if (!pre) {
                    if (la && in_range(da + col - a.vnew, 2, n_rows_hv(a), a.status))
                        *reinterpret_cast<uint32_t *>(da + col) = pack_bf2(va0, va1);
                    if (lb && in_range(db + col - a.vnew, 2, n_rows_hv(a), a.status))
                        *reinterpret_cast<uint32_t *>(db + col) = pack_bf2(vb0, vb1);
                }
                epi::put_pair(sm.a_v, ra, col, va0 * cfa, va1 * cfa);
                epi::put_pair(sm.a_v, rb, col, vb0 * cfb, vb1 * cfb);
            }
        }
        if (tid == 0) tma_store_wait_read();  // h_c has been read out of a_s
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        // 4. h += K^T A_V
        if (tid == 0) {
            tc_fence_after();
            const uint32_t av = smem_u32(sm.a_v), ks = smem_u32(sm.stage[st] + 2 * kBox);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tbase, sdesc(ks + s * 2048, kBox, 1024), sdesc(av + s * 2048, kBox, 1024), idS, true);
            mma_commit(&sm.mma_bar);
            if (!pre && L == 64) {  // the staged v_new rows of this value half
                tma_store_3d(&maps.vn, 64 * vb, hv, t0, sm.stage[st]);
                tma_store_commit();
            }
        }
        ok = mbar_wait(&sm.mma_bar, phase) && ok;
        phase ^= 1;
        tc_fence_after();
        if (tid == 0 && ok && i + 2 < nch) {
            tma_store_wait_read();  // the staged v_new rows have left the stage
            issue_stage(maps, sm, a, st, c + 2, chunk_t0(i + 2), h, hv, vb, !phi);
        }
    }
    ok = __syncthreads_and(ok);
    if (ok && to_final && a.ht && in_range(sbase, 32, n_states(a), a.status)) {
        float r[32];
        tmem_ld32(tH, r);
        tmem_ld_wait();
        float4 *dst = reinterpret_cast<float4 *>(a.ht + sbase);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
    if (ok && to_final && a.pool && slot > 0 && pool_in(pslot)) {  // final state back into the slot, transposed
        float r[32];
        tmem_ld32(tH, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) pslot[(size_t)j * kDim] = r[j];
    }
    if (ok && pass == 1 && !to_final &&
        in_range(send - a.seg_end, 32, (long long)a.N * (a.seg_max - 1) * a.HV * kDim * 2 * kDim, a.status)) {
        // a segment's end state (h columns, and Phi in a pre-scan)
        float r[32];
        tmem_ld32(tH, r);
        tmem_ld_wait();
        float4 *dst = reinterpret_cast<float4 *>(send);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
    if (tid == 0) tma_store_wait_all();
    if (!ok && tid == 0) {
        // drain outstanding TMA copies (bounded) before leaving
        if (a.status) atomicOr(a.status, 2);
        mbar_wait(&sm.tma_bar[0], 0, kDrainLimitNs);
        mbar_wait(&sm.tma_bar[1], 0, kDrainLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 128);
}

// Start states of segments 1 .. S-1 of every split sequence: H_1 = end of segment 0,
// H_{s+1} = Phi_s H_s + beta_s (Phi_s, beta_s from the pre-scan of segment s).  The
// reverse scan uses the same records in reverse segment order (Psi_rho, beta'_rho).
// grid (8 HV, N): 16 value columns of one (sequence, value head) per CTA; thread t
// owns row k = t / 2 and 8 columns; sums run over k' in order (fp32).
__global__ void __launch_bounds__(256) k_seg_stitch(const ChunkArgs a) {
    const int hv = blockIdx.x >> 3, v0 = 16 * (blockIdx.x & 7), n = blockIdx.y;
    const int nseq = max(0, min(a.seq_chunk_off[n + 1], a.num_chunks) - a.seq_chunk_off[n]);
    const int S = max(1, (nseq + a.seg_len - 1) / a.seg_len);
    if (S < 2 || !in_range(S - 1, 1, a.seg_max, a.status)) return;
    __shared__ float H[kDim][16];
    const int t = threadIdx.x, k = t >> 1, cc = 8 * (t & 1);
    const size_t eh = (size_t)kDim * 2 * kDim;  // floats of one (segment, head) end record
    auto end_rec = [&](int sg) { return a.seg_end + (((size_t)n * (a.seg_max - 1) + sg) * a.HV + hv) * eh; };
    {
        const float *e0 = end_rec(0) + (size_t)k * 2 * kDim + v0 + cc;
#pragma unroll
        for (int j = 0; j < 8; ++j) H[k][cc + j] = e0[j];
    }
    __syncthreads();
    for (int sg = 1; sg <= S - 1; ++sg) {
        float *dst = a.seg_start + (((size_t)n * (a.seg_max - 1) + sg - 1) * a.HV + hv) * kDim * kDim +
                     (size_t)k * kDim + v0 + cc;
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = H[k][cc + j];
        if (sg == S - 1) break;
        const float *rec = end_rec(sg) + (size_t)k * 2 * kDim;  // row k: beta_s [0, K), Phi_s [K, 2K)
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        for (int k2 = 0; k2 < kDim; k2 += 4) {
            const float4 ph = *reinterpret_cast<const float4 *>(rec + kDim + k2);
            const float pv[4] = {ph.x, ph.y, ph.z, ph.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += pv[u] * H[k2 + u][cc + j];
        }
        __syncthreads();  // every thread has read H
#pragma unroll
        for (int j = 0; j < 8; ++j) H[k][cc + j] = acc[j] + rec[v0 + cc + j];
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_seg_stitch(const ChunkArgs &a, cudaStream_t s) {
    TimerScope ts(a.timer, GDN_KERNEL_SEG_STITCH, s);
    k_seg_stitch<<<dim3(8 * a.HV, a.N), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_state_tc(const ChunkArgs &a, cudaStream_t s) {
    StateMaps m;
    memset(&m, 0, sizeof(m));
    const uint64_t rowb = 128 * 2;
    // w^T / u^T: rows of one chunk's 64 tokens (128 bytes), [C][HV][128] of them
    const uint64_t wrows = (uint64_t)a.num_chunks * a.HV * kDim;
    if (a.T > 0 && (!encode_rows_bf16(&m.w, a.w, 1, wrows, 128, 128, 128, kChunk) ||
        !encode_rows_bf16(&m.k, a.k, a.H, a.T, rowb, rowb * a.H, 64) ||
        !encode_rows_bf16(&m.u, a.u, 1, wrows, 128, 128, 64, kChunk) ||
        !encode_rows_bf16(&m.hc, a.hc, 1, (uint64_t)a.num_chunks * a.HV * 128, rowb, rowb, 128) ||
        !encode_rows_bf16(&m.vn, a.vnew, a.HV, a.T, rowb, rowb * a.HV, 64)))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(StateSmem) + 1024;
    static_assert(2 * (sizeof(StateSmem) + 2048) <= 233472, "two CTAs per SM");
    cudaError_t e = cudaSuccess;
    for (const void *f : {(const void *)k_state_tc<0>, (const void *)k_state_tc<1>, (const void *)k_state_tc<2>})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
            cudaSuccess)
            return e;
    if (a.seg_len == 0) {
        TimerScope ts(a.timer, GDN_KERNEL_STATE, s);
        k_state_tc<0><<<dim3(2 * a.HV, a.N), kThr, smem, s>>>(a, m);
        return cudaGetLastError();
    }
    const unsigned ny = (unsigned)a.N * (unsigned)(a.seg_max - 1);
    {
        TimerScope ts(a.timer, GDN_KERNEL_STATE, s);
        k_state_tc<1><<<dim3(4 * a.HV, ny), kThr, smem, s>>>(a, m);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_seg_stitch(a, s)) != cudaSuccess) return e;
    TimerScope ts(a.timer, GDN_KERNEL_STATE, s);
    k_state_tc<2><<<dim3(2 * a.HV, ny), kThr, smem, s>>>(a, m);
    return cudaGetLastError();
}

}  // namespace gdn
