// gdn_api.cu -- the extern "C" entry points declared in include/gdn.h: host-side
// validation (before any launch), carving of the caller's saved / workspace
// buffers, and the launch order of the chunk and decode kernels.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/gdn.h"
#include "gdn_kernels.h"

namespace {

using gdn::bf16;
constexpr size_t kAlign = 256;

// Sequential sub-allocator over a caller buffer; with base == nullptr it only counts.
struct Carver {
    char *base;
    size_t off = 0;
    explicit Carver(void *b) : base(static_cast<char *>(b)) {}
    template <typename T>
    T *take(size_t count) {
        off = (off + kAlign - 1) / kAlign * kAlign;
        T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
    size_t used() const { return (off + kAlign - 1) / kAlign * kAlign; }
};

struct Dims {
    int N, T, H, HV, C;  // C = chunk count
    int longest;         // chunks of the longest sequence
    float scale;
    int beta_f32;        // beta / dbeta are fp32 (else bf16); fused-gating calls need bf16
    int seg_len, seg_max;  // segment-parallel forward scan (seg_len 0: not split)
};

// Plan of the forward state scan.  A scan CTA walks the chunks of one (sequence,
// value head, value half) one after another, so a few long sequences leave most of
// the GPU idle.  Cutting every sequence into segments of L chunks lets segment 0
// and the pre-scans of segments 1 .. S-2 run at once (pass 1; a pre-scan carries
// the 128 transition columns as well, so it is two CTAs more per value head), then
// segments 1 .. S-1 re-scan from their stitched start states (pass 2).  The model
// counts scan steps: a pass takes max(its longest CTA, its CTA-steps / the number of
// resident scan CTAs), with 2 per SM on 152 SMs; the stitch costs half a step per
// segment plus three steps for the extra launches.  The plan is a pure function of
// the problem (the same bits on every device): a split is taken only when the model
// gains at least 20 % and its buffers stay under 1 GiB.
// The problem's scan_segment_chunks overrides the model: -1 never splits, L > 0
// cuts every sequence into segments of L chunks whenever that gives 3 or more.
void plan_segments(const gdn_problem *p, Dims *d) {
    d->seg_len = 0;
    d->seg_max = 1;
    const double slots = 2.0 * 152.0;
    const int N = d->N, HV = d->HV;
    int longest = 0;
    double total = 0.0;
    for (int n = 0; n < N; ++n) {
        const int c = (int)(((int64_t)p->cu_seqlens_host[n + 1] - p->cu_seqlens_host[n] + gdn::kChunk - 1) /
                            gdn::kChunk);
        longest = c > longest ? c : longest;
        total += c;
    }
    if (p->scan_segment_chunks < 0) return;
    if (p->scan_segment_chunks > 0) {
        const int L = p->scan_segment_chunks;
        const int smax = (longest + L - 1) / L;
        if (smax >= 3 && smax <= 4096) {
            d->seg_len = L;
            d->seg_max = smax;
        }
        return;
    }
    if (longest < 24) return;
    const double t0 = fmax((double)longest, 2.0 * HV * total / slots);
    double best = 0.8 * t0;
    static const int cand[] = {8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512};
    for (int L : cand) {
        int smax = 1;
        double w1 = 0.0, w2 = 0.0;
        for (int n = 0; n < N; ++n) {
            const int c = (int)(((int64_t)p->cu_seqlens_host[n + 1] - p->cu_seqlens_host[n] + gdn::kChunk - 1) /
                                gdn::kChunk);
            const int S = c > 0 ? (c + L - 1) / L : 1;
            smax = S > smax ? S : smax;
            if (S == 1) {
                w1 += 2.0 * HV * c;
            } else {
                w1 += 2.0 * HV * L + 4.0 * HV * L * (S - 2);
                w2 += 2.0 * HV * (c - L);
            }
        }
        if (smax < 3 || smax > 64) continue;
        const double bytes = (double)N * (smax - 1) * HV * (3.0 * gdn::kDim * gdn::kDim * 4.0);
        if (bytes > 1073741824.0) continue;
        const double chain1 = fmin((double)L, (double)longest);
        const double t = fmax(chain1, w1 / slots) + fmax((double)L, w2 / slots) + 0.5 * (smax - 2) + 3.0;
        if (t < best) {
            best = t;
            d->seg_len = L;
            d->seg_max = smax;
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

gdn_status check_problem(const gdn_problem *p, Dims *d) {
    if (!p) return GDN_ERR_INVALID_ARG;
    if (p->num_seqs < 1 || p->total_tokens < 0 || p->total_tokens > 0x7fffffffLL)
        return GDN_ERR_INVALID_ARG;
    if (p->num_k_heads < 1 || p->num_v_heads < 1 || p->num_k_heads > 65535 ||
        p->num_v_heads > 65535)
        return GDN_ERR_INVALID_ARG;
    if (p->head_dim_k != 128 || p->head_dim_v != 128) return GDN_ERR_UNSUPPORTED;
    if (p->num_v_heads % p->num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
    if (p->beta_dtype != GDN_DTYPE_BF16 && p->beta_dtype != GDN_DTYPE_F32) return GDN_ERR_INVALID_ARG;
    if (p->scan_segment_chunks < -1) return GDN_ERR_INVALID_ARG;
    if (!aligned_to(p->device_status, 4)) return GDN_ERR_INVALID_ARG;
    if (!p->cu_seqlens_host || !p->cu_seqlens_dev) return GDN_ERR_INVALID_ARG;
    const int32_t *cu = p->cu_seqlens_host;
    if (cu[0] != 0 || (int64_t)cu[p->num_seqs] != p->total_tokens) return GDN_ERR_INVALID_ARG;
    int64_t chunks = 0, longest = 0;
    for (int n = 0; n < p->num_seqs; ++n) {
        if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARG;
        const int64_t c = ((int64_t)cu[n + 1] - cu[n] + gdn::kChunk - 1) / gdn::kChunk;
        chunks += c;
        longest = c > longest ? c : longest;
    }
    d->longest = (int)longest;
    d->N = p->num_seqs;
    d->T = (int)p->total_tokens;
    d->H = p->num_k_heads;
    d->HV = p->num_v_heads;
    d->C = (int)chunks;
    d->scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->head_dim_k);
    d->beta_f32 = p->beta_dtype == GDN_DTYPE_F32;
    plan_segments(p, d);
    return GDN_OK;
}

// The tensors gdn_chunk_fwd keeps for gdn_chunk_bwd, in a fixed order.
void carve_saved(Carver &cv, const Dims &d, gdn::ChunkArgs &a) {
    const size_t D = gdn::kDim;
    a.hc = cv.take<bf16>((size_t)d.C * d.HV * D * D);
    a.vnew = cv.take<bf16>((size_t)d.T * d.HV * D);
    a.w = cv.take<bf16>((size_t)d.C * d.HV * D * gdn::kChunk);
    a.Tm = cv.take<bf16>((size_t)d.C * d.HV * gdn::kChunk * gdn::kChunk);
    a.rq = cv.take<float>((size_t)d.T * d.H);
    a.rk = cv.take<float>((size_t)d.T * d.H);
    a.G = cv.take<float>((size_t)d.T * d.HV);
    a.sc = cv.take<float>((size_t)d.C * d.HV * gdn::kScRec);
}

void carve_table(Carver &cv, const Dims &d, gdn::ChunkArgs &a) {
    a.seq_chunk_off = cv.take<int>((size_t)d.N + 1);
    a.chunk_start = cv.take<int>((size_t)d.C);
    a.chunk_len = cv.take<int>((size_t)d.C);
    a.seq_order = cv.take<int>((size_t)d.N);
}

// Segment buffers of a split forward scan (none when the scan is not split).
void carve_segments(Carver &cv, const Dims &d, gdn::ChunkArgs &a) {
    a.seg_len = d.seg_len;
    a.seg_max = d.seg_max;
    if (d.seg_len == 0) return;
    const size_t recs = (size_t)d.N * (d.seg_max - 1) * d.HV;
    a.seg_end = cv.take<float>(recs * gdn::kDim * 2 * gdn::kDim);
    a.seg_start = cv.take<float>(recs * gdn::kDim * gdn::kDim);
}

void carve_fwd_ws(Carver &cv, const Dims &d, gdn::ChunkArgs &a, bool with_saved) {
    carve_table(cv, d, a);
    a.u = cv.take<bf16>((size_t)d.C * d.HV * gdn::kDim * gdn::kChunk);
    carve_segments(cv, d, a);
    if (with_saved) carve_saved(cv, d, a);
}

void carve_bwd_ws(Carver &cv, const Dims &d, gdn::ChunkArgs &a) {
    const size_t D = gdn::kDim;
    carve_table(cv, d, a);
    a.dvloc = cv.take<bf16>((size_t)d.T * d.HV * D);
    a.dvnew = cv.take<bf16>((size_t)d.T * d.HV * D);
    a.dhc = cv.take<bf16>((size_t)d.C * d.HV * D * D);
    a.dW = cv.take<bf16>((size_t)d.T * d.HV * D);
    a.dkpart = cv.take<bf16>((size_t)d.T * d.H * D);
    a.dGp = cv.take<float>((size_t)d.T * d.HV);
    a.gpart = cv.take<float>((size_t)d.C * d.HV * 2);
    carve_segments(cv, d, a);  // the reverse scan's segments (shared with a recomputed forward)
}

size_t saved_bytes(const Dims &d) {
    Carver cv(nullptr);
    gdn::ChunkArgs a{};
    carve_saved(cv, d, a);
    return cv.used();
}

// Workspace of gdn_chunk_fwd (mode 0), gdn_chunk_bwd with a saved buffer (1) and
// gdn_chunk_bwd in recompute-state mode (2: the saved tensors follow the backward
// scratch; the forward's u lives in dv_loc, which the backward writes only after
// the recomputed state scan has read u).
size_t ws_bytes(const Dims &d, int mode) {
    Carver cv(nullptr);
    gdn::ChunkArgs a{};
    if (mode == 0) {
        carve_fwd_ws(cv, d, a, true);
    } else {
        carve_bwd_ws(cv, d, a);
        if (mode == 2) carve_saved(cv, d, a);
    }
    return cv.used();
}

void fill_common(gdn::ChunkArgs &a, const Dims &d, const gdn_problem *p, const void *q,
                 const void *k, const void *v, const float *g, const void *beta,
                 const float *h0) {
    a.N = d.N;
    a.T = d.T;
    a.H = d.H;
    a.HV = d.HV;
    a.num_chunks = d.C;
    a.max_seq_chunks = d.longest;
    a.scale = d.scale;
    a.q = static_cast<const bf16 *>(q);
    a.k = static_cast<const bf16 *>(k);
    a.v = static_cast<const bf16 *>(v);
    a.g = g;
    a.beta = beta;
    a.beta_mode = d.beta_f32 ? 1 : 0;
    a.h0 = h0;
    a.cu_dev = p->cu_seqlens_dev;
    a.status = p->device_status;
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// Fused-gating arguments of the *_gated entry points (all null otherwise).
struct Gate {
    const void *a, *b;             // bf16 [T, HV] (decode: [batch, HV])
    const float *A_log, *dt_bias;  // fp32 [HV]
    void *da, *db;                 // bf16 [T, HV] (backward)
    float *dA_log, *ddt_bias;      // fp32 [HV] (backward)
};

// The gate / beta inputs of a chunk call: g and beta, or the fused gate's a, b,
// A_log and dt_bias (2-byte aligned bf16, 4-byte aligned fp32).
gdn_status check_gate_inputs(const Dims &d, const gdn_problem *p, const float *g, const void *beta,
                             const Gate *gt) {
    if (gt) {
        if (p->beta_dtype != GDN_DTYPE_BF16) return GDN_ERR_INVALID_ARG;  // a and b are bf16
        if (d.T > 0 && (!gt->a || !gt->b)) return GDN_ERR_INVALID_ARG;
        if (!gt->A_log || !gt->dt_bias) return GDN_ERR_INVALID_ARG;
        if (!aligned_to(gt->a, 2) || !aligned_to(gt->b, 2) || !aligned_to(gt->A_log, 4) ||
            !aligned_to(gt->dt_bias, 4))
            return GDN_ERR_INVALID_ARG;
        return GDN_OK;
    }
    if (d.T > 0 && (!g || !beta)) return GDN_ERR_INVALID_ARG;
    if (!aligned_to(g, 4) || !aligned_to(beta, d.beta_f32 ? 4 : 2)) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

void fill_gate(gdn::ChunkArgs &a, const Gate *gt) {
    if (!gt) return;
    a.beta_mode = 2;
    a.ga = static_cast<const bf16 *>(gt->a);
    a.gb = static_cast<const bf16 *>(gt->b);
    a.A_log = gt->A_log;
    a.dt_bias = gt->dt_bias;
}

// Paged-prefill arguments (the initial and final states live in decode-pool slots).
struct Paged {
    float *pool;                 // [num_slots, HV, V, K]
    int32_t num_slots;
    const int32_t *indices;      // device [N]
    const int32_t *resume;       // device [N] or null
    int32_t *status;             // device or null
};

gdn_status chunk_fwd_impl(const gdn_problem *p, const void *q, const void *k, const void *v,
                          const float *g, const void *beta, const Gate *gt,
                          const float *initial_state, void *o, float *final_state, void *saved,
                          void *workspace, size_t ws_size, gdn_stream_t stream,
                          gdn_kernel_timer *timer, const Paged *pg = nullptr) {
    Dims d;
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    if (d.T > 0 && (!q || !k || !v || !o)) return GDN_ERR_INVALID_ARG;
    if ((st = check_gate_inputs(d, p, g, beta, gt)) != GDN_OK) return st;
    if (pg) {
        if (!pg->pool || pg->num_slots < 1 || !pg->indices || !aligned16(pg->pool) ||
            !aligned_to(pg->indices, 4) || !aligned_to(pg->resume, 4) || !aligned_to(pg->status, 4))
            return GDN_ERR_INVALID_ARG;
        if ((int64_t)pg->num_slots * d.HV > (int64_t)1 << 40) return GDN_ERR_INVALID_ARG;
    }
    const void *ptrs[] = {q, k, v, initial_state, o, final_state, saved, workspace};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
        (saved && (reinterpret_cast<uintptr_t>(saved) % kAlign) != 0))
        return GDN_ERR_INVALID_ARG;
    if (ws_size < ws_bytes(d, 0)) return GDN_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    gdn::ChunkArgs a{};
    fill_common(a, d, p, q, k, v, g, beta, initial_state);
    fill_gate(a, gt);
    a.timer = timer;
    a.o = static_cast<bf16 *>(o);
    a.ht = final_state;
    if (pg) {
        a.pool = pg->pool;
        a.num_slots = pg->num_slots;
        a.pool_idx = pg->indices;
        a.pool_resume = pg->resume;
        a.pool_status = pg->status;
    }
    Carver wc(workspace);
    carve_fwd_ws(wc, d, a, saved == nullptr);
    if (saved) {
        Carver sc(saved);
        carve_saved(sc, d, a);
    }
    cudaError_t e;
    if ((e = gdn::launch_plan(a, s)) != cudaSuccess) return cuda_status(e);
    if ((e = gdn::launch_prep(a, s)) != cudaSuccess) return cuda_status(e);
    if ((e = gdn::launch_fwd_chunks(a, s)) != cudaSuccess) return cuda_status(e);
    return GDN_OK;
}

gdn_status chunk_bwd_impl(const gdn_problem *p, const void *q, const void *k, const void *v,
                          const float *g, const void *beta, const Gate *gt,
                          const float *initial_state, const void *saved, const void *d_o,
                          const float *d_final_state, void *dq, void *dk, void *dv, float *dg,
                          void *dbeta, float *dh0, void *workspace, size_t ws_size,
                          gdn_stream_t stream, gdn_kernel_timer *timer) {
    Dims d;
    gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    const bool recompute = !saved && saved_bytes(d) > 0;  // T == 0 saves nothing
    if (d.T > 0 && (!q || !k || !v || !d_o || !dq || !dk || !dv)) return GDN_ERR_INVALID_ARG;
    if ((st = check_gate_inputs(d, p, g, beta, gt)) != GDN_OK) return st;
    if (gt) {
        if (d.T > 0 && (!gt->da || !gt->db)) return GDN_ERR_INVALID_ARG;
        if (!gt->dA_log || !gt->ddt_bias) return GDN_ERR_INVALID_ARG;
        if (!aligned_to(gt->da, 2) || !aligned_to(gt->db, 2) || !aligned_to(gt->dA_log, 4) ||
            !aligned_to(gt->ddt_bias, 4))
            return GDN_ERR_INVALID_ARG;
    } else {
        if (d.T > 0 && (!dg || !dbeta)) return GDN_ERR_INVALID_ARG;
        if (!aligned_to(dg, 4) || !aligned_to(dbeta, d.beta_f32 ? 4 : 2)) return GDN_ERR_INVALID_ARG;
    }
    const void *ptrs[] = {q, k, v, initial_state, saved, d_o, d_final_state, dq, dk, dv, dh0,
                          workspace};
    for (const void *x : ptrs)
        if (x && !aligned16(x)) return GDN_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
        (reinterpret_cast<uintptr_t>(saved) % kAlign) != 0)
        return GDN_ERR_INVALID_ARG;
    if (ws_size < ws_bytes(d, recompute ? 2 : 1)) return GDN_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    gdn::ChunkArgs a{};
    fill_common(a, d, p, q, k, v, g, beta, initial_state);
    fill_gate(a, gt);
    a.timer = timer;
    Carver wc(workspace);
    carve_bwd_ws(wc, d, a);
    if (recompute) {
        carve_saved(wc, d, a);
        a.u = a.dvloc;  // read by the recomputed state scan before dv_loc is written
    } else {
        Carver sc(const_cast<void *>(saved));
        carve_saved(sc, d, a);
    }
    a.d_o = static_cast<const bf16 *>(d_o);
    a.d_ht = d_final_state;
    a.dq = static_cast<bf16 *>(dq);
    a.dk = static_cast<bf16 *>(dk);
    a.dv = static_cast<bf16 *>(dv);
    a.dh0 = dh0;
    if (gt) {
        a.dbeta = gt->db;
        a.da = static_cast<bf16 *>(gt->da);
        a.dA_log = gt->dA_log;
        a.ddt_bias = gt->ddt_bias;
    } else {
        a.dbeta = dbeta;
        a.dg = dg;
    }
    cudaError_t e;
    if ((e = gdn::launch_plan(a, s)) != cudaSuccess) return cuda_status(e);
    if (recompute) {  // the forward's saved tensors, rebuilt by the forward's own kernels
        if ((e = gdn::launch_prep(a, s)) != cudaSuccess) return cuda_status(e);
        if ((e = gdn::launch_recompute_chunks(a, s)) != cudaSuccess) return cuda_status(e);
    }
    if ((e = gdn::launch_bwd_chunks(a, s)) != cudaSuccess) return cuda_status(e);
    if (gt && (e = gdn::launch_gate_reduce(a, s)) != cudaSuccess) return cuda_status(e);
    return GDN_OK;
}

gdn_status decode_impl(int32_t batch, int32_t num_k_heads, int32_t num_v_heads, int32_t head_dim_k,
                       int32_t head_dim_v, float scale, const void *q, const void *k, const void *v,
                       const float *g, const float *beta, const Gate *gt, float *state_pool,
                       int32_t num_slots, const int32_t *state_indices, void *o,
                       int32_t *device_status, gdn_stream_t stream, gdn_kernel_timer *timer) {
    if (batch < 0 || num_k_heads < 1 || num_v_heads < 1 || num_slots < 1)
        return GDN_ERR_INVALID_ARG;
    if (head_dim_k != 128 || head_dim_v != 128) return GDN_ERR_UNSUPPORTED;
    if (num_v_heads % num_k_heads != 0) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)batch * num_v_heads > 0x7fffffffLL) return GDN_ERR_INVALID_ARG;
    if (batch == 0) return GDN_OK;
    if (!q || !k || !v || !state_pool || !state_indices || !o) return GDN_ERR_INVALID_ARG;
    if (gt) {
        if (!gt->a || !gt->b || !gt->A_log || !gt->dt_bias) return GDN_ERR_INVALID_ARG;
        if (!aligned_to(gt->a, 2) || !aligned_to(gt->b, 2) || !aligned_to(gt->A_log, 4) ||
            !aligned_to(gt->dt_bias, 4))
            return GDN_ERR_INVALID_ARG;
    } else {
        if (!g || !beta || !aligned_to(g, 4) || !aligned_to(beta, 4)) return GDN_ERR_INVALID_ARG;
    }
    if (!aligned16(state_pool)) return GDN_ERR_INVALID_ARG;
    const float s = scale > 0.f ? scale : 1.0f / sqrtf((float)head_dim_k);
    gdn::DecodeGate dg{};
    if (gt) {
        dg.a = static_cast<const bf16 *>(gt->a);
        dg.b = static_cast<const bf16 *>(gt->b);
        dg.A_log = gt->A_log;
        dg.dt_bias = gt->dt_bias;
    }
    cudaError_t e = gdn::launch_decode(
        batch, num_k_heads, num_v_heads, s, static_cast<const bf16 *>(q),
        static_cast<const bf16 *>(k), static_cast<const bf16 *>(v), g, beta, dg, state_pool,
        num_slots, state_indices, static_cast<bf16 *>(o), device_status,
        reinterpret_cast<cudaStream_t>(stream), timer);
    return cuda_status(e);
}

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: invalid argument";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: K and V must be 128 and HV % H == 0";
        case GDN_ERR_WORKSPACE_TOO_SMALL: return "GDN_ERR_WORKSPACE_TOO_SMALL: workspace below the size query";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA launch failed";
    }
    return "unknown gdn_status";
}

size_t gdn_chunk_saved_bytes(const gdn_problem *p) {
    Dims d;
    if (check_problem(p, &d) != GDN_OK) return 0;
    return saved_bytes(d);
}

gdn_status gdn_chunk_scan_plan(const gdn_problem *p, int32_t *seg_len, int32_t *num_segments) {
    Dims d;
    const gdn_status st = check_problem(p, &d);
    if (st != GDN_OK) return st;
    if (!seg_len || !num_segments) return GDN_ERR_INVALID_ARG;
    *seg_len = d.seg_len;
    *num_segments = d.seg_len ? d.seg_max : 1;
    return GDN_OK;
}

size_t gdn_chunk_workspace_bytes(const gdn_problem *p, int for_backward) {
    Dims d;
    if (for_backward < 0 || for_backward > 2) return 0;
    if (check_problem(p, &d) != GDN_OK) return 0;
    return ws_bytes(d, for_backward);
}


gdn_status gdn_chunk_fwd_timed(const gdn_problem *p, const void *q, const void *k,
                               const void *v, const float *g, const void *beta,
                               const float *initial_state, void *o, float *final_state,
                               void *saved, void *workspace, size_t ws_size,
                               gdn_stream_t stream, gdn_kernel_timer *timer) {
    return chunk_fwd_impl(p, q, k, v, g, beta, nullptr, initial_state, o, final_state, saved,
                          workspace, ws_size, stream, timer);
}

gdn_status gdn_chunk_bwd_timed(const gdn_problem *p, const void *q, const void *k,
                               const void *v, const float *g, const void *beta,
                               const float *initial_state, const void *saved, const void *d_o,
                               const float *d_final_state, void *dq, void *dk, void *dv,
                               float *dg, void *dbeta, float *dh0, void *workspace,
                               size_t ws_size, gdn_stream_t stream, gdn_kernel_timer *timer) {
    return chunk_bwd_impl(p, q, k, v, g, beta, nullptr, initial_state, saved, d_o, d_final_state,
                          dq, dk, dv, dg, dbeta, dh0, workspace, ws_size, stream, timer);
}

gdn_status gdn_chunk_prefill_paged(const gdn_problem *p, const void *q, const void *k,
                                   const void *v, const float *g, const void *beta,
                                   float *state_pool, int32_t num_slots,
                                   const int32_t *state_indices, const int32_t *has_initial_state,
                                   void *o, int32_t *device_status, void *workspace,
                                   size_t ws_size, gdn_stream_t stream) {
    const Paged pg{state_pool, num_slots, state_indices, has_initial_state, device_status};
    return chunk_fwd_impl(p, q, k, v, g, beta, nullptr, nullptr, o, nullptr, nullptr, workspace,
                          ws_size, stream, nullptr, &pg);
}

gdn_status gdn_chunk_fwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const void *a, const void *b, const float *A_log,
                               const float *dt_bias, const float *initial_state, void *o,
                               float *final_state, void *saved, void *workspace, size_t ws_size,
                               gdn_stream_t stream) {
    const Gate gt{a, b, A_log, dt_bias, nullptr, nullptr, nullptr, nullptr};
    return chunk_fwd_impl(p, q, k, v, nullptr, nullptr, &gt, initial_state, o, final_state, saved,
                          workspace, ws_size, stream, nullptr);
}

gdn_status gdn_chunk_bwd_gated(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const void *a, const void *b, const float *A_log,
                               const float *dt_bias, const float *initial_state,
                               const void *saved, const void *d_o, const float *d_final_state,
                               void *dq, void *dk, void *dv, void *da, void *db, float *dA_log,
                               float *ddt_bias, float *dh0, void *workspace, size_t ws_size,
                               gdn_stream_t stream) {
    const Gate gt{a, b, A_log, dt_bias, da, db, dA_log, ddt_bias};
    return chunk_bwd_impl(p, q, k, v, nullptr, nullptr, &gt, initial_state, saved, d_o,
                          d_final_state, dq, dk, dv, nullptr, nullptr, dh0, workspace, ws_size,
                          stream, nullptr);
}

gdn_status gdn_decode_step_gated(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, float scale,
                                 const void *q, const void *k, const void *v, const void *a,
                                 const void *b, const float *A_log, const float *dt_bias,
                                 float *state_pool, int32_t num_slots,
                                 const int32_t *state_indices, void *o, int32_t *device_status,
                                 gdn_stream_t stream) {
    const Gate gt{a, b, A_log, dt_bias, nullptr, nullptr, nullptr, nullptr};
    return decode_impl(batch, num_k_heads, num_v_heads, head_dim_k, head_dim_v, scale, q, k, v,
                       nullptr, nullptr, &gt, state_pool, num_slots, state_indices, o,
                       device_status, stream, nullptr);
}

gdn_status gdn_decode_step_timed(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                                 int32_t head_dim_k, int32_t head_dim_v, float scale,
                                 const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, float *state_pool, int32_t num_slots,
                                 const int32_t *state_indices, void *o, int32_t *device_status,
                                 gdn_stream_t stream, gdn_kernel_timer *timer) {
    return decode_impl(batch, num_k_heads, num_v_heads, head_dim_k, head_dim_v, scale, q, k, v, g,
                       beta, nullptr, state_pool, num_slots, state_indices, o, device_status,
                       stream, timer);
}

gdn_status gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *initial_state, void *o,
                         float *final_state, void *saved, void *workspace, size_t ws_size,
                         gdn_stream_t stream) {
    return gdn_chunk_fwd_timed(p, q, k, v, g, beta, initial_state, o, final_state, saved,
                               workspace, ws_size, stream, nullptr);
}

gdn_status gdn_chunk_bwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *initial_state,
                         const void *saved, const void *d_o, const float *d_final_state,
                         void *dq, void *dk, void *dv, float *dg, void *dbeta, float *dh0,
                         void *workspace, size_t ws_size, gdn_stream_t stream) {
    return gdn_chunk_bwd_timed(p, q, k, v, g, beta, initial_state, saved, d_o, d_final_state,
                               dq, dk, dv, dg, dbeta, dh0, workspace, ws_size, stream, nullptr);
}

gdn_status gdn_decode_step(int32_t batch, int32_t num_k_heads, int32_t num_v_heads,
                           int32_t head_dim_k, int32_t head_dim_v, float scale, const void *q,
                           const void *k, const void *v, const float *g, const float *beta,
                           float *state_pool, int32_t num_slots, const int32_t *state_indices,
                           void *o, int32_t *device_status, gdn_stream_t stream) {
    return gdn_decode_step_timed(batch, num_k_heads, num_v_heads, head_dim_k, head_dim_v, scale,
                                 q, k, v, g, beta, state_pool, num_slots, state_indices, o,
                                 device_status, stream, nullptr);
}

gdn_status gdn_check_indices(const int32_t *state_indices, int32_t batch, int32_t num_slots,
                             int32_t *bad_row) {
    if (bad_row) *bad_row = -1;
    if (batch < 0 || num_slots < 1 || (batch > 0 && !state_indices)) return GDN_ERR_INVALID_ARG;
    // one bit per slot: O(batch + num_slots) and no ordering of the rows
    uint64_t *seen = static_cast<uint64_t *>(calloc((static_cast<size_t>(num_slots) + 63) / 64, 8));
    if (!seen) return GDN_ERR_INVALID_ARG;
    gdn_status st = GDN_OK;
    for (int32_t i = 0; i < batch; ++i) {
        const int32_t s = state_indices[i];
        if (s <= 0) continue;
        const uint64_t bit = uint64_t(1) << (s & 63);
        if (s >= num_slots || (seen[s >> 6] & bit)) {
            if (bad_row) *bad_row = i;
            st = GDN_ERR_INVALID_ARG;
            break;
        }
        seen[s >> 6] |= bit;
    }
    free(seen);
    return st;
}

const char *gdn_kernel_name(int32_t id) {
    static const char *names[GDN_KERNEL_COUNT] = {
        "plan", "prep", "intra", "state", "out", "dvloc", "bstate", "bintra_a", "bintra_b",
        "decode", "seg_stitch"};
    return (id >= 0 && id < GDN_KERNEL_COUNT) ? names[id] : "unknown";
}

}  // extern "C"
