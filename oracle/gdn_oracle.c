/*
 * gdn_oracle.c -- plain, slow fp64 CPU reference of the gated delta rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only tests/, the smoke check and the bench's CPU-baseline leg use
 * it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (sources, by page title and section):
 *  - "cake_gdn: deterministic chunked GDN training kernels" (miles #3597),
 *    Summary: chunk_gated_delta_rule forward + backward, K = V = 128 in
 *    production (any K, V here), in-kernel q/k L2 norm, cu_seqlens packing,
 *    grouped value heads passed to the kernel directly.
 *  - "C6: GDN decode-step goldens and recurrent/conv state contract"
 *    (RL-Kernel #469), "What" and "Provider": the L2 norm is
 *    x / sqrt(sum(x*x) + 1e-6) (divide by sqrt), scale multiplies q after
 *    the norm, k is never scaled, key head = value head // (HV / H), state pool
 *    [num_blocks, HV, V, K] addressed by ssm_state_indices, every index <= 0
 *    skipped with a zero output row.
 *  - "[Cake 1/13] gdn: chunked gated delta rule ..." (miles-ext-kernels #1),
 *    "API and flags": initial / final state fp32 [N, HV, K, V] (K-major, the
 *    transpose of the decode layout), HV % H == 0, a call without tokens
 *    passes the state through.
 *  - The recurrence itself: S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T)
 *    + beta_t v_t k_t^T, o_t = S_t q_t (S is V x K), written per token as
 *      S' = exp(g_t) S_{t-1};  p = S' k;  delta = beta_t (v_t - p);
 *      S_t = S' + delta k^T;    o_t = S_t q.
 *  - Fused gating: "C6: GDN decode-step goldens and recurrent/conv state
 *    contract" (RL-Kernel #469), "What" and "Provider": beta = sigmoid(b) and
 *    g = -exp(A_log) softplus(a + dt_bias), computed in fp32 in the provider
 *    (fp64 here) with the softplus threshold at 20 (softplus(x) = x above it).
 *  - The chunked (WY) form: "Qwen3.5-397B RL trainer on 128 v7x" (maxtext
 *    #5799), GDN context-parallel m-scan and dh-scan commits: the chunk
 *    transition M_c = g_last I - k_bwd^T (t_inv k_beta_g) and the reverse
 *    recurrence dh <- g_last dh + q_g^T do - k_beta_g^T t_inv^T (attn^T do +
 *    k_bwd dh), with t_inv the inverse of the unit lower-triangular
 *    intra-chunk matrix.
 *
 * Every array is a dense row-major double array.  Work is split in "units":
 * unit u = n * HV + hv (sequence n, value head hv) for the chunk entry points,
 * and u = b * HV + hv for decode.  Units write disjoint outputs, so callers
 * may run disjoint unit ranges on several threads at once.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define L2_EPS 1e-6

/* Planted mistakes for the test suite's discrimination checks (0 = none).
 * Each number breaks one step; the tests assert every one of them fails at
 * least one pin.  Never set outside tests. */
static int g_mutation = 0;
void gdn_oracle_set_mutation(int m) { g_mutation = m; }
int gdn_oracle_get_mutation(void) { return g_mutation; }

/* x / sqrt(sum x^2 + 1e-6), times mul; r receives sqrt(sum x^2 + 1e-6). */
static void l2_normalise(const double *x, int n, int use_l2norm, double mul,
                         double *out, double *r)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double rr = use_l2norm ? sqrt(ss + L2_EPS) : 1.0;
    if (use_l2norm && g_mutation == 5) rr = sqrt(ss) + L2_EPS;
    for (int i = 0; i < n; ++i) out[i] = mul * x[i] / rr;
    if (r) *r = rr;
}

/* Backward of n = x / r, r = sqrt(|x|^2 + eps):  dx = (dn - n (n . dn)) / r. */
static void l2_backward(const double *x, const double *dn, int n, int use_l2norm,
                        double *dx)
{
    if (!use_l2norm) {
        for (int i = 0; i < n; ++i) dx[i] = dn[i];
        return;
    }
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = sqrt(ss + L2_EPS);
    double ndn = 0.0;
    for (int i = 0; i < n; ++i) ndn += (x[i] / r) * dn[i];
    for (int i = 0; i < n; ++i) dx[i] = (dn[i] - (x[i] / r) * ndn) / r;
}

static int key_head_of(int hv, int H, int HV)
{
    int r = HV / H;
    if (g_mutation == 7) return hv % H;
    return hv / r;
}

/* One token of the recurrence on S (V x K, row v = S[v*K ...]).
 * kh, qh: normalised key / scaled query; a = exp(g); b = beta.
 * Writes o (V) and, if p_out / d_out are given, the prediction p and delta. */
static void token_step(double *S, int K, int V, const double *kh, const double *qh,
                       const double *vt, double a, double b, double *o,
                       double *p_out, double *d_out)
{
    if (g_mutation != 1)
        for (int i = 0; i < V * K; ++i) S[i] *= a;
    for (int vi = 0; vi < V; ++vi) {
        const double *row = S + (size_t)vi * K;
        double p = 0.0;
        for (int c = 0; c < K; ++c) p += row[c] * kh[c];
        if (g_mutation == 2 && a != 0.0) p /= a;  /* prediction from the undecayed state */
        double d = b * (vt[vi] - p);
        if (p_out) p_out[vi] = p;
        if (d_out) d_out[vi] = d;
        double *wrow = S + (size_t)vi * K;
        if (g_mutation == 3) {  /* output read before the write */
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += wrow[c] * qh[c];
            o[vi] = acc;
        }
        for (int c = 0; c < K; ++c) wrow[c] += d * kh[c];
    }
    if (g_mutation == 1)
        for (int i = 0; i < V * K; ++i) S[i] *= a;
    if (g_mutation != 3) {
        for (int vi = 0; vi < V; ++vi) {
            const double *row = S + (size_t)vi * K;
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += row[c] * qh[c];
            o[vi] = acc;
        }
    }
}

static void load_state(double *S, const double *h0, int n, int hv, int HV, int K, int V)
{
    /* h0 is K-major [N, HV, K, V]; S = h0^T is V x K. */
    if (!h0) { memset(S, 0, sizeof(double) * (size_t)K * V); return; }
    const double *src = h0 + ((size_t)n * HV + hv) * K * V;
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < V; ++b) S[(size_t)b * K + a] = src[(size_t)a * V + b];
}

static void store_state(const double *S, double *ht, int n, int hv, int HV, int K, int V)
{
    double *dst = ht + ((size_t)n * HV + hv) * K * V;
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < V; ++b) dst[(size_t)a * V + b] = S[(size_t)b * K + a];
}

/* Per-token forward.  q, k: [T, H, K]; v: [T, HV, V]; g, beta: [T, HV];
 * h0, ht: [N, HV, K, V] (nullable); o: [T, HV, V]. */
void gdn_oracle_fwd(int N, const int *cu, int H, int HV, int K, int V, double scale,
                    int use_l2norm, const double *q, const double *k, const double *v,
                    const double *g, const double *beta, const double *h0, double *o,
                    double *ht, int unit_begin, int unit_end)
{
    double *S = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *qh = (double *)malloc(sizeof(double) * K);
    double *kh = (double *)malloc(sizeof(double) * K);
    for (int u = unit_begin; u < unit_end; ++u) {
        int n = u / HV, hv = u % HV, h = key_head_of(hv, H, HV);
        load_state(S, h0, n, hv, HV, K, V);
        for (int t = cu[n]; t < cu[n + 1]; ++t) {
            l2_normalise(q + ((size_t)t * H + h) * K, K, use_l2norm, scale, qh, NULL);
            l2_normalise(k + ((size_t)t * H + h) * K, K, use_l2norm,
                         g_mutation == 4 ? scale : 1.0, kh, NULL);
            token_step(S, K, V, kh, qh, v + ((size_t)t * HV + hv) * V,
                       exp(g[(size_t)t * HV + hv]), beta[(size_t)t * HV + hv],
                       o + ((size_t)t * HV + hv) * V, NULL, NULL);
        }
        if (ht) store_state(S, ht, n, hv, HV, K, V);
    }
    free(S); free(qh); free(kh);
}

/* Per-token backward, hand-derived from the per-token forward, in reverse
 * token order.  Forward states are recovered from checkpoints taken every
 * 64 tokens and recomputed one segment at a time.
 *
 * Outputs per unit (n, hv): dq_part, dk_part [T, HV, K] are the gradients of
 * q and k (after the L2-norm backward) through this value head only; the
 * caller sums them over the HV/H value heads of each key head.
 * dv [T, HV, V]; dg, dbeta [T, HV]; dh0 [N, HV, K, V] (nullable).
 * d_ht [N, HV, K, V] is the gradient of the final state (nullable = 0). */
void gdn_oracle_bwd(int N, const int *cu, int H, int HV, int K, int V, double scale,
                    int use_l2norm, const double *q, const double *k, const double *v,
                    const double *g, const double *beta, const double *h0,
                    const double *d_o, const double *d_ht, double *dq_part,
                    double *dk_part, double *dv, double *dg, double *dbeta,
                    double *dh0, int unit_begin, int unit_end)
{
    const int SEG = 64;
    size_t SZ = (size_t)K * V;
    double *dS = (double *)malloc(sizeof(double) * SZ);
    double *dSp = (double *)malloc(sizeof(double) * SZ);
    double *Sp = (double *)malloc(sizeof(double) * SZ);
    double *seg = (double *)malloc(sizeof(double) * SZ * (SEG + 1));
    double *qh = (double *)malloc(sizeof(double) * K);
    double *kh = (double *)malloc(sizeof(double) * K);
    double *dqh = (double *)malloc(sizeof(double) * K);
    double *dkh = (double *)malloc(sizeof(double) * K);
    double *tmpk = (double *)malloc(sizeof(double) * K);
    double *p = (double *)malloc(sizeof(double) * V);
    double *dlt = (double *)malloc(sizeof(double) * V);
    double *ddl = (double *)malloc(sizeof(double) * V);
    double *dp = (double *)malloc(sizeof(double) * V);
    double *otmp = (double *)malloc(sizeof(double) * V);
    for (int u = unit_begin; u < unit_end; ++u) {
        int n = u / HV, hv = u % HV, h = key_head_of(hv, H, HV);
        int t0 = cu[n], L = cu[n + 1] - cu[n];
        int nseg = (L + SEG - 1) / SEG;
        double *ck = (double *)malloc(sizeof(double) * SZ * (nseg > 0 ? nseg : 1));
        /* forward pass: checkpoint the state at each segment start */
        double *S = seg;  /* scratch */
        load_state(S, h0, n, hv, HV, K, V);
        for (int s = 0; s < nseg; ++s) {
            memcpy(ck + SZ * s, S, sizeof(double) * SZ);
            int ts = t0 + s * SEG, te = ts + SEG < t0 + L ? ts + SEG : t0 + L;
            for (int t = ts; t < te; ++t) {
                l2_normalise(q + ((size_t)t * H + h) * K, K, use_l2norm, scale, qh, NULL);
                l2_normalise(k + ((size_t)t * H + h) * K, K, use_l2norm, 1.0, kh, NULL);
                token_step(S, K, V, kh, qh, v + ((size_t)t * HV + hv) * V,
                           exp(g[(size_t)t * HV + hv]), beta[(size_t)t * HV + hv], otmp,
                           NULL, NULL);
            }
        }
        /* seed */
        if (d_ht) {
            const double *src = d_ht + ((size_t)n * HV + hv) * SZ;
            for (int a = 0; a < K; ++a)
                for (int b = 0; b < V; ++b) dS[(size_t)b * K + a] = src[(size_t)a * V + b];
        } else {
            memset(dS, 0, sizeof(double) * SZ);
        }
        for (int s = nseg - 1; s >= 0; --s) {
            int ts = t0 + s * SEG, te = ts + SEG < t0 + L ? ts + SEG : t0 + L;
            int len = te - ts;
            memcpy(seg, ck + SZ * s, sizeof(double) * SZ);
            for (int j = 0; j < len; ++j) {
                int t = ts + j;
                memcpy(seg + SZ * (j + 1), seg + SZ * j, sizeof(double) * SZ);
                l2_normalise(q + ((size_t)t * H + h) * K, K, use_l2norm, scale, qh, NULL);
                l2_normalise(k + ((size_t)t * H + h) * K, K, use_l2norm, 1.0, kh, NULL);
                token_step(seg + SZ * (j + 1), K, V, kh, qh, v + ((size_t)t * HV + hv) * V,
                           exp(g[(size_t)t * HV + hv]), beta[(size_t)t * HV + hv], otmp,
                           NULL, NULL);
            }
            for (int j = len - 1; j >= 0; --j) {
                int t = ts + j;
                const double *Sprev = seg + SZ * j, *Scur = seg + SZ * (j + 1);
                const double *qt = q + ((size_t)t * H + h) * K;
                const double *kt = k + ((size_t)t * H + h) * K;
                const double *vt = v + ((size_t)t * HV + hv) * V;
                const double *dot = d_o + ((size_t)t * HV + hv) * V;
                double a = exp(g[(size_t)t * HV + hv]), b = beta[(size_t)t * HV + hv];
                l2_normalise(qt, K, use_l2norm, scale, qh, NULL);
                l2_normalise(kt, K, use_l2norm, 1.0, kh, NULL);
                for (size_t i = 0; i < SZ; ++i) Sp[i] = a * Sprev[i];
                for (int vi = 0; vi < V; ++vi) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += Sp[(size_t)vi * K + c] * kh[c];
                    p[vi] = acc;
                    dlt[vi] = b * (vt[vi] - acc);
                }
                /* o_t = S_t qh:  dqh = S_t^T do,  dS += do qh^T */
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int vi = 0; vi < V; ++vi) acc += Scur[(size_t)vi * K + c] * dot[vi];
                    dqh[c] = acc;
                }
                for (int vi = 0; vi < V; ++vi)
                    for (int c = 0; c < K; ++c) dS[(size_t)vi * K + c] += dot[vi] * qh[c];
                /* S_t = S' + delta kh^T */
                for (int vi = 0; vi < V; ++vi) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += dS[(size_t)vi * K + c] * kh[c];
                    ddl[vi] = acc;
                }
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int vi = 0; vi < V; ++vi) acc += dS[(size_t)vi * K + c] * dlt[vi];
                    dkh[c] = acc;
                }
                /* delta = b (v - p) */
                double db = 0.0;
                for (int vi = 0; vi < V; ++vi) {
                    db += ddl[vi] * (vt[vi] - p[vi]);
                    dv[((size_t)t * HV + hv) * V + vi] = b * ddl[vi];
                    dp[vi] = (g_mutation == 6 ? b : -b) * ddl[vi];
                }
                dbeta[(size_t)t * HV + hv] = db;
                /* p = S' kh */
                for (int vi = 0; vi < V; ++vi)
                    for (int c = 0; c < K; ++c)
                        dSp[(size_t)vi * K + c] = dS[(size_t)vi * K + c] + dp[vi] * kh[c];
                for (int c = 0; c < K; ++c) {
                    double acc = 0.0;
                    for (int vi = 0; vi < V; ++vi) acc += Sp[(size_t)vi * K + c] * dp[vi];
                    dkh[c] += acc;
                }
                /* S' = a Sprev */
                double da = 0.0;
                for (size_t i = 0; i < SZ; ++i) da += dSp[i] * Sprev[i];
                dg[(size_t)t * HV + hv] = a * da;
                for (size_t i = 0; i < SZ; ++i) dS[i] = a * dSp[i];
                /* L2-norm backward (qh = scale * q / r_q, kh = k / r_k) */
                for (int c = 0; c < K; ++c) tmpk[c] = scale * dqh[c];
                l2_backward(qt, tmpk, K, use_l2norm, dq_part + ((size_t)t * HV + hv) * K);
                l2_backward(kt, dkh, K, use_l2norm, dk_part + ((size_t)t * HV + hv) * K);
            }
        }
        if (dh0) store_state(dS, dh0, n, hv, HV, K, V);
        free(ck);
    }
    free(dS); free(dSp); free(Sp); free(seg); free(qh); free(kh); free(dqh); free(dkh);
    free(tmpk); free(p); free(dlt); free(ddl); free(dp); free(otmp);
}

/* Chunked (WY) forward, any chunk size C >= 1, exact in fp64.  Per chunk of
 * length L <= C (chunks never span sequences; the last one may be partial),
 * with h the K x V state at the chunk start (h = S^T):
 *   G_i   = sum_{j <= i} g_j                          (chunk-local cumsum)
 *   A_ij  = beta_i (kh_i . kh_j) exp(G_i - G_j),  j < i   (strictly lower)
 *   Tm    = (I + A)^-1                                 (unit lower triangular)
 *   w     = Tm diag(beta exp(G)) Kh,   u = Tm diag(beta) V
 *   v_new = u - w h
 *   o     = diag(exp(G)) Qh h + tril(Qh Kh^T (.) exp(G_i - G_j)) v_new
 *   h    <- exp(G_L) h + (diag(exp(G_L - G)) Kh)^T v_new
 * Optional outputs: h_chunks [num_chunks, HV, K, V] (the state at each chunk
 * start, chunks numbered in packing order) and v_new [T, HV, V]. */
void gdn_oracle_fwd_chunked(int N, const int *cu, int H, int HV, int K, int V,
                            double scale, int use_l2norm, int C, const double *q,
                            const double *k, const double *v, const double *g,
                            const double *beta, const double *h0, double *o, double *ht,
                            double *h_chunks, double *v_new_out, int unit_begin,
                            int unit_end)
{
    size_t SZ = (size_t)K * V;
    double *hs = (double *)malloc(sizeof(double) * SZ);
    double *Qh = (double *)malloc(sizeof(double) * (size_t)C * K);
    double *Kh = (double *)malloc(sizeof(double) * (size_t)C * K);
    double *G = (double *)malloc(sizeof(double) * C);
    double *A = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *Tm = (double *)malloc(sizeof(double) * (size_t)C * C);
    double *w = (double *)malloc(sizeof(double) * (size_t)C * K);
    double *uu = (double *)malloc(sizeof(double) * (size_t)C * V);
    double *vn = (double *)malloc(sizeof(double) * (size_t)C * V);
    for (int u = unit_begin; u < unit_end; ++u) {
        int n = u / HV, hv = u % HV, h = key_head_of(hv, H, HV);
        long chunk_base = 0;
        for (int m = 0; m < n; ++m) chunk_base += (cu[m + 1] - cu[m] + C - 1) / C;
        /* hs = h0[n, hv] (K-major K x V) */
        if (h0) memcpy(hs, h0 + ((size_t)n * HV + hv) * SZ, sizeof(double) * SZ);
        else memset(hs, 0, sizeof(double) * SZ);
        int ci = 0;
        for (int cs = cu[n]; cs < cu[n + 1]; cs += C, ++ci) {
            int L = cu[n + 1] - cs < C ? cu[n + 1] - cs : C;
            if (h_chunks)
                memcpy(h_chunks + ((size_t)(chunk_base + ci) * HV + hv) * SZ, hs,
                       sizeof(double) * SZ);
            double acc = 0.0;
            for (int i = 0; i < L; ++i) {
                int t = cs + i;
                l2_normalise(q + ((size_t)t * H + h) * K, K, use_l2norm, scale, Qh + (size_t)i * K, NULL);
                l2_normalise(k + ((size_t)t * H + h) * K, K, use_l2norm, 1.0, Kh + (size_t)i * K, NULL);
                acc += g[(size_t)t * HV + hv];
                G[i] = acc;
            }
            for (int i = 0; i < L; ++i) {
                double bi = beta[(size_t)(cs + i) * HV + hv];
                for (int j = 0; j < L; ++j) {
                    double a = 0.0;
                    if (j < i) {
                        double kk = 0.0;
                        for (int c = 0; c < K; ++c) kk += Kh[(size_t)i * K + c] * Kh[(size_t)j * K + c];
                        a = bi * kk * (g_mutation == 11 ? exp(G[j] - G[i]) : exp(G[i] - G[j]));  /* 11: flipped */
                    }
                    A[(size_t)i * C + j] = a;
                }
            }
            /* Tm = (I + A)^-1 by forward substitution, column by column */
            for (int j = 0; j < L; ++j) {
                for (int i = 0; i < L; ++i) {
                    double x = (i == j) ? 1.0 : 0.0;
                    for (int m = j; m < i; ++m) x -= A[(size_t)i * C + m] * Tm[(size_t)m * C + j];
                    Tm[(size_t)i * C + j] = (i < j) ? 0.0 : x;
                }
            }
            /* w = Tm diag(beta e^G) Kh;  u = Tm diag(beta) V */
            for (int i = 0; i < L; ++i) {
                for (int c = 0; c < K; ++c) {
                    double s = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        double bj = beta[(size_t)(cs + j) * HV + hv];
                        s += Tm[(size_t)i * C + j] * bj * exp(G[j]) * Kh[(size_t)j * K + c];
                    }
                    w[(size_t)i * K + c] = s;
                }
                for (int c = 0; c < V; ++c) {
                    double s = 0.0;
                    for (int j = 0; j <= i; ++j) {
                        double bj = beta[(size_t)(cs + j) * HV + hv];
                        s += Tm[(size_t)i * C + j] * bj * v[((size_t)(cs + j) * HV + hv) * V + c];
                    }
                    uu[(size_t)i * V + c] = s;
                }
            }
            /* v_new = u - w h */
            for (int i = 0; i < L; ++i)
                for (int c = 0; c < V; ++c) {
                    double s = 0.0;
                    for (int a = 0; a < K; ++a) s += w[(size_t)i * K + a] * hs[(size_t)a * V + c];
                    vn[(size_t)i * V + c] = uu[(size_t)i * V + c] - s;
                    if (v_new_out) v_new_out[((size_t)(cs + i) * HV + hv) * V + c] = vn[(size_t)i * V + c];
                }
            /* o = diag(e^G) Qh h + tril(Qh Kh^T (.) decay) v_new */
            for (int i = 0; i < L; ++i) {
                double *orow = o + ((size_t)(cs + i) * HV + hv) * V;
                double eg = exp(G[i]);
                for (int c = 0; c < V; ++c) {
                    double s = 0.0;
                    for (int a = 0; a < K; ++a) s += Qh[(size_t)i * K + a] * hs[(size_t)a * V + c];
                    orow[c] = eg * s;
                }
                for (int j = 0; j <= i; ++j) {
                    double qk = 0.0;
                    for (int a = 0; a < K; ++a) qk += Qh[(size_t)i * K + a] * Kh[(size_t)j * K + a];
                    double m = qk * exp(G[i] - G[j]);
                    for (int c = 0; c < V; ++c) orow[c] += m * vn[(size_t)j * V + c];
                }
            }
            /* h <- e^{G_L} h + (diag(e^{G_L - G}) Kh)^T v_new */
            double GL = G[L - 1], egl = exp(GL);
            for (size_t i = 0; i < SZ; ++i) hs[i] *= egl;
            for (int j = 0; j < L; ++j) {
                double f = g_mutation == 12 ? exp(G[j] - GL) : exp(GL - G[j]);  /* 12: flipped */
                for (int a = 0; a < K; ++a) {
                    double ka = f * Kh[(size_t)j * K + a];
                    for (int c = 0; c < V; ++c) hs[(size_t)a * V + c] += ka * vn[(size_t)j * V + c];
                }
            }
        }
        if (ht) memcpy(ht + ((size_t)n * HV + hv) * SZ, hs, sizeof(double) * SZ);
    }
    free(hs); free(Qh); free(Kh); free(G); free(A); free(Tm); free(w); free(uu); free(vn);
}

/* Single-token decode step over a slot-indexed state pool ("C6: GDN
 * decode-step goldens ...", "Provider" and "State contract").
 * q, k: [B, H, K]; v: [B, HV, V]; g, beta: [B, HV];
 * pool: [num_slots, HV, V, K] (V-major rows, S itself), updated in place;
 * idx: [B] slot per row, <= 0 = null (row skipped, output row zero, slot
 * untouched); o: [B, HV, V].  Units are rows u = b * HV + hv.  An index
 * >= num_slots is treated like a null row and counted in the return value. */
int gdn_oracle_decode(int B, int H, int HV, int K, int V, double scale, int use_l2norm,
                      const double *q, const double *k, const double *v, const double *g,
                      const double *beta, double *pool, int num_slots, const int *idx,
                      double *o, int unit_begin, int unit_end)
{
    int bad = 0;
    double *qh = (double *)malloc(sizeof(double) * K);
    double *kh = (double *)malloc(sizeof(double) * K);
    (void)B;
    for (int u = unit_begin; u < unit_end; ++u) {
        int b = u / HV, hv = u % HV, h = key_head_of(hv, H, HV);
        double *orow = o + ((size_t)b * HV + hv) * V;
        int slot = idx[b];
        if (slot <= 0 || slot >= num_slots) {
            if (slot >= num_slots) ++bad;
            for (int c = 0; c < V; ++c) orow[c] = 0.0;
            continue;
        }
        double *S = pool + ((size_t)slot * HV + hv) * K * V;
        l2_normalise(q + ((size_t)b * H + h) * K, K, use_l2norm, scale, qh, NULL);
        l2_normalise(k + ((size_t)b * H + h) * K, K, use_l2norm, 1.0, kh, NULL);
        token_step(S, K, V, kh, qh, v + ((size_t)b * HV + hv) * V,
                   g_mutation == 13 ? 1.0 : exp(g[(size_t)b * HV + hv]),  /* 13: decay left out */
                   beta[(size_t)b * HV + hv], orow, NULL, NULL);
    }
    free(qh); free(kh);
    return bad;
}

/* ---------------------------------------------------------------- fused gating
 * a, b, g, beta, dg, dbeta, da, db: [n, HV] (n tokens or decode rows); A_log,
 * dt_bias, dA_log, ddt_bias: [HV].  softplus(x) = x for x > 20, log(1 + e^x)
 * otherwise, so its derivative is 1 above the threshold and sigmoid(x) below. */
static double softplus_thr(double x) { return x > 20.0 ? x : log1p(exp(x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

void gdn_oracle_gate_fwd(int n, int HV, const double *a, const double *b, const double *A_log,
                         const double *dt_bias, double *g, double *beta)
{
    for (int t = 0; t < n; ++t)
        for (int h = 0; h < HV; ++h) {
            const size_t i = (size_t)t * HV + h;
            g[i] = -exp(A_log[h]) * softplus_thr(a[i] + dt_bias[h]);
            beta[i] = sigmoid(b[i]);
        }
}

/* Backward of gdn_oracle_gate_fwd for incoming dg, dbeta:
 *   da = dg * (-e^{A_log}) * softplus'(a + dt_bias),   ddt_bias = sum_t da,
 *   dA_log = sum_t dg * g,                             db = dbeta * beta (1 - beta). */
void gdn_oracle_gate_bwd(int n, int HV, const double *a, const double *b, const double *A_log,
                         const double *dt_bias, const double *dg, const double *dbeta,
                         double *da, double *db, double *dA_log, double *ddt_bias)
{
    for (int h = 0; h < HV; ++h) {
        dA_log[h] = 0.0;
        ddt_bias[h] = 0.0;
    }
    for (int t = 0; t < n; ++t)
        for (int h = 0; h < HV; ++h) {
            const size_t i = (size_t)t * HV + h;
            const double x = a[i] + dt_bias[h], e = exp(A_log[h]);
            const double dsp = x > 20.0 ? 1.0 : sigmoid(x);
            const double gi = -e * softplus_thr(x);
            da[i] = dg[i] * -e * (g_mutation == 9 ? softplus_thr(x) : dsp);
            dA_log[h] += dg[i] * gi;
            ddt_bias[h] += da[i];
            const double be = sigmoid(b[i]);
            db[i] = dbeta[i] * (g_mutation == 8 ? be : be * (1.0 - be));
        }
}
