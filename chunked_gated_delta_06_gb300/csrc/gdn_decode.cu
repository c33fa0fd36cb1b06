// gdn_decode.cu -- single-token gated-delta decode step over a slot-indexed
// fp32 state pool.
//
// Follows "C6: GDN decode-step goldens and recurrent/conv state contract"
// (RL-Kernel #469), sections What / Provider / State contract:
//   qhat = scale * q / sqrt(sum q^2 + 1e-6),  khat = k / sqrt(sum k^2 + 1e-6)
//   key head = value head // (HV / H)
//   S <- e^g S;  p = S khat;  S += beta (v - p) khat^T;  o = S qhat
// with g and beta given, or computed in the kernel from the fused gate's
// pre-activations (Provider: beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias)),
// on the pool [num_slots, HV, V, K] (row v of S holds K contiguous floats),
// indices <= 0 skipped with a zero output row.
//
// Layout choice: one block per (row b, value head); each warp owns 16 rows of
// S and each lane one float4 of a row, so every row is one coalesced 512-byte
// load and store and both dot products (S khat, S qhat) come from the same
// registers: o_v = e^g (S qhat)_v + delta_v (khat . qhat), with
// delta_v = beta (v_v - e^g (S khat)_v).  The per-row reductions run in a fixed
// shuffle order, so a row's result does not depend on its batch position.
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kDecodeWarps = 8;
constexpr int kRowsPerWarp = kDim / kDecodeWarps;  // 16

__device__ __forceinline__ float4 ld_stream(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ void st_stream(float *p, float4 v) {
    __stcs(reinterpret_cast<float4 *>(p), v);
}

__global__ void __launch_bounds__(kDecodeWarps * 32)
    k_decode(int H, int HV, float scale, const bf16 *__restrict__ q, const bf16 *__restrict__ k,
             const bf16 *__restrict__ v, const float *__restrict__ g,
             const float *__restrict__ beta, const DecodeGate gate, float *__restrict__ pool,
             int num_slots, const int32_t *__restrict__ idx, bf16 *__restrict__ o,
             int32_t *status) {
    const int b = blockIdx.x / HV, hv = blockIdx.x % HV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = idx[b];
    bf16 *orow = o + ((size_t)b * HV + hv) * kDim;
    if (slot <= 0 || slot >= num_slots) {
        if (threadIdx.x < kDim) orow[threadIdx.x] = f2bf(0.f);
        if (slot >= num_slots && threadIdx.x == 0 && status) *status = 1;
        return;
    }
    const int h = hv / (HV / H);
    if (!in_range(((size_t)slot * HV + hv) * kDim * kDim, kDim * kDim, (long long)num_slots * HV * kDim * kDim,
                  status) ||
        !in_range(((size_t)b * H + h) * kDim, kDim, (long long)(gridDim.x / HV) * H * kDim, status))
        return;
    float *S = pool + ((size_t)slot * HV + hv) * kDim * kDim;
    const int r0 = warp * kRowsPerWarp;
    // issue the state loads first: 16 rows x float4 per lane
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) s[j] = ld_stream(S + (size_t)(r0 + j) * kDim + lane * 4);
    // normalised q, k slices of this lane (4 elements each)
    const bf16 *qr = q + ((size_t)b * H + h) * kDim + lane * 4;
    const bf16 *kr = k + ((size_t)b * H + h) * kDim + lane * 4;
    float qv[4], kv[4], sq = 0.f, sk = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        qv[u] = bf2f(qr[u]);
        kv[u] = bf2f(kr[u]);
        sq += qv[u] * qv[u];
        sk += kv[u] * kv[u];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float rq = sqrtf(sq + kNormEps), rk = sqrtf(sk + kNormEps);
    float kq = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        qv[u] = scale * qv[u] / rq;
        kv[u] = kv[u] / rk;
        kq += kv[u] * qv[u];
    }
    kq = warp_sum(kq);
    // decay and beta: given, or from the fused gate (fp32, softplus threshold 20)
    const size_t gi = (size_t)b * HV + hv;
    const float gv = gate.a ? -expf(gate.A_log[hv]) * gate_softplus(bf2f(gate.a[gi]) + gate.dt_bias[hv])
                            : g[gi];
    const float a = expf(gv);
    const float bt = gate.a ? gate_sigmoid(bf2f(gate.b[gi])) : beta[gi];
    const bf16 *vrow = v + ((size_t)b * HV + hv) * kDim;
    float my_o = 0.f;
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        float pk = s[j].x * kv[0] + s[j].y * kv[1] + s[j].z * kv[2] + s[j].w * kv[3];
        float pq = s[j].x * qv[0] + s[j].y * qv[1] + s[j].z * qv[2] + s[j].w * qv[3];
        pk = warp_sum(pk);
        pq = warp_sum(pq);
        const float d = bt * (bf2f(vrow[r0 + j]) - a * pk);
        float4 t;
        t.x = a * s[j].x + d * kv[0];
        t.y = a * s[j].y + d * kv[1];
        t.z = a * s[j].z + d * kv[2];
        t.w = a * s[j].w + d * kv[3];
        st_stream(S + (size_t)(r0 + j) * kDim + lane * 4, t);
        const float ov = a * pq + d * kq;
        if (lane == j) my_o = ov;
    }
    if (lane < kRowsPerWarp) orow[r0 + lane] = f2bf(my_o);
}

}  // namespace

cudaError_t launch_decode(int B, int H, int HV, float scale, const bf16 *q, const bf16 *k,
                          const bf16 *v, const float *g, const float *beta, const DecodeGate &gate,
                          float *pool, int num_slots, const int32_t *idx, bf16 *o, int32_t *status,
                          cudaStream_t s, gdn_kernel_timer *timer) {
    if (B == 0) return cudaSuccess;
    TimerScope ts(timer, GDN_KERNEL_DECODE, s);
    k_decode<<<(unsigned)((size_t)B * HV), kDecodeWarps * 32, 0, s>>>(
        H, HV, scale, q, k, v, g, beta, gate, pool, num_slots, idx, o, status);
    return cudaGetLastError();
}

}  // namespace gdn
