// gdn_common.cuh -- small device helpers shared by the libgdn kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kChunk = 64;   // chunk length C
constexpr int kDim = 128;    // K = V = 128
constexpr float kNormEps = 1e-6f;

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float bf2f(bf16 x) { return __bfloat162float(x); }
// two packed bf16 (the first in the low half) -> their float values (exact)
__device__ __forceinline__ float2 bf2_to_f2(uint32_t x) {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
__device__ __forceinline__ bf16 f2bf(float x) { return __float2bfloat16_rn(x); }

// Bounds-checked builds (nvcc -DGDN_CHECKED): every direct global access of the
// kernels first passes its element index range [i, i + w) and its buffer's extent n
// to in_range().  A range outside [0, n) ORs GDN_DEVICE_INDEX_OUT_OF_RANGE (4) into
// the caller's status word and the access is skipped (a load gives 0); nothing traps.
// In the normal build in_range() is the constant true and the checks compile away.
#ifdef GDN_CHECKED
constexpr bool kChecked = true;
__device__ __forceinline__ bool in_range(long long i, long long w, long long n, int *status) {
    if (i >= 0 && w >= 0 && i + w <= n) return true;
    if (status) atomicOr(status, 4);
    return false;
}
#else
constexpr bool kChecked = false;
__device__ __forceinline__ bool in_range(long long, long long, long long, int *) { return true; }
#endif

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Fused gating ("C6: GDN decode-step goldens and recurrent/conv state contract",
// Provider): beta = sigmoid(b), g = -exp(A_log) softplus(a + dt_bias) in fp32, with
// softplus(x) = x above the threshold 20 (its slope there is 1, sigmoid(x) below).
__device__ __forceinline__ float gate_softplus(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float gate_softplus_slope(float x) {
    return x > 20.f ? 1.f : 1.f / (1.f + expf(-x));
}
__device__ __forceinline__ float gate_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }


}  // namespace gdn
