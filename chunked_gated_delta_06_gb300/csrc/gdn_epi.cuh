// gdn_epi.cuh -- small epilogue helpers shared by the backward chunk kernels:
// bf16 packing into 128-byte-swizzled operand rows, and fixed-order column sums
// over the rows of an M=64 tcgen05 result (row m in lane m % 16 of warp m / 16).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_umma.cuh"

namespace gdn {
namespace epi {

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&t);
}

// Write 32 consecutive fp32 values of row `row`, columns [col0, col0 + 32), as
// bf16 into a 64-wide SW128 tile.
__device__ __forceinline__ void put_row32(unsigned char *tile, int row, int col0, const float *x) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(tile + umma::sw128_off(row, col0 + q * 8)) =
            make_uint4(pack_bf2(x[q * 8 + 0], x[q * 8 + 1]), pack_bf2(x[q * 8 + 2], x[q * 8 + 3]),
                       pack_bf2(x[q * 8 + 4], x[q * 8 + 5]), pack_bf2(x[q * 8 + 6], x[q * 8 + 7]));
}

// Column sums over the 16 rows that lanes 0..15 of the warp hold (one value per
// column for 32 columns).  Butterfly: each step keeps half of the columns and
// adds the partner's copy of them, so lane l (< 16) ends with the sums of
// columns 2 (l & 15) and 2 (l & 15) + 1.  Lanes 16..31 only exchange among
// themselves.  The order of the additions is fixed.
__device__ __forceinline__ void colsum16(const float (&x)[32], int lane, float &s0, float &s1) {
    float a[16], b[8], c[4];
    const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float send = b3 ? x[j] : x[16 + j];
        a[j] = (b3 ? x[16 + j] : x[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float send = b2 ? a[j] : a[8 + j];
        b[j] = (b2 ? a[8 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b1 ? b[j] : b[4 + j];
        c[j] = (b1 ? b[4 + j] : b[j]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float send0 = b0 ? c[0] : c[2], send1 = b0 ? c[1] : c[3];
    const float r0 = __shfl_xor_sync(0xffffffffu, send0, 1);
    const float r1 = __shfl_xor_sync(0xffffffffu, send1, 1);
    s0 = (b0 ? c[2] : c[0]) + r0;
    s1 = (b0 ? c[3] : c[1]) + r1;
}

}  // namespace epi
}  // namespace gdn
