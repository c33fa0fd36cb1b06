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

// ---- M=64 results read as 16x256b fragments: all 32 lanes of a warp work.
// For the 16 TMEM lanes (result rows) of warp w and 32 columns from column
// address c, tcgen05.ld.16x256b.x4 gives lane t the registers
//   x[4k + e] = D[16 w + t/4 + 8 (e >> 1)][c + 8k + 2 (t % 4) + (e & 1)],  k, e = 0..3
// (checked on the GPU: two rows, eight columns per lane).
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, float (&x)[16]) {
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(u[i]);
}

// Store of the same fragment layout (16 lanes from the address's lane, 32 columns).
__device__ __forceinline__ void tmem_st16x256_x4(uint32_t taddr, const float (&x)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])), "r"(__float_as_uint(x[2])),
          "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])), "r"(__float_as_uint(x[5])),
          "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7])), "r"(__float_as_uint(x[8])),
          "r"(__float_as_uint(x[9])), "r"(__float_as_uint(x[10])), "r"(__float_as_uint(x[11])),
          "r"(__float_as_uint(x[12])), "r"(__float_as_uint(x[13])), "r"(__float_as_uint(x[14])),
          "r"(__float_as_uint(x[15]))
        : "memory");
}

// Column sums over the 16 rows of a 16x256b fragment: y[2k + p] is this lane's
// two-row partial of column 8k + 2 (t % 4) + p.  Three butterfly steps over the
// eight lanes that share t % 4 leave lane t with the sum of column
// 8 (c8 >> 1) + 2 (t % 4) + (c8 & 1), c8 = t / 4.  Fixed order.
__device__ __forceinline__ float colsum_frag(const float (&y)[8], int lane) {
    float a[4], b[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b4 ? y[j] : y[4 + j];
        a[j] = (b4 ? y[4 + j] : y[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b3 ? a[j] : a[2 + j];
        b[j] = (b3 ? a[2 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? b[0] : b[1];
    return (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
}

// The column that colsum_frag leaves in lane t, relative to the fragment's first column.
__device__ __forceinline__ int colsum_frag_col(int lane) {
    const int c8 = lane >> 2;
    return 8 * (c8 >> 1) + 2 * (lane & 3) + (c8 & 1);
}

// Sum over the four lanes of a quad (the eight columns of one row that a fragment
// spreads over lanes 4q .. 4q + 3).
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// Sums over the 32 lanes of a warp of 32 values per lane, transposed: lane l ends with
// the sum over all lanes of x[l].  Five butterfly steps (16 + 8 + 4 + 2 + 1 shuffles):
// at the step of offset o a lane keeps the half of its values whose index has bit o
// equal to its own lane bit o, and adds the partner's copy of that half.  Fixed order.
__device__ __forceinline__ float lanesum16(const float (&a)[16], int lane);
__device__ __forceinline__ float lanesum32(const float (&x)[32], int lane) {
    float a[16];
    const bool hi = lane & 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float send = hi ? x[j] : x[16 + j];
        a[j] = (hi ? x[16 + j] : x[j]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    return lanesum16(a, lane);
}

// The last four steps of lanesum32, for values already halved by the offset-16 step:
// lane l holds, for j < 16, a partial of index (l & 16) + j; it ends with the sum
// over all lanes of index l.
__device__ __forceinline__ float lanesum16(const float (&a)[16], int lane) {
    float b[8], c[4], d[2];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const bool hi = lane & 8;
        const float send = hi ? a[j] : a[8 + j];
        b[j] = (hi ? a[8 + j] : a[j]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool hi = lane & 4;
        const float send = hi ? b[j] : b[4 + j];
        c[j] = (hi ? b[4 + j] : b[j]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const bool hi = lane & 2;
        const float send = hi ? c[j] : c[2 + j];
        d[j] = (hi ? c[2 + j] : c[j]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const bool hi = lane & 1;
    return (hi ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, hi ? d[0] : d[1], 1);
}

// bf16 pair (columns col, col + 1 of row `row`) into a 64-wide SW128 tile.
__device__ __forceinline__ void put_pair(unsigned char *tile, int row, int col, float a, float b) {
    *reinterpret_cast<uint32_t *>(tile + umma::sw128_off(row, col)) = pack_bf2(a, b);
}

__device__ __forceinline__ float2 get_pair(const unsigned char *tile, int row, int col) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(tile + umma::sw128_off(row, col)));
}

}  // namespace epi
}  // namespace gdn
