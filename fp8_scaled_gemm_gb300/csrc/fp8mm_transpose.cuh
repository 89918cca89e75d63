// fp8mm_transpose.cuh -- byte transpose [R, C] -> [C, R], used to bring an
// operand stored with its M (or N) dimension contiguous into the K-contiguous
// layout the MMA kernels read.
//
// Tiles of 64 x 64 bytes pass through shared memory: 256 threads each load
// one 16-byte row segment of the tile (coalesced), and after the barrier each
// gathers one 16-byte segment of a column and stores it as a row segment of
// the output (coalesced). Edges and unaligned rows fall back to byte accesses.
// HBM-bound: one read and one write of every byte.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fp8t {

constexpr int kTile = 64;
constexpr int kThreads = 256;
constexpr int kPitch = kTile + 4;    // bytes per shared-memory row (bank spread)

struct TransposeParams {
    const uint8_t *in;      // [R, C] row-major
    uint8_t *out;           // [C, R] row-major
    long long R, C;
    long long tiles_r, tiles_c;
    int vec_in;             // rows of `in` are 16-byte aligned (C % 16 == 0, aligned base)
    int vec_out;            // rows of `out` are 16-byte aligned (R % 16 == 0, aligned base)
};

__global__ void __launch_bounds__(kThreads) transpose_u8_kernel(const TransposeParams p)
{
    __shared__ __align__(16) uint8_t t[kTile * kPitch];
    fp8mm::ptx::grid_launch_dependents();
    fp8mm::ptx::grid_dependency_wait();

    const int seg_row = static_cast<int>(threadIdx.x) >> 2;        // 0..63
    const int seg_col = (static_cast<int>(threadIdx.x) & 3) * 16;  // 0, 16, 32, 48
    const long long tiles = p.tiles_r * p.tiles_c;
    for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const long long r0 = (tile / p.tiles_c) * kTile;
        const long long c0 = (tile % p.tiles_c) * kTile;

        // load row segment (r0 + seg_row, c0 + seg_col .. +16)
        {
            const long long r = r0 + seg_row;
            const long long c = c0 + seg_col;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (r < p.R) {
                const uint8_t *src = p.in + r * p.C + c;
                if (p.vec_in && c + 16 <= p.C) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
                    w[0] = v.x;
                    w[1] = v.y;
                    w[2] = v.z;
                    w[3] = v.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c + j < p.C)
                            w[j >> 2] |= static_cast<uint32_t>(src[j]) << (8 * (j & 3));
                }
            }
            uint32_t *dst = reinterpret_cast<uint32_t *>(t + seg_row * kPitch + seg_col);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = w[j];
        }
        __syncthreads();

        // output row c0 + seg_row (an input column), columns r0 + seg_col .. +16
        {
            const long long orow = c0 + seg_row;
            const long long ocol = r0 + seg_col;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < 16; ++j)
                w[j >> 2] |= static_cast<uint32_t>(t[(seg_col + j) * kPitch + seg_row]) << (8 * (j & 3));
            if (orow < p.C) {
                uint8_t *dst = p.out + orow * p.R + ocol;
                if (p.vec_out && ocol + 16 <= p.R) {
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (ocol + j < p.R)
                            dst[j] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace fp8t
