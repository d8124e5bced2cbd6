// Operand images of the tensor-core V kernel, shared by the kernels that
// write them (relabel: the state tiles; pack: the weights) and the kernel
// that reads them.
//
// An image is a [rows x cols] matrix of bf16 stored as core matrices of
// 8 rows x 8 elements (16 bytes, 128 contiguous bytes each), chunk-major
// inside each 8-row group.  For fp32 workloads an image has three planes
// (x = x0 + x1 + x2, each the nearest bf16 of what is left); for the bf16
// workload one plane.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ofrl {
namespace tc {

constexpr int TM = 128;     // batch rows per tile
constexpr int HH = 128;     // hidden width handled by the tensor-core kernel
constexpr int KX = 64;      // state columns, zero-padded
constexpr uint32_t kPlaneH = TM * HH * 2;    // one plane of a [128 x 128] image
constexpr uint32_t kPlaneX = TM * KX * 2;    // one plane of a [128 x 64] image

// Byte offset of element (r, c) inside one plane of an image with C columns.
__host__ __device__ __forceinline__ uint32_t img_off(int r, int c, int C) {
    return (uint32_t)((r >> 3) * (C >> 3) * 128 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// Bytes of one network's packed weights: W1 image then W2 image, 3 planes.
__host__ __device__ constexpr int64_t weight_image_bytes() { return 3 * (int64_t)(kPlaneX + kPlaneH); }
// Bytes of one state-tile image (3 planes).
__host__ __device__ constexpr int64_t x_tile_bytes() { return 3 * (int64_t)kPlaneX; }

__device__ __forceinline__ void split3(float x, __nv_bfloat16& b0, __nv_bfloat16& b1, __nv_bfloat16& b2) {
    b0 = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(b0);
    b1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(b1);
    b2 = __float2bfloat16_rn(r2);
}

// Write 4 consecutive values of row r, columns c..c+3 (c a multiple of 4)
// into an image with C columns and np planes of `plane` bytes.
__device__ __forceinline__ void put4(uint8_t* img, uint32_t plane, int np, int C, int r, int c, const float (&x)[4]) {
    __nv_bfloat16 t[3][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (np == 3) split3(x[j], t[0][j], t[1][j], t[2][j]);
        else t[0][j] = __float2bfloat16_rn(x[j]);
    }
    const uint32_t o = img_off(r, c, C);
    for (int p = 0; p < np; ++p) *reinterpret_cast<uint2*>(img + (uint32_t)p * plane + o) = *reinterpret_cast<const uint2*>(&t[p][0]);
}

}  // namespace tc
}  // namespace ofrl
