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

// A state-tile image ([128 x 64], S state columns zero-padded) holds 1.0 in
// its last column when S < 64: the W1 image is zero there, so z1 is
// unchanged, and the weight-gradient GEMM dz1^T X then also yields the bias
// gradient sum_rows dz1 in that column.  Rows past the batch stay all zero.
__host__ __device__ __forceinline__ bool ones_column(int c, int S) { return S < KX && c == KX - 1; }

// Byte offset of element (r, c) inside one plane of an image with C columns.
__host__ __device__ __forceinline__ uint32_t img_off(int r, int c, int C) {
    return (uint32_t)((r >> 3) * (C >> 3) * 128 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

// Bytes of one network's packed weights for hidden width H: the W1 image
// ([H x 64]) then the W2 image ([H x H]), room for 3 planes each.
__host__ __device__ constexpr int64_t weight_image_bytes(int H = HH) { return 3 * 2 * (int64_t)H * (KX + H); }
// Offset of the W2 image inside them.
__host__ __device__ constexpr int64_t w2_image_offset(int H = HH) { return 3 * 2 * (int64_t)H * KX; }
// Bytes of one state-tile image (3 planes).
__host__ __device__ constexpr int64_t x_tile_bytes() { return 3 * (int64_t)kPlaneX; }

// Two fp32 values to a bf16 pair in one register (round to nearest even):
// lo in bits 0-15 (the lower address in memory), hi in bits 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// Split a pair of fp32 values into three bf16 pairs, x = x0 + x1 + x2, each
// term the nearest bf16 of what the previous terms leave.
__device__ __forceinline__ void split3x2(float a, float b, uint32_t& p0, uint32_t& p1, uint32_t& p2) {
    p0 = pack_bf16x2(a, b);
    a -= bf16_lo(p0);
    b -= bf16_hi(p0);
    p1 = pack_bf16x2(a, b);
    a -= bf16_lo(p1);
    b -= bf16_hi(p1);
    p2 = pack_bf16x2(a, b);
}

// The first two of those terms only (x0 + x1: 16 significand bits), for
// operands that only the three leading products read.
__device__ __forceinline__ void split2x2(float a, float b, uint32_t& p0, uint32_t& p1) {
    p0 = pack_bf16x2(a, b);
    a -= bf16_lo(p0);
    b -= bf16_hi(p0);
    p1 = pack_bf16x2(a, b);
}

// Write 4 consecutive values of row r, columns c..c+3 (c a multiple of 4)
// into an image with C columns and np planes of `plane` bytes.
__device__ __forceinline__ void put4(uint8_t* img, uint32_t plane, int np, int C, int r, int c, const float (&x)[4]) {
    const uint32_t o = img_off(r, c, C);
    if (np == 3) {
        uint32_t a0, a1, a2, b0, b1, b2;
        split3x2(x[0], x[1], a0, a1, a2);
        split3x2(x[2], x[3], b0, b1, b2);
        *reinterpret_cast<uint2*>(img + o) = make_uint2(a0, b0);
        *reinterpret_cast<uint2*>(img + plane + o) = make_uint2(a1, b1);
        *reinterpret_cast<uint2*>(img + 2 * plane + o) = make_uint2(a2, b2);
    } else {
        *reinterpret_cast<uint2*>(img + o) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    }
}

}  // namespace tc
}  // namespace ofrl
