// Device-side definitions shared by the library's kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/irm.h"
#include "ptx.cuh"

namespace irm {

constexpr int kDLat = IRM_D_LAT;
constexpr int kDRope = IRM_D_ROPE;
constexpr int kDRow = IRM_D_ROW;
constexpr int kPage = IRM_PAGE_ROWS;

// Bits of the device status word (first word of every workspace).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBounds = 2;

// RoPE phase increments: F[j] = round(theta_j / (2 pi) * 2^64), theta_j = 10000^(-2j/64).
// The phase of position offset delta is (delta * F[j]) mod 2^64 in units of 2^-64 turns,
// which is exact integer arithmetic for every int32 delta; only the final conversion of
// the top 32 bits to an angle in [-pi, pi) is rounded (fixed-point phase accumulation).
struct RopePhase {
  uint64_t F[32];
};

// cos/sin of delta * theta_j, angle reduced exactly to one turn before the fp32 sincos.
__device__ __forceinline__ void rope_cos_sin(int32_t delta, uint64_t F, float& c, float& s) {
  const uint64_t ph = (uint64_t)(int64_t)delta * F;          // wraps modulo 2^64 = one turn
  const int32_t hi = (int32_t)(ph >> 32);                    // turns in [-1/2, 1/2) * 2^32
  const float ang = (float)hi * 1.4629180792671596e-9f;      // * 2 pi / 2^32 -> [-pi, pi)
  __sincosf(ang, &s, &c);
}

// Rotates one NeoX pair-vector: x holds k_r[8v .. 8v+7], y holds k_r[32+8v .. 32+8v+7]
// (bf16, 16 bytes each).  Pair e couples x[e] and y[e] with frequency index j = 8v + e.
__device__ __forceinline__ void rotate_pairs8(uint4& x, uint4& y, const float* cs_c,
                                              const float* cs_s) {
  __nv_bfloat162* xp = reinterpret_cast<__nv_bfloat162*>(&x);
  __nv_bfloat162* yp = reinterpret_cast<__nv_bfloat162*>(&y);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 xf = __bfloat1622float2(xp[q]);
    const float2 yf = __bfloat1622float2(yp[q]);
    const float c0 = cs_c[2 * q], s0 = cs_s[2 * q], c1 = cs_c[2 * q + 1], s1 = cs_s[2 * q + 1];
    const float x0 = fmaf(xf.x, c0, -yf.x * s0), y0 = fmaf(xf.x, s0, yf.x * c0);
    const float x1 = fmaf(xf.y, c1, -yf.y * s1), y1 = fmaf(xf.y, s1, yf.y * c1);
    xp[q] = __floats2bfloat162_rn(x0, x1);
    yp[q] = __floats2bfloat162_rn(y0, y1);
  }
}

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

}  // namespace irm
