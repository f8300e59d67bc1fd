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

// Interleaved pairing: rotates the 4 pairs (v[2i], v[2i+1]) held in one 16-byte chunk.
__device__ __forceinline__ void rotate_pairs4_within(uint4& v, const float* cs_c, const float* cs_s) {
  __nv_bfloat162* vp = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(vp[q]);
    const float x = fmaf(f.x, cs_c[q], -f.y * cs_s[q]), y = fmaf(f.x, cs_s[q], f.y * cs_c[q]);
    vp[q] = __floats2bfloat162_rn(x, y);
  }
}

// A lane rotates 8 pairs held in two 16-byte k_r chunks: chunk a (as x) and chunk b (as y).
// Frequency index of its pair e (0..7): NeoX half split (b = a + 4), pair e = (x[e], y[e]),
// index 8a + e; interleaved, pairs 0-3 = (x[2i], x[2i+1]), index 4a + i, and pairs 4-7 =
// (y[2i], y[2i+1]), index 4b + i.
__device__ __forceinline__ int pair_index(int interleaved, int a, int b, int e) {
  return interleaved ? (e < 4 ? 4 * a + e : 4 * b + (e - 4)) : 8 * a + e;
}
__device__ __forceinline__ void rotate_pairs8_any(uint4& x, uint4& y, const float* cs_c, const float* cs_s,
                                                  int interleaved) {
  if (interleaved) {
    rotate_pairs4_within(x, cs_c, cs_s);
    rotate_pairs4_within(y, cs_c + 4, cs_s + 4);
  } else {
    rotate_pairs8(x, y, cs_c, cs_s);
  }
}

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

}  // namespace irm
