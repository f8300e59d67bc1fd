// Pieces of the KV gather pipeline shared by the attention kernels: the chunk-table window
// that turns target positions into source rows and deltas, and the in-shared-memory
// rotation of a staged k_r slab by R(delta) ("Irminsul论文详解" §4 δ-rotation; technical
// summary §2.2).
#pragma once
#include <climits>
#include <cstdint>

#include "irm_common.cuh"

namespace irm {

constexpr uint32_t kFullMask = 0xffffffffu;

// A warp's window of 32 consecutive chunk records of one request (one record per lane).
struct ChunkWindow {
  const irm_chunk* chunks;
  int c_end;  // one past the request's last chunk
  int win;    // first chunk of the window
  int start, end, delta;
  long long off;

  __device__ __forceinline__ void load(int lane) {
    const int c = win + lane;
    if (c < c_end) {
      const irm_chunk ch = chunks[c];
      start = ch.p_tgt;
      end = ch.p_tgt + ch.len;
      off = ch.pool_offset;
      delta = ch.reused ? ch.p_tgt - ch.p_src : 0;
    } else {
      start = end = INT_MAX;
      off = 0;
      delta = 0;
    }
  }

  // Position the window at the last chunk with p_tgt <= T0 (chunks tile the context in
  // target order), narrowing [c_begin, c_end) 32-fold per step with one ballot.
  __device__ __forceinline__ void seek(int c_begin, int T0, int lane) {
    int lo = c_begin, hi = c_end;
    while (hi - lo > 32) {
      const int step = (hi - lo + 31) / 32;
      const int c = lo + lane * step;
      const bool le = (c < hi) && (chunks[c].p_tgt <= T0);
      const unsigned msk = __ballot_sync(kFullMask, le);
      const int k = msk ? 31 - __clz((int)msk) : 0;
      lo = lo + k * step;
      hi = min(hi, lo + step);
    }
    win = lo;
    load(lane);
  }

  // Row map of the 64-row tile starting at target position T: src[r] = source row of
  // position T + r (-1 past the context: zero filled), dl[r] = its delta.  The few window
  // chunks overlapping the tile are found with one ballot and broadcast in turn; the window
  // slides forward when the tile runs past it.  A table that does not cover the context or
  // points outside the row store sets the bounds bit of `status`.
  __device__ __forceinline__ void build_map(int T, int ctx, int64_t n_rows, int32_t* src, int32_t* dl,
                                            int* status, int lane) {
    const int t0 = T + lane, t1 = T + lane + 32;
    const int t_end = min(T + 64, ctx);
    int src0 = -1, src1 = -1, d0 = 0, d1 = 0;
    for (int guard = 0; guard < 65 && T < t_end; ++guard) {
      const int nvalid = min(32, c_end - win);
      if (nvalid <= 0) {
        if (lane == 0) set_status(status, kDevErrBounds);
        break;
      }
      unsigned ov = __ballot_sync(kFullMask, lane < nvalid && start < t_end && end > T);
      while (ov != 0u) {
        const int k = __ffs(ov) - 1;
        ov &= ov - 1u;
        const int st = __shfl_sync(kFullMask, start, k), en = __shfl_sync(kFullMask, end, k);
        const long long of = __shfl_sync(kFullMask, off, k);
        const int dd = __shfl_sync(kFullMask, delta, k);
        if (t0 >= st && t0 < en && t0 < t_end) {
          const long long r = of + (t0 - st);
          if (r < 0 || r >= n_rows) set_status(status, kDevErrBounds); else src0 = (int)r;
          d0 = dd;
        }
        if (t1 >= st && t1 < en && t1 < t_end) {
          const long long r = of + (t1 - st);
          if (r < 0 || r >= n_rows) set_status(status, kDevErrBounds); else src1 = (int)r;
          d1 = dd;
        }
      }
      const int last_end = __shfl_sync(kFullMask, end, nvalid - 1);
      if (last_end >= t_end) break;
      win += nvalid;
      load(lane);
    }
    src[lane] = src0;
    src[lane + 32] = src1;
    dl[lane] = d0;
    dl[lane + 32] = d1;
  }
};

// Rotate 8 rows [r0, r0 + 8) of a staged k_r slab by R(delta[row]) with one warp: a lane takes
// chunks v and v + 4 of one row (NeoX: k_r[8v .. 8v+7] and their partners k_r[32+8v .. 32+8v+7];
// interleaved: the 4 pairs inside each chunk).  A 16-byte access is served a quarter-warp at a
// time, so the 8 lanes of a quarter take rows p and p + 4 (r0 a multiple of 8): their swizzled
// chunk positions v ^ p and v ^ (p + 4) are 8 distinct ones, every bank once.
// dprev / cs_c / cs_s carry the lane's last (cos, sin) between calls (recomputed only when the
// row's delta changes; chunks are runs of equal delta).
__device__ __forceinline__ void rotate_krope_8rows(uint8_t* kr, const int32_t* delta, const uint64_t* phaseF,
                                                   int interleaved, int r0, int lane, int& dprev,
                                                   float (&cs_c)[8], float (&cs_s)[8]) {
  const int r = r0 + (lane >> 3) + 4 * ((lane >> 2) & 1), v = lane & 3;
  const int d = delta[r];
  if (d == 0) return;
  if (d != dprev) {
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin(d, phaseF[pair_index(interleaved, v, v + 4, e)], cs_c[e], cs_s[e]);
    dprev = d;
  }
  uint4* px = reinterpret_cast<uint4*>(kr + r * 128 + (((uint32_t)v ^ (uint32_t)(r & 7)) << 4));
  uint4* py = reinterpret_cast<uint4*>(kr + r * 128 + (((uint32_t)(4 + v) ^ (uint32_t)(r & 7)) << 4));
  uint4 x = *px, y = *py;
  rotate_pairs8_any(x, y, cs_c, cs_s, interleaved);
  *px = x;
  *py = y;
}

// The four 16-byte k_r chunks CTA `rank` of a column-split pair holds (stored chunk c =
// 0..3 of its half slab): NeoX, pairs 16 rank .. 16 rank + 15 as chunks 2 rank, 2 rank + 1
// (their first elements) and 4 + 2 rank, 5 + 2 rank (their partners); interleaved, the
// same pairs as the contiguous chunks 4 rank .. 4 rank + 3.
__device__ __forceinline__ int half_chunk(int interleaved, int rank, int c) {
  return interleaved ? 4 * rank + c : (c < 2 ? 2 * rank + c : 4 + 2 * rank + (c - 2));
}

// Rotate 16 rows [r0, r0 + 16) of a staged half k_r slab (a CTA's 16 pairs per row, stored as
// the chunks half_chunk(., rank, 0..3) at swizzled chunk positions cb .. cb + 3; cb = 0 or 4,
// two stages share a slab).  A lane takes stored chunks c and c + 2 of one row; the 8 lanes of a
// quarter-warp (one 16-byte access phase) share c and take 8 consecutive rows (r0 a multiple of
// 16), so their swizzled positions (cb + c) ^ (r & 7) are 8 distinct ones, every bank once.
// dprev / cs_c / cs_s carry the lane's last (cos, sin) between calls.
__device__ __forceinline__ void rotate_krope_half_16rows(uint8_t* kr, const int32_t* delta, const uint64_t* phaseF,
                                                         int interleaved, int rank, int r0, int cb, int lane,
                                                         int& dprev, float (&cs_c)[8], float (&cs_s)[8]) {
  const int r = r0 + (lane & 7) + 8 * (lane >> 4), c = (lane >> 3) & 1;
  const int d = delta[r];
  if (d == 0) return;
  if (d != dprev) {
    const int ga = half_chunk(interleaved, rank, c), gb = half_chunk(interleaved, rank, c + 2);
#pragma unroll
    for (int e = 0; e < 8; ++e) rope_cos_sin(d, phaseF[pair_index(interleaved, ga, gb, e)], cs_c[e], cs_s[e]);
    dprev = d;
  }
  uint4* px = reinterpret_cast<uint4*>(kr + r * 128 + (((uint32_t)(cb + c) ^ (uint32_t)(r & 7)) << 4));
  uint4* py = reinterpret_cast<uint4*>(kr + r * 128 + (((uint32_t)(cb + 2 + c) ^ (uint32_t)(r & 7)) << 4));
  uint4 x = *px, y = *py;
  rotate_pairs8_any(x, y, cs_c, cs_s, interleaved);
  *px = x;
  *py = y;
}

// Warp-uniform bounded waits: every lane polls (and so acquires) the barrier, and the
// verdict is agreed with __all_sync so no lane leaves a loop its warp-mates stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(kFullMask, ok);
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort_flag) {
  const bool ok = mbar_wait_cluster(bar, parity, abort_flag);
  return __all_sync(kFullMask, ok);
}

// Element-wise round_f32(a + b) of two fp16 pairs (low halves first), with the mixed-precision
// add of sm_100 and later: the first add widens b exactly, the second rounds once.  The result
// does not depend on which pair is a and which is b.
__device__ __forceinline__ float2 add_f16x2_f16x2_f32(uint32_t a, uint32_t b) {
  float2 r;
  asm("{\n .reg .f16 a0, a1, b0, b1;\n .reg .f32 t0, t1;\n"
      " mov.b32 {a0, a1}, %2;\n mov.b32 {b0, b1}, %3;\n"
      " add.rn.f32.f16 t0, b0, 0f00000000;\n add.rn.f32.f16 t1, b1, 0f00000000;\n"
      " add.rn.f32.f16 %0, a0, t0;\n add.rn.f32.f16 %1, a1, t1;\n}\n"
      : "=f"(r.x), "=f"(r.y)
      : "r"(a), "r"(b));
  return r;
}

// max(a, b, c) in one instruction (three-input form of max.f32 on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace irm
