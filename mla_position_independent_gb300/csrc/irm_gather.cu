// Standalone rotate+gather path: cached rows of a chunk pool are copied into a paged KV
// layout, cKV unchanged and k_r turned by R(delta) on the way ("Irminsul论文详解" §5: a
// registry hit contributes (cKV, R(delta) k_r,base); §4: only the 64-d slice is touched).
// Pure bandwidth: every row is read once (1152 B) and written once (1152 B) with 16-byte
// vector accesses; a CTA walks its range of rows chunk by chunk, so each chunk's 32
// (cos, sin) pairs are computed once per CTA and the row addresses are contiguous on both
// sides.
#include <cuda_runtime.h>

#include "irm_common.cuh"
#include "irm_internal.h"

namespace irm {

// Exclusive prefix sum of the context lengths: row_start[b] = sum_{b' < b} ctx_b'.
// One CTA; ctx_b = p_tgt + len of the request's last chunk (requests are non-empty).
__global__ void __launch_bounds__(1024) row_start_kernel(const irm_chunk* __restrict__ chunks,
                                                         const int32_t* __restrict__ indptr, int B,
                                                         int64_t* __restrict__ row_start) {
  __shared__ int64_t carry;
  __shared__ int64_t part[32];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int64_t v = 0;
    if (b < B) {
      const irm_chunk last = chunks[indptr[b + 1] - 1];
      v = (int64_t)last.p_tgt + last.len;
    }
    int64_t x = v;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) part[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t w = (lane < (int)(blockDim.x >> 5)) ? part[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      part[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t excl = carry + (warp > 0 ? part[warp - 1] : 0) + x - v;
    if (b < B) row_start[b] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) row_start[B] = carry;
}

constexpr int kGatherThreads = 256;
constexpr int kUnroll = 4;
constexpr int kMinRowsPerCta = 128;
constexpr int kGatherCtasPerSm = 4;  // resident CTAs per SM (64 registers a thread at most)

// The CTAs share the batch's rows (requests laid end to end) in equal contiguous ranges, so
// every CTA moves the same bytes whatever the chunk lengths (sharing whole chunks left the
// CTAs that drew the last long chunks running alone at the end).  A CTA finds the chunk that
// holds its first row, then walks the chunks in order, copying the part of each that lies
// in its range; (cos, sin) are computed once per chunk it visits.
__global__ void __launch_bounds__(kGatherThreads, kGatherCtasPerSm) rotate_gather_kernel(const __grid_constant__ GatherArgs a) {
  __shared__ float cs_c[32], cs_s[32];
  __shared__ int b_sh, c_sh;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t r_begin = (int64_t)blockIdx.x * a.total_rows / gridDim.x;
  const int64_t r_end = (int64_t)(blockIdx.x + 1) * a.total_rows / gridDim.x;
  if (r_begin >= r_end) return;
  const int64_t* rowb = a.inline_rows ? a.rows : a.row_start;
  if (tid < 32) {
    // the request holding row r_begin: last b with rowb[b] <= r_begin (requests are non-empty)
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rowb[mid] <= r_begin) lo = mid; else hi = mid;
    }
    // its chunk holding that row: last c with p_tgt <= r_begin - rowb[b], 32-fold per ballot
    const int32_t t0 = (int32_t)(r_begin - rowb[lo]);
    int cl = a.indptr[lo], ch = a.indptr[lo + 1];
    while (ch - cl > 1) {
      const int step = (ch - cl + 31) / 32;
      const int c = cl + lane * step;
      const bool le = c < ch && a.chunks[c].p_tgt <= t0;
      const unsigned m = __ballot_sync(0xffffffffu, le);
      const int k = m ? 31 - __clz((int)m) : 0;
      cl = cl + k * step;
      ch = min(ch, cl + step);
    }
    if (lane == 0) {
      b_sh = lo;
      c_sh = cl;
    }
  }
  __syncthreads();
  int b = b_sh;
  int c = c_sh;
  int64_t r = r_begin;
  const int n_chunks = (int)a.n_chunks;
  for (int guard = 0; r < r_end && c < n_chunks && b < a.B && guard < n_chunks; ++guard) {
    const irm_chunk chk = a.chunks[c];
    const int32_t delta = chk.reused ? chk.p_tgt - chk.p_src : 0;
    const int64_t g0 = rowb[b] + chk.p_tgt;  // the chunk's first row in the batch
    const int lo = (int)max((int64_t)0, r - g0);
    const int hi = (int)min((int64_t)chk.len, r_end - g0);
    if (tid < 32) {
      float cc = 1.f, ss = 0.f;
      if (delta != 0) rope_cos_sin(delta, a.phase.F[tid], cc, ss);
      cs_c[tid] = cc;
      cs_s[tid] = ss;
    }
    __syncthreads();
    // The table in the workspace is the validated one; these checks only keep a table that
    // was overwritten meanwhile (calls overlapping on one workspace) inside every buffer.
    bool src_ok = chk.len > 0 && chk.p_tgt >= 0 && chk.pool_offset >= 0 && chk.pool_offset + chk.len <= a.n_rows &&
                  g0 + chk.len <= a.total_rows;
    if (a.paged_out != nullptr)
      src_ok = src_ok && (int64_t)chk.p_tgt + chk.len <= (int64_t)a.max_pages * kPage;
    if (!src_ok) {
      if (tid == 0) set_status(a.status, kDevErrBounds);
    }
    if (src_ok && hi > lo) {
      const int len = hi - lo;
      const int64_t pool0 = chk.pool_offset + lo;
      const int32_t p0 = chk.p_tgt + lo;
      if (a.out_src != nullptr) {
        for (int i = tid; i < len; i += kGatherThreads) {
          a.out_src[g0 + lo + i] = (int32_t)(pool0 + i);
          a.out_delta[g0 + lo + i] = delta;
          a.out_pos_src[g0 + lo + i] = p0 + i - delta;
        }
      }
      if (a.paged_out != nullptr) {
        const uint4* src = reinterpret_cast<const uint4*>(a.kv) + pool0 * (kDRow / 8);
        uint4* dst = reinterpret_cast<uint4*>(a.paged_out);
        const int32_t* ptab = a.page_table + (int64_t)b * a.max_pages;
        // cKV: 64 16-byte vectors per row; 4 rows per pass of 256 threads, kUnroll passes.
        const int n_items = len * 64;
        for (int i0 = 0; i0 < n_items; i0 += kGatherThreads * kUnroll) {
          uint4 v[kUnroll];
          int64_t d_off[kUnroll];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int it = i0 + u * kGatherThreads + tid;
            d_off[u] = -1;
            if (it < n_items) {
              const int row = it >> 6, vec = it & 63;
              const int t = p0 + row;
              const int32_t page = ptab[t / kPage];
              if (page >= 0 && page < a.n_pages) {
                v[u] = __ldcs(src + (int64_t)row * (kDRow / 8) + vec);
                d_off[u] = ((int64_t)page * kPage + (t % kPage)) * (kDRow / 8) + vec;
              } else {
                set_status(a.status, kDevErrBounds);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u)
            if (d_off[u] >= 0) __stcs(dst + d_off[u], v[u]);
        }
        // k_r: a thread takes 16-byte vectors 64+pv and 68+pv of a row (NeoX: pairs 8pv..8pv+7,
        // first elements then partners; interleaved: the 4 pairs inside each vector).
        const int n_kr = len * 4;
        for (int it = tid; it < n_kr; it += kGatherThreads) {
          const int row = it >> 2, pv = it & 3;
          const int t = p0 + row;
          const int32_t page = ptab[t / kPage];
          if (page < 0 || page >= a.n_pages) continue;  // recorded by the cKV loop
          const uint4* s = src + (int64_t)row * (kDRow / 8) + 64;
          uint4 x = __ldcs(s + pv), y = __ldcs(s + 4 + pv);
          if (delta != 0) {
            float c8[8], s8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = pair_index(a.interleaved, pv, pv + 4, e);
              c8[e] = cs_c[j];
              s8[e] = cs_s[j];
            }
            rotate_pairs8_any(x, y, c8, s8, a.interleaved);
          }
          uint4* d = dst + ((int64_t)page * kPage + (t % kPage)) * (kDRow / 8) + 64;
          __stcs(d + pv, x);
          __stcs(d + 4 + pv, y);
        }
      }
    }
    __syncthreads();  // cs_c / cs_s are reused by the next chunk
    r = max(r, g0 + (chk.len > 0 ? chk.len : 1));
    if (++c >= a.indptr[b + 1]) ++b;
  }
}

// Copies up to three host arrays into a device block: the sources are page-locked host memory
// that the GPU reads directly (device-accessible addresses), in 4-byte words (every array is a
// whole number of them).  One launch instead of one copy-engine transfer per array.
__global__ void __launch_bounds__(256) host_copy_kernel(const __grid_constant__ HostCopyArgs a) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int p = 0; p < a.n; ++p) {
    const uint32_t* __restrict__ src = static_cast<const uint32_t*>(a.src[p]);
    uint32_t* __restrict__ dst = reinterpret_cast<uint32_t*>(a.dst + a.off[p]);
    const int64_t words = (int64_t)(a.bytes[p] / 4);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += stride) dst[i] = src[i];
  }
}

cudaError_t launch_host_copy(const HostCopyArgs& a, cudaStream_t stream) {
  size_t most = 0;
  for (int p = 0; p < a.n; ++p) most = a.bytes[p] > most ? a.bytes[p] : most;
  const int64_t words = (int64_t)(most / 4);
  const int grid = (int)(words < 256 ? 1 : (words + 255) / 256 < 1024 ? (words + 255) / 256 : 1024);
  host_copy_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_row_start(const irm_chunk* chunks, const int32_t* indptr, int B,
                             int64_t* row_start, cudaStream_t stream) {
  row_start_kernel<<<1, 1024, 0, stream>>>(chunks, indptr, B, row_start);
  return cudaGetLastError();
}

cudaError_t launch_rotate_gather(const GatherArgs& a, int num_sms, cudaStream_t stream) {
  if (a.n_chunks <= 0 || a.total_rows <= 0) return cudaSuccess;
  // one wave of resident CTAs, each with an equal share of the rows
  const int64_t want = (int64_t)num_sms * kGatherCtasPerSm;
  const int64_t by_rows = (a.total_rows + kMinRowsPerCta - 1) / kMinRowsPerCta;
  const int grid = (int)(by_rows < want ? by_rows : want);
  rotate_gather_kernel<<<grid, kGatherThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irm
