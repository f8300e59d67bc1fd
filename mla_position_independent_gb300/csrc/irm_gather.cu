// Standalone rotate+gather path: cached rows of a chunk pool are copied into a paged KV
// layout, cKV unchanged and k_r turned by R(delta) on the way ("Irminsul论文详解" §5: a
// registry hit contributes (cKV, R(delta) k_r,base); §4: only the 64-d slice is touched).
// Pure bandwidth: every row is read once (1152 B) and written once (1152 B) with 16-byte
// vector accesses; one CTA walks one chunk at a time so the chunk's 32 (cos, sin) pairs
// are computed once and the row addresses are contiguous on both sides.
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

__global__ void __launch_bounds__(kGatherThreads) rotate_gather_kernel(const GatherArgs a) {
  __shared__ float cs_c[32], cs_s[32];
  __shared__ int req_sh;
  const int tid = threadIdx.x;
  for (int64_t c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
    const irm_chunk ch = a.chunks[c];
    const int32_t delta = ch.reused ? ch.p_tgt - ch.p_src : 0;
    if (tid < 32) {
      float cc = 1.f, ss = 0.f;
      if (delta != 0) rope_cos_sin(delta, a.phase.F[tid], cc, ss);
      cs_c[tid] = cc;
      cs_s[tid] = ss;
    }
    if (tid == 0) {  // owning request: last b with indptr[b] <= c
      int lo = 0, hi = a.B;  // invariant indptr[lo] <= c < indptr[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.indptr[mid] <= c) lo = mid; else hi = mid;
      }
      req_sh = lo;
    }
    __syncthreads();
    const int b = req_sh;
    const int len = ch.len;
    // The table in the workspace is the validated one; these checks only keep a table that
    // was overwritten meanwhile (calls overlapping on one workspace) inside every buffer.
    bool src_ok = len > 0 && ch.p_tgt >= 0 && ch.pool_offset >= 0 && ch.pool_offset + len <= a.n_rows;
    if (a.paged_out != nullptr)
      src_ok = src_ok && (int64_t)ch.p_tgt + len <= (int64_t)a.max_pages * kPage;
    int64_t r0 = 0;
    if (a.out_src != nullptr && src_ok) {
      r0 = a.row_start[b] + ch.p_tgt;
      src_ok = r0 + len <= a.row_start[a.B];
    }
    if (!src_ok) {
      if (tid == 0) set_status(a.status, kDevErrBounds);
    }
    if (a.out_src != nullptr && src_ok) {
      for (int i = tid; i < len; i += kGatherThreads) {
        a.out_src[r0 + i] = (int32_t)(ch.pool_offset + i);
        a.out_delta[r0 + i] = delta;
        a.out_pos_src[r0 + i] = ch.p_tgt + i - delta;
      }
    }
    if (a.paged_out != nullptr && src_ok) {
      const uint4* src = reinterpret_cast<const uint4*>(a.kv) + ch.pool_offset * (kDRow / 8);
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
            const int t = ch.p_tgt + row;
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
        const int t = ch.p_tgt + row;
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
    __syncthreads();  // cs_c / req_sh reused by the next chunk
  }
}

// Copies up to three host arrays into a device block: the sources are page-locked host memory
// that the GPU reads directly (device-accessible addresses), in 4-byte words (every array is a
// whole number of them).  One launch instead of one copy-engine transfer per array.
__global__ void __launch_bounds__(256) host_copy_kernel(HostCopyArgs a) {
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
  if (a.n_chunks <= 0) return cudaSuccess;
  const int64_t want = (int64_t)num_sms * 8;
  const int grid = (int)(a.n_chunks < want ? a.n_chunks : want);
  rotate_gather_kernel<<<grid, kGatherThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irm
