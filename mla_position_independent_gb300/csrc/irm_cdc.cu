// Content-defined chunking of token streams on the GPU ("Irminsul: MLA-Native
// Position-Independent Caching for Agentic LLM Serving" technical summary §2.2: a rolling
// Gear hash over 64-token windows emits chunk boundaries, each chunk is fingerprinted with
// xxHash64; "Irminsul论文详解" §6: 7-bit boundary test, chunk length clipped to [32, 512]).
//
//   h_i = sum_{k<64, k<=i} G[x_{i-k}] 2^k  (mod 2^64),  i.e.  h_i = 2 h_{i-1} + G[x_i]
//   candidate(i): top `bits` bits of h_i zero (threshold reading) or low `bits` bits zero
//   a chunk from s ends at the first candidate i >= s + min_len - 1, else at s + max_len - 1,
//   else at the stream's end.
//
// Passes:
//   1. cdc_hash_kernel (grid-wide): a warp takes runs of 128-position steps of one stream,
//      4 positions per lane, and forms all hashes with one 4-step shuffle scan per step (see
//      the kernel); the candidate tests become bitmask words by shuffle-OR of lane nibbles.
//   2. The chunk boundaries depend on where the previous chunk started, so they are resolved
//      from the bitmask in order, one ballot per chunk (next_end: the words covering
//      [start + min_len - 1, start + max_len - 1] masked, then a find-first-set).  To use the
//      whole GPU on long streams the walk is speculative: cdc_spec_kernel walks every
//      4096-token segment with its own warp (its bitmask words staged in shared memory) as if a chunk started at the segment start, and
//      records its chunk ends; cdc_fixup_kernel (one warp per stream) then follows the true
//      chain: entering a segment at its true start, it re-walks only until it reaches one of
//      the segment's speculative ends (from then on both walks agree, usually after one or
//      two chunks) and copies the rest.
//   3. cdc_fingerprint_kernel: four lanes per chunk (one per xxHash64 accumulator), xxHash64
//      of its token ids as little-endian int32 bytes.
// Token ids outside the Gear table are read as G = 0 and recorded in the status word.
#include <cuda_runtime.h>
#include <climits>

#include "irm_common.cuh"
#include "irm_internal.h"

namespace irm {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kHashWarps = 8;          // warps per block of the hash pass

// Gear word of token t from SplitMix64 (Steele, Lea, Flood 2014): the generator's (t+1)-th
// output for the seed, its state seed + (t + 1) * gamma passed through the output mix.
__device__ __forceinline__ uint64_t splitmix_word(uint64_t seed, int32_t t) {
  uint64_t z = seed + (uint64_t)(t + 1) * 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ bool cdc_candidate(uint64_t h, int bits, int mode) {
  return mode == 1 ? (h & ((1ull << bits) - 1ull)) == 0ull : (h >> (64 - bits)) == 0ull;
}

constexpr int kSeg = 4096;                           // tokens per speculative walk segment
constexpr int kWinWords = (kSeg + 1024) / 32;         // bitmask words a walk keeps in shared memory

// Prefix sums over streams (two blocks): slot_base[s] = sum_{s' < s} (len_s' / min_len + 1)
// (output slots) and seg_base[s] = sum_{s' < s} ceil(len_s' / kSeg) (speculative segments).
__global__ void __launch_bounds__(1024) cdc_base_kernel(const int64_t* __restrict__ offsets, int S,
                                                        int min_len, int64_t* __restrict__ slot_base,
                                                        int64_t* __restrict__ seg_base) {
  const int seg = blockIdx.x;  // block 0: output slots, block 1: speculative segments
  int64_t* base = seg ? seg_base : slot_base;
  __shared__ int64_t carry;
  __shared__ int64_t part[32];
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int b0 = 0; b0 < S; b0 += blockDim.x) {
    const int s = b0 + threadIdx.x;
    const int64_t ln = s < S ? offsets[s + 1] - offsets[s] : 0;
    const int64_t v = s < S ? (seg ? (ln + kSeg - 1) / kSeg : ln / min_len + 1) : 0;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) part[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t w = lane < (int)(blockDim.x >> 5) ? part[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += y;
      }
      part[lane] = w;
    }
    __syncthreads();
    const int64_t excl = carry + (warp > 0 ? part[warp - 1] : 0) + x - v;
    if (s < S) base[s] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + v;
    __syncthreads();
  }
  if (threadIdx.x == 0) base[S] = carry;
}

// A warp takes a run of kRunSteps steps of 128 positions of one stream, lane l holding the
// 4 consecutive positions 4l .. 4l+3 of a step.  With g0..g3 their Gear words, the lane's block
// contributes L = 8 g0 + 4 g1 + 2 g2 + g3 to the hash at its last position, and a 4-step
// shuffle scan X_l = sum_{j <= l} L_j 2^(4 (l - j)) gives the hash there:
// h(4l+3) = h_prev 2^(4l+4) + X_l (terms shifted by 64 or more vanish).  The lane then steps
// h = 2 h + g through its own 4 positions from h(4l-1).  The step before the run (its 128
// positions include the 64 the run's first hash depends on) is hashed the same way, first.
constexpr int kRunSteps = 4;
__device__ __forceinline__ uint64_t gear_word(const CdcArgs& a, int32_t x, int* bad) {
  if (x < 0 || x >= a.vocab) {
    *bad = 1;
    return 0;
  }
  return a.gear != nullptr ? __ldg(a.gear + x) : splitmix_word(a.gear_seed, x);
}

__global__ void __launch_bounds__(32 * kHashWarps) cdc_hash_kernel(const CdcArgs a) {
  const int s = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t off = a.offsets[s], len = a.offsets[s + 1] - off;
  const int64_t nsteps = (len + 127) / 128;
  const int64_t r0 = ((int64_t)blockIdx.x * kHashWarps + warp) * kRunSteps;
  if (r0 >= nsteps) return;
  const int32_t* tok = a.tokens + off;
  uint32_t* words = a.words + (off >> 5) + s;  // word base of the stream (see the header)
  const int64_t nwords = (len + 31) / 32;
  int bad = 0;
  uint64_t h_prev = 0;
  const int64_t r1 = min(nsteps, r0 + kRunSteps);
  for (int64_t r = (r0 > 0 ? r0 - 1 : 0); r < r1; ++r) {
    const int64_t p = 128 * r + 4 * lane;  // the lane's first position
    uint64_t g[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) g[e] = p + e < len ? gear_word(a, __ldg(tok + p + e), &bad) : 0ull;
    uint64_t x = (g[0] << 3) + (g[1] << 2) + (g[2] << 1) + g[3];
#pragma unroll
    for (int d = 1; d < 16; d <<= 1) {  // shifts 4, 8, 16, 32 (the shift-64 step vanishes)
      const uint64_t y = __shfl_up_sync(kFull, x, d);
      if (lane >= d) x += y << (4 * d);
    }
    const uint64_t h_last = (lane < 15 ? (h_prev << (4 * lane + 4)) : 0ull) + x;
    uint64_t h = __shfl_up_sync(kFull, h_last, 1);  // hash at position 4l - 1
    if (lane == 0) h = h_prev;
    uint32_t nib = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h = (h << 1) + g[e];
      if (p + e < len && cdc_candidate(h, a.bits, a.mode)) nib |= 1u << e;
    }
    // word j of the step collects the nibbles of lanes 8j .. 8j+7
    uint32_t wv = nib << (4 * (lane & 7));
    wv |= __shfl_xor_sync(kFull, wv, 1);
    wv |= __shfl_xor_sync(kFull, wv, 2);
    wv |= __shfl_xor_sync(kFull, wv, 4);
    if (r >= r0 && (lane & 7) == 0) {
      const int64_t w = 4 * r + (lane >> 3);
      if (w < nwords) words[w] = wv;
    }
    h_prev = __shfl_sync(kFull, h_last, 31);
  }
  if (__any_sync(kFull, bad) && lane == 0) set_status(a.status, kDevErrBounds);
}

// Candidate bitmask of a stream as a warp reads it: words [win0, win0 + nwin) from a copy
// in shared memory, the rest from global memory.
struct WordSrc {
  const uint32_t* g;  // global words of the stream
  const uint32_t* win;
  int64_t win0, nwin;
  __device__ __forceinline__ uint32_t operator()(int w) const {
    const int r = w - (int)win0;
    return (r >= 0 && r < (int)nwin) ? win[r] : __ldg(g + w);
  }
};

// End of the chunk that starts at stream-local position t (t < len): the first candidate in
// [t + min_len - 1, min(t + max_len - 1, len - 1)], else that upper limit.  Warp-uniform.
__device__ __forceinline__ int next_end(const WordSrc& words, int len, int t, int min_len, int max_len,
                                        int lane) {
  // 32-bit positions: a stream holds at most INT32_MAX tokens and max_len <= 65536
  const int lo = t + min_len - 1, last = (int)min((int64_t)t + max_len - 1, (int64_t)len - 1);
  if (lo > last) return last;
  const int wl = last >> 5;
  for (int w0 = lo >> 5; w0 <= wl; w0 += 32) {
    const int w = w0 + lane;
    uint32_t m = w <= wl ? words(w) : 0u;
    const int p0 = 32 * w;
    if (lo > p0) m &= ~0u << (uint32_t)(lo - p0);  // only the lane of word lo >> 5: lo - p0 < 32
    if (last < p0 + 31) m &= last < p0 ? 0u : (last - p0 == 31 ? ~0u : (1u << (uint32_t)(last - p0 + 1)) - 1u);
    const uint32_t any = __ballot_sync(kFull, m != 0u);
    if (any != 0u) {
      const int src = __ffs(any) - 1;
      const uint32_t mw = __shfl_sync(kFull, m, src);
      return 32 * (w0 + src) + (__ffs(mw) - 1);
    }
  }
  return last;
}

// Speculative walk of one segment: chunk ends from a chunk start at the segment start until
// a chunk ends at or past the segment's last position.
__global__ void __launch_bounds__(128) cdc_spec_kernel(const CdcArgs a, int64_t n_segs) {
  __shared__ uint32_t win_sh[4][kWinWords];
  const int64_t g = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (g >= n_segs) return;
  int lo = 0, hi = a.S;  // stream owning segment g: last s with seg_base[s] <= g
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.seg_base[mid] <= g) lo = mid; else hi = mid;
  }
  const int s = lo;
  const int64_t k = g - a.seg_base[s];
  const int64_t off = a.offsets[s], len = a.offsets[s + 1] - off;
  const int64_t seg_end = min(len, (k + 1) * kSeg);  // one past the segment
  // the segment's bitmask words (and those a chunk crossing its end reads) to shared memory
  uint32_t* win = win_sh[threadIdx.x >> 5];
  const int64_t nwords = (len + 31) / 32, wbeg = k * kSeg / 32;
  const int64_t nwin = min((int64_t)kWinWords, nwords - wbeg);
  const uint32_t* gw = a.words + (off >> 5) + s;
  for (int64_t r = lane; r < nwin; r += 32) win[r] = __ldg(gw + wbeg + r);
  __syncwarp();
  const WordSrc words{gw, win, wbeg, nwin};
  int32_t* ends = a.spec_ends + g * a.spec_cap;
  int64_t t = k * kSeg, c = 0;
  while (t < seg_end && c < a.spec_cap) {
    const int64_t e = next_end(words, len, t, a.min_len, a.max_len, lane);
    if (lane == 0) ends[c] = (int32_t)e;
    ++c;
    t = e + 1;
  }
  if (lane == 0) a.spec_count[g] = (int32_t)c;
}

// The true chain of one stream: re-walk from the true start of each segment until a
// speculative end of that segment is met, then take the segment's remaining ends.
constexpr int kFixWin = 64;  // bitmask words the fix-up keeps for a segment's first 2048 positions
__global__ void __launch_bounds__(128) cdc_fixup_kernel(const CdcArgs a) {
  __shared__ uint32_t win_sh[4][kFixWin];
  const int s = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (s >= a.S) return;
  const int64_t off = a.offsets[s], len = a.offsets[s + 1] - off;
  const uint32_t* gw = a.words + (off >> 5) + s;
  uint32_t* win = win_sh[threadIdx.x >> 5];
  const int64_t cb = a.base[s], gb = a.seg_base[s];
  const int64_t nseg = (len + kSeg - 1) / kSeg;
  const int64_t nwords = (len + 31) / 32;
  // What segment k needs first (its speculative end count, first 32 ends and the bitmask of
  // its first 2048 positions) is loaded one segment ahead, so those loads overlap the work
  // on the segment before.
  uint32_t pa = 0, pb = 0;
  int32_t pend = INT_MAX;
  int pcnt = 0;
  auto prefetch = [&](int64_t k) {
    if (k >= nseg) return;
    const int64_t w0 = k * kSeg / 32;
    pa = w0 + lane < nwords ? __ldg(gw + w0 + lane) : 0u;
    pb = w0 + 32 + lane < nwords ? __ldg(gw + w0 + 32 + lane) : 0u;
    pcnt = a.spec_count[gb + k];
    pend = lane < a.spec_cap ? a.spec_ends[(gb + k) * a.spec_cap + lane] : INT_MAX;
  };
  prefetch(0);
  int64_t t = 0, count = 0;
  auto emit = [&](int64_t start, int64_t e) {
    if (lane == 0) {
      a.chunk_start[cb + count] = (int32_t)start;
      a.chunk_len[cb + count] = (int32_t)(e - start + 1);
    }
    ++count;
  };
  for (int64_t k = 0; k < nseg && t < len; ++k) {
    const int64_t seg_end = min(len, (k + 1) * kSeg);
    const int nspec = pcnt;
    const int32_t first = pend;
    __syncwarp();
    win[lane] = pa;
    win[32 + lane] = pb;
    __syncwarp();
    prefetch(k + 1);
    if (t >= seg_end) continue;  // a chunk longer than a segment covers this one
    const int32_t* ends = a.spec_ends + (gb + k) * a.spec_cap;
    const WordSrc words{gw, win, k * kSeg / 32, min((int64_t)kFixWin, nwords - k * kSeg / 32)};
    // re-walk until a chunk ends where a speculative one does (the segment-start case
    // agrees from its first chunk: both walks start at the same place)
    int p = 0;  // first speculative end not below the last true end
    bool met = false;
    if (t == k * kSeg) {
      met = true;
      p = -1;
    }
    // the segment's speculative ends, 32 at a time in registers (lane i: ends[sb + i])
    int sb = 0;
    int32_t mine = lane < nspec ? first : INT_MAX;
    while (!met && t < seg_end) {
      const int64_t e = next_end(words, len, t, a.min_len, a.max_len, lane);
      emit(t, e);
      t = e + 1;
      for (;;) {  // first speculative end >= e
        const uint32_t ge = __ballot_sync(kFull, mine >= e);
        if (ge != 0u) {
          const int i = __ffs(ge) - 1;
          p = sb + i;
          met = __shfl_sync(kFull, mine, i) == e;
          break;
        }
        sb += 32;
        if (sb >= nspec) {
          p = nspec;
          break;
        }
        mine = sb + lane < nspec ? ends[sb + lane] : INT_MAX;
      }
    }
    if (met) {
      // speculative chunks after index p (all of them when p == -1) are the true ones
      for (int i0 = p + 1; i0 < nspec; i0 += 32) {
        const int i = i0 + lane;
        if (i < nspec) {
          const int64_t st = i == 0 ? k * kSeg : (int64_t)ends[i - 1] + 1;
          a.chunk_start[cb + count + (i - (p + 1))] = (int32_t)st;
          a.chunk_len[cb + count + (i - (p + 1))] = (int32_t)(ends[i] - st + 1);
        }
      }
      if (nspec > p + 1) {
        count += nspec - (p + 1);
        t = (int64_t)ends[nspec - 1] + 1;
      }
    }
  }
  if (lane == 0) a.n_chunks[s] = (int32_t)count;
}

// xxHash64 (four 64-bit lanes over 32-byte stripes, lane merge, 8/4/1-byte tails, final
// avalanche) of the chunk's token ids as little-endian int32 bytes.
constexpr uint64_t kP1 = 11400714785074694791ull, kP2 = 14029467366897019727ull,
                   kP3 = 1609587929392839161ull, kP4 = 9650029242287828579ull,
                   kP5 = 2870177450012600261ull;
__device__ __forceinline__ uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
__device__ __forceinline__ uint64_t xx_round(uint64_t acc, uint64_t v) { return rotl(acc + v * kP2, 31) * kP1; }
__device__ __forceinline__ uint64_t pair64(const int32_t* p) {
  return (uint64_t)(uint32_t)__ldg(p) | ((uint64_t)(uint32_t)__ldg(p + 1) << 32);
}

// xxHash64 of n token ids by 4 cooperating lanes (q = lane & 3 owns accumulator v_{q+1}, i.e.
// bytes 8q .. 8q + 7 of every 32-byte stripe); the group's lane 0 merges the accumulators,
// hashes the tail and returns the result (other lanes return 0).
__device__ uint64_t chunk_xxh64_x4(const int32_t* __restrict__ t, int n, uint64_t seed, int q,
                                   uint32_t gmask, int src0) {
  const int64_t bytes = 4 * (int64_t)n;
  const int stripes = n / 8;
  uint64_t h = 0;
  if (bytes >= 32) {
    uint64_t v = q == 0 ? seed + kP1 + kP2 : q == 1 ? seed + kP2 : q == 2 ? seed : seed - kP1;
    int i = 0;
    for (; i + 16 <= stripes; i += 16) {  // sixteen stripes' loads in flight before their rounds
      uint64_t d[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) d[u] = pair64(t + 8 * (i + u) + 2 * q);
#pragma unroll
      for (int u = 0; u < 16; ++u) v = xx_round(v, d[u]);
    }
    for (; i + 4 <= stripes; i += 4) {
      const uint64_t d0 = pair64(t + 8 * i + 2 * q), d1 = pair64(t + 8 * (i + 1) + 2 * q);
      const uint64_t d2 = pair64(t + 8 * (i + 2) + 2 * q), d3 = pair64(t + 8 * (i + 3) + 2 * q);
      v = xx_round(xx_round(xx_round(xx_round(v, d0), d1), d2), d3);
    }
    for (; i < stripes; ++i) v = xx_round(v, pair64(t + 8 * i + 2 * q));
    const uint64_t v1 = __shfl_sync(gmask, v, src0), v2 = __shfl_sync(gmask, v, src0 + 1);
    const uint64_t v3 = __shfl_sync(gmask, v, src0 + 2), v4 = __shfl_sync(gmask, v, src0 + 3);
    h = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
    h = (h ^ xx_round(0, v1)) * kP1 + kP4;
    h = (h ^ xx_round(0, v2)) * kP1 + kP4;
    h = (h ^ xx_round(0, v3)) * kP1 + kP4;
    h = (h ^ xx_round(0, v4)) * kP1 + kP4;
  } else {
    h = seed + kP5;
  }
  if (q != 0) return 0;
  h += (uint64_t)bytes;
  int i = 8 * stripes;
  for (; i + 2 <= n; i += 2) {
    h ^= xx_round(0, pair64(t + i));
    h = rotl(h, 27) * kP1 + kP4;
  }
  if (i < n) {  // one 4-byte word left (token lengths are whole words: no 1-byte tail)
    h ^= (uint64_t)(uint32_t)__ldg(t + i) * kP1;
    h = rotl(h, 23) * kP2 + kP3;
  }
  h ^= h >> 33;
  h *= kP2;
  h ^= h >> 29;
  h *= kP3;
  h ^= h >> 32;
  return h;
}

// Four lanes per chunk; blockIdx.y = stream, the x dimension walks its chunks.
__global__ void __launch_bounds__(256) cdc_fingerprint_kernel(const CdcArgs a) {
  const int s = blockIdx.y;
  const int64_t c = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2;
  const int q = threadIdx.x & 3, lane = threadIdx.x & 31;
  const uint32_t gmask = 0xfu << (lane & ~3);
  // the 4 lanes of a chunk agree on the test (same c), so the group shuffles stay within it
  if (a.chunk_hash == nullptr || c >= a.n_chunks[s]) return;
  const int64_t t = a.base[s] + c;
  const int32_t st = a.chunk_start[t], n = a.chunk_len[t];
  const uint64_t h = chunk_xxh64_x4(a.tokens + a.offsets[s] + st, n, a.seed, q, gmask, lane & ~3);
  if (q == 0) a.chunk_hash[t] = h;
}

}  // namespace

int cdc_segment_len() { return kSeg; }

cudaError_t launch_cdc(const CdcArgs& a, int64_t max_stream_len, int64_t slots, int64_t n_segs,
                       cudaStream_t stream) {
  if (a.S <= 0) return cudaSuccess;
  cdc_base_kernel<<<2, 1024, 0, stream>>>(a.offsets, a.S, a.min_len, a.base, a.seg_base);
  const int64_t steps = (max_stream_len + 127) / 128;
  const int64_t per_block = (int64_t)kHashWarps * kRunSteps;
  const int64_t gx = steps > 0 ? (steps + per_block - 1) / per_block : 0;
  if (gx > 0) {
    dim3 grid((unsigned)gx, (unsigned)a.S);
    cdc_hash_kernel<<<grid, 32 * kHashWarps, 0, stream>>>(a);
  }
  if (n_segs > 0) cdc_spec_kernel<<<(unsigned)((n_segs + 3) / 4), 128, 0, stream>>>(a, n_segs);
  cdc_fixup_kernel<<<(a.S + 3) / 4, 128, 0, stream>>>(a);
  if (a.chunk_hash != nullptr && slots > 0) {
    const int64_t per_stream = max_stream_len / a.min_len + 1;  // most slots one stream owns
    dim3 grid((unsigned)((4 * per_stream + 255) / 256), (unsigned)a.S);
    cdc_fingerprint_kernel<<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace irm
