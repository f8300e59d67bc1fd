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
// Passes (two kernels):
//   1. cdc_segment_kernel, W warps (2 or 4) per 4096-token segment of a stream: they hash
//      the segment and the max_len - 1 positions after it (a chunk starting in the segment
//      ends there at the latest) into a candidate bitmask in shared memory (the segment's own
//      words also go to global memory); one of them walks the chunks speculatively from the
//      segment start (one ballot per chunk: next_end), and all W fingerprint those chunks
//      while their tokens are hot.
//   2. cdc_resolve_kernel, one CTA per stream.  A walk entering a segment anywhere meets the
//      segment's speculative chain within a chunk or two, after which both agree; the segment
//      then exits where its speculative walk does.  So each warp takes one segment, enters it
//      at the previous segment's speculative exit, re-walks until it meets the speculative
//      chain, and counts (and records and fingerprints) its chunks; a prefix over the counts
//      places every segment's chunks (the recorded ones, then the speculative ones copied
//      with their fingerprints).  A segment whose re-walk does not meet its chain (possible only with
//      very long chunks) makes the rest of the stream follow the exact chain in order.
// Token ids outside the Gear table are read as G = 0 and recorded in the status word.
#include <cuda_runtime.h>
#include <climits>

#include "irm_common.cuh"
#include "irm_internal.h"

namespace irm {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kSegsPerCta = 2;        // segments per CTA of the segment pass
constexpr int kResWarps = 16;         // warps per CTA of the resolve pass (segments at a time)

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


// Stream offsets and per-stream bases: in the kernel parameters when the batch is small, else
// in the workspace.
struct StreamTab {
  const int64_t* offsets;
  const int64_t* base;      // first output slot of each stream
  const int64_t* seg_base;  // first segment of each stream
};
__device__ __forceinline__ StreamTab stream_tab(const CdcArgs& a) {
  return a.inline_streams ? StreamTab{a.ib.offsets, a.ib.base, a.ib.seg_base}
                          : StreamTab{a.offsets, a.base, a.seg_base};
}

// Pass 1: W warps per segment (two segments per CTA; each segment's warps sync on their own
// named barrier, never the whole block).
// Hashing: the window [p0, p_end) is cut into steps of 256 positions, lane l holding the 8
// consecutive positions 8l .. 8l+7 of a step.  With g0..g7 their Gear words, the lane's block
// contributes L = sum_e g_e 2^(7-e) to the hash at its last position (Horner), and a 3-step
// shuffle scan X_l = sum_{j <= l} L_j 2^(8 (l - j)) gives the hash there:
// h(8l+7) = h_prev 2^(8l+8) + X_l (terms shifted by 64 or more vanish).  The lane then steps
// h = 2 h + g through its own 8 positions from h(8l-1).  A warp's first step needs the hash
// at the position before it, h_prev = sum_{k<64} G[x_{q-1-k}] 2^k: lane l takes positions
// q-64+2l and q-63+2l and a butterfly sums the 32 shifted pairs.  Each step's tokens are
// loaded one step ahead (two 16-byte loads a lane when the stream is 16-byte aligned).  The
// W warps of a segment hash a W-th of its steps each; the first walks.  W = 4 when the batch
// has few segments for the GPU (more warps to hide the 64-bit arithmetic's latency), else 2.
static_assert(kSegsPerCta == 2, "seg_sync");
// Named barrier of a segment's warps (ids fixed at compile time, so that the kernel uses only
// the barriers it names).
template <int W>
__device__ __forceinline__ void seg_sync(int seg) {
  if (seg == 0) named_bar_sync(1, 32 * W); else named_bar_sync(2, 32 * W);
}
template <int W>
__global__ void __launch_bounds__(32 * W * kSegsPerCta) cdc_segment_kernel(const __grid_constant__ CdcArgs a) {
  constexpr int kSegWarpsPer = W;
  extern __shared__ uint32_t win_all[];  // per segment: candidate words of positions [p0, p_end)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pair = warp / kSegWarpsPer, half = warp % kSegWarpsPer;  // segment in the CTA, its warp
  const int64_t g = (int64_t)blockIdx.x * kSegsPerCta + pair;
  if (g >= a.n_segs) return;  // a segment's warps leave together
  const int win_words = (kSeg + a.max_len - 1 + 31) / 32;
  uint32_t* win = win_all + pair * win_words;
  const StreamTab st = stream_tab(a);
  int lo = 0, hi = a.S;  // the stream owning segment g: last s with seg_base[s] <= g
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (st.seg_base[mid] <= g) lo = mid; else hi = mid;
  }
  const int s = lo;
  const int64_t k = g - st.seg_base[s];
  const int64_t off = st.offsets[s], len = st.offsets[s + 1] - off;
  const int64_t p0 = k * kSeg;
  const int64_t seg_end = min(len, p0 + kSeg);                 // one past the segment
  const int64_t p_end = min(len, p0 + kSeg + a.max_len - 1);   // one past the last end reachable
  const int nwin = (int)((p_end - p0 + 31) / 32);
  const int seg_words = (int)((seg_end - p0 + 31) / 32);
  const int32_t* tok = a.tokens + off;
  uint32_t* gw = a.words + (off >> 5) + s;  // word base of the stream (see the header)
  const int64_t w0 = p0 >> 5;
  const uint64_t* gear = a.gear;
  const uint64_t gseed = a.gear_seed;
  const int vocab = a.vocab, bits = a.bits, mode = a.mode;
  // ---- candidate bitmask of the window (stream positions fit in 32 bits)
  {
    constexpr int kStep = 256;
    const int len32 = (int)len, p032 = (int)p0;
    const int nsteps_all = (int)((p_end - p0 + kStep - 1) / kStep);
    const int rbeg = half * nsteps_all / kSegWarpsPer, rend = (half + 1) * nsteps_all / kSegWarpsPer;
    const bool vec = (reinterpret_cast<uintptr_t>(tok) & 15u) == 0;
    int bad = 0;
    auto word = [&](int32_t x) -> uint64_t {
      if ((uint32_t)x >= (uint32_t)vocab) {
        bad = 1;
        return 0ull;
      }
      return gear != nullptr ? __ldg(gear + x) : splitmix_word(gseed, x);
    };
    auto load_step = [&](int rr, int32_t (&t8)[8]) {
      const int pb = p032 + kStep * rr + 8 * lane;
      if (vec && pb + 8 <= len32) {
        const int4 u = __ldg(reinterpret_cast<const int4*>(tok + pb));
        const int4 v = __ldg(reinterpret_cast<const int4*>(tok + pb + 4));
        t8[0] = u.x; t8[1] = u.y; t8[2] = u.z; t8[3] = u.w;
        t8[4] = v.x; t8[5] = v.y; t8[6] = v.z; t8[7] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) t8[e] = pb + e < len32 ? __ldg(tok + pb + e) : 0;
      }
    };
    uint64_t h_prev = 0;
    const int q = p032 + kStep * rbeg;  // the warp's first position
    if (rbeg < rend && q > 0) {
      const int pa = q - 64 + 2 * lane;
      const uint64_t ga = pa >= 0 ? word(__ldg(tok + pa)) : 0ull;
      const uint64_t gb = pa + 1 >= 0 ? word(__ldg(tok + pa + 1)) : 0ull;
      uint64_t t = ((ga << 1) + gb) << (62 - 2 * lane);  // positions q-1-(63-2l) and q-1-(62-2l)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) t += __shfl_xor_sync(kFull, t, o);
      h_prev = t;
    }
    int32_t cur[8];
    if (rbeg < rend) load_step(rbeg, cur);
    for (int r = rbeg; r < rend; ++r) {
      int32_t nxt[8];
      if (r + 1 < rend) load_step(r + 1, nxt);
      const int pb = p032 + kStep * r + 8 * lane;  // the lane's first position
      uint64_t gv[8];
      if (pb + 8 <= len32) {
#pragma unroll
        for (int e = 0; e < 8; ++e) gv[e] = word(cur[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gv[e] = pb + e < len32 ? word(cur[e]) : 0ull;
      }
      uint64_t xs = gv[0];
#pragma unroll
      for (int e = 1; e < 8; ++e) xs = (xs << 1) + gv[e];
#pragma unroll
      for (int d = 1; d < 8; d <<= 1) {  // shifts 8, 16, 32 (the shift-64 step vanishes)
        const uint64_t y = __shfl_up_sync(kFull, xs, d);
        if (lane >= d) xs += y << (8 * d);
      }
      const uint64_t h_last = (lane < 7 ? (h_prev << (8 * lane + 8)) : 0ull) + xs;
      uint64_t h = __shfl_up_sync(kFull, h_last, 1);  // hash at position 8l - 1
      if (lane == 0) h = h_prev;
      uint32_t byte = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        h = (h << 1) + gv[e];
        if (pb + e < len32 && cdc_candidate(h, bits, mode)) byte |= 1u << e;
      }
      // word j of the step collects the bytes of lanes 4j .. 4j+3
      uint32_t wv = byte << (8 * (lane & 3));
      wv |= __shfl_xor_sync(kFull, wv, 1);
      wv |= __shfl_xor_sync(kFull, wv, 2);
      if ((lane & 3) == 0) {
        const int w = 8 * r + (lane >> 2);
        if (w < nwin) win[w] = wv;
        if (w < seg_words) gw[w0 + w] = wv;  // the segment's own words, for the resolve pass
      }
      h_prev = __shfl_sync(kFull, h_last, 31);
#pragma unroll
      for (int e = 0; e < 8; ++e) cur[e] = nxt[e];
    }
    if (__any_sync(kFull, bad) && lane == 0) set_status(a.status, kDevErrBounds);
  }
  seg_sync<W>(pair);  // the segment's window is complete
  // ---- speculative walk from the segment start until a chunk ends at or past its end
  int32_t* ends = a.spec_ends + g * a.spec_cap;
  int* count_sh = reinterpret_cast<int*>(win_all + kSegsPerCta * win_words) + pair;
  if (half == 0) {
    const WordSrc words{gw, win, w0, nwin};
    int64_t t = p0;
    int c = 0;
    while (t < seg_end && c < a.spec_cap) {
      const int e = next_end(words, (int)len, (int)t, a.min_len, a.max_len, lane);
      if (lane == 0) ends[c] = e;
      ++c;
      t = (int64_t)e + 1;
    }
    if (lane == 0) {
      a.spec_count[g] = c;
      a.spec_exit[g] = (int32_t)t;
      *count_sh = c;
    }
  }
  seg_sync<W>(pair);  // the walk's ends are visible to the segment's warps
  const int c = *count_sh;
  // ---- fingerprints of the speculative chunks, four lanes per chunk
  if (a.chunk_hash != nullptr) {
    const int q = lane & 3;
    const uint32_t gmask = 0xfu << (lane & ~3);
    for (int i = (32 * half + lane) >> 2; i < c; i += 8 * kSegWarpsPer) {
      const int stt = i == 0 ? (int)p0 : ends[i - 1] + 1;
      const uint64_t h = chunk_xxh64_x4(tok + stt, ends[i] - stt + 1, a.seed, q, gmask, lane & ~3);
      if (q == 0) a.spec_hash[g * a.spec_cap + i] = h;
    }
  }
}

// Brings the 128-byte line holding p into the SM's L1 (no fault, no wait).
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }

// One segment of the chain, warp-collective: entering segment k of stream s at position t (the
// first chunk start at or after the segment start), re-walk until a chunk ends where a
// speculative one does, then take the rest of the speculative chunks.  Returns the chunks the
// segment contributes; *exit = the first chunk start after the segment; *met = the walk met
// the speculative chain (so that *exit is the speculative exit).  With `out` >= 0 the chunks
// are written from output slot `out` on (re-walked ones fingerprinted here).
struct SegCtx {
  const int32_t* tok;
  const uint32_t* gw;
  int64_t len, gb;
};
// The chunks a counting walk re-walked before it met the speculative chain (start, length,
// fingerprint), kept in shared memory so that placing them needs no second walk.
constexpr int kRec = 8;  // at most 8: the recorded chunks are fingerprinted by 4-lane groups of one warp
struct SegRec {
  int32_t start[kRec], len[kRec];
  uint64_t hash[kRec];
  int n;  // re-walked chunks recorded, -1 when there were more than kRec
  int p;  // the speculative chunk the walk met (-1: it started on the chain)
};
__device__ int walk_segment(const CdcArgs& a, const SegCtx& x, int64_t k, int64_t t, int64_t out, int lane,
                            int64_t* exit, bool* met_out, SegRec* rec = nullptr) {
  const int64_t seg_start = k * kSeg, seg_end = min(x.len, seg_start + kSeg);
  if (t >= seg_end) {  // a chunk longer than a segment covers this one
    *exit = t;
    *met_out = false;
    return 0;
  }
  const int64_t gseg = x.gb + k;
  const int32_t* ends = a.spec_ends + gseg * a.spec_cap;
  const int nspec = a.spec_count[gseg];
  const WordSrc words{x.gw, nullptr, 0, 0};
  int count = 0;
  int p = -1;  // last speculative chunk already covered by the re-walk
  bool met = t == seg_start;  // both walks start at the same place
  if (!met) {
    int sb = 0;  // the speculative ends, 32 at a time in registers (lane i: ends[sb + i])
    int32_t mine = lane < nspec ? ends[lane] : INT_MAX;
    while (t < seg_end) {
      const int e = next_end(words, (int)x.len, (int)t, a.min_len, a.max_len, lane);
      if (out >= 0) {
        if (lane == 0) {
          a.chunk_start[out + count] = (int32_t)t;
          a.chunk_len[out + count] = (int32_t)(e - t + 1);
        }
        if (a.chunk_hash != nullptr && lane < 4) {
          const uint64_t h = chunk_xxh64_x4(x.tok + t, (int)(e - t + 1), a.seed, lane, 0xfu, 0);
          if (lane == 0) a.chunk_hash[out + count] = h;
        }
      } else if (rec != nullptr && count < kRec && lane == 0) {
        rec->start[count] = (int32_t)t;  // fingerprinted after the walk, all at once
        rec->len[count] = (int32_t)(e - t + 1);
      }
      ++count;
      t = (int64_t)e + 1;
      bool found = false;
      for (;;) {  // first speculative end >= e
        const uint32_t ge = __ballot_sync(kFull, mine >= e);
        if (ge != 0u) {
          const int i = __ffs(ge) - 1;
          if (__shfl_sync(kFull, mine, i) == e) {
            met = true;
            p = sb + i;
          }
          found = true;
          break;
        }
        sb += 32;
        if (sb >= nspec) break;
        mine = sb + lane < nspec ? ends[sb + lane] : INT_MAX;
      }
      if (met || !found) break;
    }
  }
  if (rec != nullptr) {
    // fingerprints of the recorded chunks, four lanes per chunk (kRec <= 8), each chunk's
    // tokens asked for at once first (a chunk of max_len tokens is several batches of loads)
    __syncwarp();
    const int j = lane >> 2, q = lane & 3;
    if (j < min(count, kRec)) {
      uint64_t h = 0;
      if (a.chunk_hash != nullptr) {
        const int32_t* ct = x.tok + rec->start[j];
        const int n = rec->len[j];
        for (int i = 32 * q; i < n; i += 128) prefetch_l1(ct + i);
        h = chunk_xxh64_x4(ct, n, a.seed, q, 0xfu << (lane & ~3), lane & ~3);
      }
      if (q == 0) rec->hash[j] = h;
    }
    if (lane == 0) {
      rec->n = count <= kRec ? count : -1;
      rec->p = p;
    }
  }
  if (!met) {
    *exit = t;
    *met_out = false;
    return count;
  }
  // speculative chunks after index p are the true ones
  const int rest = nspec - (p + 1);
  if (out >= 0) {
    for (int i0 = p + 1; i0 < nspec; i0 += 32) {
      const int i = i0 + lane;
      if (i < nspec) {
        const int64_t stt = i == 0 ? seg_start : (int64_t)ends[i - 1] + 1;
        const int64_t o = out + count + (i - (p + 1));
        a.chunk_start[o] = (int32_t)stt;
        a.chunk_len[o] = (int32_t)(ends[i] - stt + 1);
        if (a.chunk_hash != nullptr) a.chunk_hash[o] = a.spec_hash[gseg * a.spec_cap + i];
      }
    }
  }
  *exit = a.spec_exit[gseg];
  *met_out = true;
  return count + rest;
}

// Places a segment that met its speculative chain from its counting walk's record: the
// re-walked chunks, then the speculative ones after the one the walk met.  Warp-collective.
__device__ void emit_recorded(const CdcArgs& a, const SegCtx& x, int64_t k, const SegRec& r, int64_t out,
                              int lane) {
  if (lane < r.n) {
    a.chunk_start[out + lane] = r.start[lane];
    a.chunk_len[out + lane] = r.len[lane];
    if (a.chunk_hash != nullptr) a.chunk_hash[out + lane] = r.hash[lane];
  }
  const int64_t seg_start = k * kSeg;
  const int64_t gseg = x.gb + k;
  const int32_t* ends = a.spec_ends + gseg * a.spec_cap;
  const int nspec = a.spec_count[gseg];
  for (int i0 = r.p + 1; i0 < nspec; i0 += 32) {
    const int i = i0 + lane;
    if (i < nspec) {
      const int64_t stt = i == 0 ? seg_start : (int64_t)ends[i - 1] + 1;
      const int64_t o = out + r.n + (i - (r.p + 1));
      a.chunk_start[o] = (int32_t)stt;
      a.chunk_len[o] = (int32_t)(ends[i] - stt + 1);
      if (a.chunk_hash != nullptr) a.chunk_hash[o] = a.spec_hash[gseg * a.spec_cap + i];
    }
  }
}

// Pass 2: one CTA per stream, kResWarps segments at a time (see the header).
__global__ void __launch_bounds__(kResWarps * 32, 2) cdc_resolve_kernel(const __grid_constant__ CdcArgs a) {
  __shared__ int cnt_sh[kResWarps];
  __shared__ int met_sh[kResWarps];
  __shared__ int64_t exit_sh[kResWarps];
  __shared__ int64_t pos_sh[kResWarps + 1];
  __shared__ int bad_sh;
  __shared__ SegRec rec_sh[kResWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const StreamTab st = stream_tab(a);
  const int s = blockIdx.x;
  const int64_t off = st.offsets[s], len = st.offsets[s + 1] - off;
  const int64_t cb = st.base[s];
  const SegCtx x{a.tokens + off, a.words + (off >> 5) + s, len, st.seg_base[s]};
  const int64_t nseg = (len + kSeg - 1) / kSeg;
  int64_t done = 0;  // chunks written so far
  for (int64_t g0 = 0; g0 < nseg; g0 += kResWarps) {
    const int64_t k = g0 + warp;
    if (k < nseg) {  // the segment's speculative chain and its fingerprints, asked for at once
      const int64_t gseg = x.gb + k, cap = a.spec_cap;
      if (32 * (int64_t)lane < cap) prefetch_l1(a.spec_ends + gseg * cap + 32 * (int64_t)lane);
      if (a.chunk_hash != nullptr && 16 * (int64_t)lane < cap)
        prefetch_l1(a.spec_hash + gseg * cap + 16 * (int64_t)lane);
      if (lane == 0) prefetch_l1(a.spec_count + gseg);
    }
    // the segment's entry, assuming the previous segment met its speculative chain
    const int64_t entry = k == 0 ? 0 : (k < nseg ? (int64_t)a.spec_exit[x.gb + k - 1] : 0);
    int64_t ex = 0;
    bool met = false;
    const int cnt = k < nseg ? walk_segment(a, x, k, entry, -1, lane, &ex, &met, &rec_sh[warp]) : 0;
    if (lane == 0) {
      cnt_sh[warp] = cnt;
      met_sh[warp] = (k < nseg - 1) ? (met ? 1 : 0) : 1;  // the last segment's exit matters to nobody
      exit_sh[warp] = ex;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      // the first segment whose exit is not its speculative one: its successors' assumed entries
      // are wrong, so the chain continues in order after it
      int bad = kResWarps;
      for (int w = 0; w < kResWarps && g0 + w < nseg; ++w)
        if (!met_sh[w]) {
          bad = w;
          break;
        }
      int64_t acc = done;
      for (int w = 0; w <= min(bad, kResWarps - 1); ++w) {
        pos_sh[w] = acc;
        acc += (g0 + w < nseg) ? cnt_sh[w] : 0;
      }
      pos_sh[kResWarps] = acc;
      bad_sh = bad;
    }
    __syncthreads();
    const int bad = bad_sh;
    if (k < nseg && warp <= bad) {
      if (met && rec_sh[warp].n >= 0) {
        emit_recorded(a, x, k, rec_sh[warp], cb + pos_sh[warp], lane);
      } else {
        int64_t ex2;
        bool met2;
        walk_segment(a, x, k, entry, cb + pos_sh[warp], lane, &ex2, &met2);
      }
    }
    done = pos_sh[kResWarps];
    if (bad < kResWarps) {
      // exact chain in order from the segment after `bad` (one warp)
      if (warp == 0) {
        int64_t t = exit_sh[bad];
        for (int64_t kk = g0 + bad + 1; kk < nseg && t < len; ++kk) {
          int64_t ex3;
          bool met3;
          done += walk_segment(a, x, kk, t, cb + done, lane, &ex3, &met3);
          t = ex3;
        }
        if (lane == 0) a.n_chunks[s] = (int32_t)done;
      }
      return;
    }
    __syncthreads();  // the shared arrays are reused by the next group
  }
  if (threadIdx.x == 0) a.n_chunks[s] = (int32_t)done;
}
}  // namespace

int cdc_segment_len() { return kSeg; }

cudaError_t launch_cdc(const CdcArgs& a, int64_t max_stream_len, int64_t slots, int64_t n_segs,
                       cudaStream_t stream) {
  (void)max_stream_len;
  (void)slots;
  if (a.S <= 0) return cudaSuccess;
  if (!a.inline_streams)
    cdc_base_kernel<<<2, 1024, 0, stream>>>(a.offsets, a.S, a.min_len, a.base, a.seg_base);
  if (n_segs > 0) {
    // each segment's window words (at most (4096 + 65535) / 32, 8.7 KB), then the walks' counts
    const size_t smem = (size_t)kSegsPerCta * ((kSeg + a.max_len - 1 + 31) / 32) * sizeof(uint32_t) +
                        kSegsPerCta * sizeof(int);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned grid = (unsigned)((n_segs + kSegsPerCta - 1) / kSegsPerCta);
    // four warps per segment while two would leave fewer than 16 warps per SM
    const bool wide = n_segs * 2 < (int64_t)16 * sms;
    auto kern = wide ? cdc_segment_kernel<4> : cdc_segment_kernel<2>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    kern<<<grid, 32 * (wide ? 4 : 2) * kSegsPerCta, smem, stream>>>(a);
  }
  cdc_resolve_kernel<<<(unsigned)a.S, kResWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irm
