// Split-KV decode for a few heads (one query token, H = 16 or 32 query rows), sm_103a.
//
// Computes, per request, O = softmax(scale * (q_lat . cKV + q_rope . R(delta) k_r)) . cKV for
// the single decode query ("Irminsul论文详解" §4; technical summary §2.2), with the k_r
// rotation applied to the staged tile in shared memory as in the fused tile kernel, but
// shaped for a handful of query rows:
//   - Operands are swapped so that KV rows, not heads, fill the tensor-core M dimension:
//     S^T = K Q^T (M = 64 KV rows, N = H, K = 576) and O^T += V^T P^T (M = 128 cKV columns
//     per block, N = H, K = 64 KV rows).  A softmax thread owns one KV row and all H heads,
//     so 64 threads share a tile's softmax instead of H.
//   - One CTA per (request, KV split) loads whole 576-column rows (no score exchange).  The
//     splits of a request form G thread-block clusters of C CTAs: after the pipeline every
//     CTA parks its unnormalised O^T and per-head (max, sum) in shared memory, and each
//     cluster merges its C splits through distributed shared memory, CTA r producing output
//     slice r (remote loads issued in batches of 8 splits, one round trip per batch).  With G = 1 that is the output; otherwise each cluster writes its slice as a
//     normalised partial, and the last cluster to finish a slice (a self-resetting counter
//     per request and slice) merges the G partials of that slice.
//   - Small UMMAs cost a fixed ~46 cycles each, so S^T is issued as few instructions as
//     possible: a stage stores the cKV slabs in pairs, interleaved by 8-row groups, so one
//     M = 128, N = 2H instruction covers two slabs (lanes of even groups hold the first
//     slab's rows against Q's first slab, odd groups the second slab's rows against Q's
//     second slab; the cross terms are never read).  The k_r slab stays a plain 64-row slab
//     (rotated in place) with its own M = 64 UMMA.  A row's two halves land 8 lanes apart in
//     one warp, so each pair of lanes shares a row and splits its heads.
//   - The running max of a head moves only when a tile exceeds it by more than 2^8 (P stays
//     <= 256; the final normalisation uses the same max, so the result is exact), so most
//     tiles need no cross-thread reduction: one barrier-OR tells whether any thread saw such
//     a score.
// KV tiles stream through two rings in shared memory instead of whole-tile stages: 16 KiB
// slab-pair units (as many as fit: 11 for H = 16) and three 8 KiB k_r slots.  Each unit has
// its own full/empty barriers, so the gather of later tiles runs ahead as soon as any unit
// frees, a k_r slot frees as soon as its tile's S^T is done, and S^T starts on the units of
// a tile as they land.
// Warp roles: 0-3 softmax, 4-11 loaders (cp.async row gather following the chunk table, and
// the k_r rotation: each loader warp rotates 8 rows of every landed k_r slot between its
// copies), 12 TMEM allocation and the S^T UMMAs, 13 the P.V UMMAs, 14 the row maps (built up to
// three tiles ahead, so the loaders never wait for one).  A single thread issues
// these small UMMAs no faster than one per ~40 cycles, so the two products get one issuing
// thread each (each thread commits and drains only its own UMMAs).  Bytes written by cp.async
// or by the rotation reach the tensor core through a proxy fence that the S^T issuer executes
// after acquiring the unit's or slot's barrier, so no loader thread fences (a loader's fence
// would also wait for its own copies in flight).  Every wait is
// bounded (2 s) and reports a timeout in the status word.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <mutex>

#include "irm_internal.h"
#include "irm_pipeline.cuh"

namespace irm {

// Timeline instrumentation, compiled only into the separately built timeline library
// (build.build(timeline=True) defines IRM_TIMELINE): the CTAs of request 0 stamp %globaltimer
// at the phases of a decode (kernel entry, set-up and its steps, each tile's scores and P.V
// issued, pipeline end, cluster merge, end) into a device array that irm_timeline_read()
// copies out.  The product library contains none of it.
#ifdef IRM_TIMELINE
constexpr int kTlCtas = 64, kTlTiles = 64;
enum : int { TL_ENTRY, TL_SETUP, TL_PIPE_END, TL_PARKED, TL_CLUSTER, TL_MERGED, TL_END,
              TL_SPLIT, TL_TMEM, TL_MAP, TL_ISSUED, TL_N };  // the last four: set-up steps
__device__ unsigned long long g_tl_cta[kTlCtas][TL_N];
__device__ unsigned long long g_tl_tile[kTlCtas][kTlTiles][3];  // data landed, S issued, P.V issued
#define IRM_TL(ev)                                                                        \
  do {                                                                                    \
    if (blockIdx.y == 0 && blockIdx.x < kTlCtas) g_tl_cta[blockIdx.x][(ev)] = globaltimer_ns(); \
  } while (0)
#define IRM_TL_TILE(j, k)                                                                           \
  do {                                                                                              \
    if (blockIdx.y == 0 && blockIdx.x < kTlCtas && (j) < kTlTiles) g_tl_tile[blockIdx.x][(j)][(k)] = globaltimer_ns(); \
  } while (0)
#else
#define IRM_TL(ev) \
  do {             \
  } while (0)
#define IRM_TL_TILE(j, k) \
  do {                    \
  } while (0)
#endif

namespace {

constexpr int kBN = 64;                         // KV rows per tile
constexpr uint32_t kSlab = kBN * 128;           // one 64-column slab of a tile
constexpr uint32_t kPairBytes = 2 * kSlab;      // ring unit: two interleaved cKV slabs
constexpr int kKrSlots = 3;                     // k_r ring (and row-map) slots
constexpr int kMaxUnits = 16;                   // slab-pair ring units at most
constexpr int kSoftmaxWarps = 4;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;

// Warp roles by head count: 8 loader warps for H = 16; 4 for H = 32, whose softmax needs the
// registers that a larger block would take away.
template <int H>
struct Roles {
  static constexpr int kLoaderWarps = H <= 16 ? 8 : 4;
  static constexpr int kMmaWarp = kSoftmaxWarps + kLoaderWarps;  // S^T issuer
  static constexpr int kPvWarp = kMmaWarp + 1;                    // P.V issuer
  static constexpr int kMapWarp = kPvWarp + 1;                    // row maps, ahead of the loaders
  static constexpr int kThreads = (kMapWarp + 1) * 32;
  static constexpr int kLoaderThreads = kLoaderWarps * 32;
  static constexpr int kRowsPerPass = kLoaderThreads / 8;  // rows one pass of the loaders covers
  static constexpr int kLoadPasses = kBN / kRowsPerPass;
  static constexpr int kRotRows = kBN / kLoaderWarps;      // k_r rows each loader warp rotates
};
constexpr uint32_t kSmemLimit = 232448;

// Fixed area at the start of shared memory.
constexpr uint32_t kOffBars = 0;                     // 64 mbarriers
constexpr uint32_t kOffMapSrc = 512;                 // int32 [kKrSlots][64]
constexpr uint32_t kOffMapDelta = kOffMapSrc + kKrSlots * kBN * 4;
constexpr uint32_t kOffPhase = kOffMapDelta + kKrSlots * kBN * 4;  // uint64 [32]
constexpr uint32_t kOffTmemPtr = kOffPhase + 32 * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kOffWmax = kOffAbort + 60;        // float [4 warps][32 heads]
constexpr uint32_t kOffWfail = kOffWmax + 512;       // int [4 warps]
constexpr uint32_t kOffLsum = kOffWfail + 64;        // float [4 warps][32 heads]
constexpr uint32_t kOffML = kOffLsum + 512;          // float m[32], l[32] of this split
constexpr uint32_t kFixedBytes = 4096;
static_assert(kOffML + 256 <= kFixedBytes, "fixed area overflow");

enum : int {
  BAR_PAIR_FULL = 0,                           // [unit] every loader thread's copies landed
  BAR_PAIR_EMPTY = BAR_PAIR_FULL + kMaxUnits,  // [unit] UMMA commit after the P.V reading it
  BAR_KR_LANDED = BAR_PAIR_EMPTY + kMaxUnits,  // [slot] every loader thread's k_r copies landed
  BAR_KR_FULL = BAR_KR_LANDED + kKrSlots,      // [slot] k_r rotated (count: loader warps)
  BAR_KR_EMPTY = BAR_KR_FULL + kKrSlots,       // [slot] UMMA commit after the tile's S^T
  BAR_MAP = BAR_KR_EMPTY + kKrSlots,           // [slot] row map of the tile published
  BAR_S_FULL = BAR_MAP + kKrSlots,             // [2] UMMA commit after S^T into score buffer
  BAR_S_EMPTY = BAR_S_FULL + 2,                // [2] softmax warps read the score buffer (count 4)
  BAR_P_FULL = BAR_S_EMPTY + 2,                // [2] softmax wrote P^T buffer (count 4)
  BAR_PV_DONE = BAR_P_FULL + 2,                // [2] UMMA commit after the P.V reading P^T buffer
  BAR_DRAIN = BAR_PV_DONE + 2,                 // [2] all UMMAs of the S^T / P.V issuer done
  NUM_BARS = BAR_DRAIN + 2,
};
static_assert(NUM_BARS <= 64, "barrier area");

constexpr uint32_t kTmemO = 0;     // O^T: 4 blocks of H columns (lane = cKV column in block)
constexpr uint32_t kTmemS = 128;   // 2 score buffers of 3H columns: paired S^T (2H), k_r part (H)
__host__ __device__ constexpr uint32_t tmem_cols(int H) { return kTmemS + 6u * (uint32_t)H <= 256u ? 256u : 512u; }

// Byte offset of 16-byte chunk c of row r of slab e (0 or 1) inside a slab pair: 8-row group
// g of slab e is the 1024-byte block 2g + e, 128-byte swizzled inside.
__host__ __device__ constexpr uint32_t pair_offset(uint32_t r, uint32_t e, uint32_t c) {
  return (2u * (r >> 3) + e) * 1024u + sw128_offset(r & 7u, c);
}
constexpr float kLn2 = 0.6931471805599453f;

struct DLayout {
  uint32_t q, p, kr, ring, total;
  int units;
};
__host__ __device__ constexpr uint32_t dl_kr(int H) {
  return (kFixedBytes + 11u * (uint32_t)H * 128u + 1023u) & ~1023u;
}
__host__ __device__ constexpr int dl_units(int H) {
  return (int)((kSmemLimit - 1024u - dl_kr(H) - kKrSlots * kSlab) / kPairBytes) > kMaxUnits
             ? kMaxUnits
             : (int)((kSmemLimit - 1024u - dl_kr(H) - kKrSlots * kSlab) / kPairBytes);
}
__host__ __device__ constexpr DLayout make_dlayout(int H) {
  // Q: 9 slabs of H rows x 128 B; P^T: 2 buffers of H rows x 128 B; the k_r ring; the unit ring
  return DLayout{kFixedBytes,
                 kFixedBytes + 9u * (uint32_t)H * 128u,
                 dl_kr(H),
                 dl_kr(H) + kKrSlots * kSlab,
                 dl_kr(H) + kKrSlots * kSlab + (uint32_t)dl_units(H) * kPairBytes + 1024u,
                 dl_units(H)};
}
static_assert(make_dlayout(32).units >= 8 && make_dlayout(16).units >= 8, "ring too small");
static_assert(make_dlayout(16).total <= kSmemLimit && make_dlayout(32).total <= kSmemLimit, "shared memory");

template <int H>
__device__ __forceinline__ void tmem_ld_h(uint32_t taddr, uint32_t (&r)[H]);
template <>
__device__ __forceinline__ void tmem_ld_h<16>(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16(taddr, r); }
template <>
__device__ __forceinline__ void tmem_ld_h<32>(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32(taddr, r); }
template <int H>
__device__ __forceinline__ void tmem_st_h(uint32_t taddr, const uint32_t (&r)[H]);
template <>
__device__ __forceinline__ void tmem_st_h<16>(uint32_t taddr, const uint32_t (&r)[16]) { tmem_st16(taddr, r); }
template <>
__device__ __forceinline__ void tmem_st_h<32>(uint32_t taddr, const uint32_t (&r)[32]) { tmem_st32(taddr, r); }

// Fold 8 partial results (log2 max or log2-sum-exp mq, sum lq, and 8 output columns va | vb)
// into a running (M, den, acc_a | acc_b): acc and den are kept relative to M, rescaled when M
// grows.
__device__ __forceinline__ void merge_batch2(const float (&mq)[8], const float (&lq)[8], const float4 (&va)[8],
                                             const float4 (&vb)[8], float& M, float& den, float4& acc_a,
                                             float4& acc_b) {
  float Mn = M;
#pragma unroll
  for (int k = 0; k < 8; ++k) Mn = fmaxf(Mn, mq[k]);
  if (Mn == -INFINITY) return;
  const float sc = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
  den *= sc;
  acc_a = make_float4(acc_a.x * sc, acc_a.y * sc, acc_a.z * sc, acc_a.w * sc);
  acc_b = make_float4(acc_b.x * sc, acc_b.y * sc, acc_b.z * sc, acc_b.w * sc);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float w = (mq[k] == -INFINITY) ? 0.f : fast_exp2(mq[k] - Mn);
    den += w * lq[k];
    acc_a.x += w * va[k].x;
    acc_a.y += w * va[k].y;
    acc_a.z += w * va[k].z;
    acc_a.w += w * va[k].w;
    acc_b.x += w * vb[k].x;
    acc_b.y += w * vb[k].y;
    acc_b.z += w * vb[k].z;
    acc_b.w += w * vb[k].w;
  }
  M = Mn;
}

// 4 fp32 values scaled by `inv`, rounded to bf16 (one 8-byte word).
__device__ __forceinline__ uint2 pack_bf16x4(float4 a, float inv) {
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x * inv, a.y * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(a.z * inv, a.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&h0);
  w.y = *reinterpret_cast<const uint32_t*>(&h1);
  return w;
}

template <int H>
__global__ void __launch_bounds__(Roles<H>::kThreads, 1) mla_decode_kernel(const __grid_constant__ DecodeArgs a) {
  using R = Roles<H>;
  if (threadIdx.x == 0) IRM_TL(TL_ENTRY);
  constexpr int kLoaderWarps = R::kLoaderWarps, kMmaWarp = R::kMmaWarp, kPvWarp = R::kPvWarp,
                kMapWarp = R::kMapWarp;
  constexpr int kThreads = R::kThreads, kLoaderThreads = R::kLoaderThreads;
  constexpr int kRowsPerPass = R::kRowsPerPass, kLoadPasses = R::kLoadPasses;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr DLayout L = make_dlayout(H);
  const int C = a.C, G = a.G;
  const int split = blockIdx.x;       // clusters are C consecutive CTAs along x
  const int crank = split % C, g = split / C;
  const int b = blockIdx.y;

  // the chunk table: in the parameter block (small tables) or in the workspace
  const irm_chunk* chunks = a.inline_table ? a.tab.chunks : a.chunks;
  const int32_t* indptr = a.inline_table ? a.tab.indptr : a.indptr;
  int c_begin, c_end, ctx = 0, c_first = -1;
  if (a.n_hints > 0) {
    const DecodeHint hint = a.hint[b * C * G + split];
    c_begin = hint.c_begin;
    c_end = hint.c_end;
    ctx = hint.ctx;
    c_first = hint.c_first;
  } else {
    c_begin = indptr[b];
    c_end = indptr[b + 1];
  }
  const bool table_ok = c_begin >= 0 && c_end > c_begin && c_end <= a.n_chunks &&
                        (c_first < 0 || (c_first >= c_begin && c_first < c_end));
  if (table_ok) {
    if (a.n_hints == 0) {
      const irm_chunk last = chunks[c_end - 1];
      ctx = last.p_tgt + last.len;
    }
  } else {
    c_begin = c_end = 0;
    c_first = -1;
  }
  const int kv_tiles = (table_ok && ctx > 0) ? (ctx + kBN - 1) / kBN : 0;
  const int kb = (int)((int64_t)split * kv_tiles / (C * G));
  const int ke = (int)((int64_t)(split + 1) * kv_tiles / (C * G));
  const int ntiles = ke - kb;
  if (threadIdx.x == 0) IRM_TL(TL_SPLIT);

  auto bar = [&](int i) -> uint32_t { return sb + kOffBars + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  int32_t* map_src = reinterpret_cast<int32_t*>(smem + kOffMapSrc);
  int32_t* map_delta = reinterpret_cast<int32_t*>(smem + kOffMapDelta);
  uint64_t* phaseF = reinterpret_cast<uint64_t*>(smem + kOffPhase);
  float* ml = reinterpret_cast<float*>(smem + kOffML);

  if (tid == 0) {
    if (!table_ok) set_status(a.status, kDevErrBounds);
    for (int u = 0; u < kMaxUnits; ++u) {
      mbar_init(bar(BAR_PAIR_FULL + u), kLoaderThreads);
      mbar_init(bar(BAR_PAIR_EMPTY + u), 1);
    }
    for (int k = 0; k < kKrSlots; ++k) {
      mbar_init(bar(BAR_KR_LANDED + k), kLoaderThreads);
      mbar_init(bar(BAR_KR_FULL + k), kLoaderWarps);
      mbar_init(bar(BAR_KR_EMPTY + k), 1);
      mbar_init(bar(BAR_MAP + k), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_S_FULL + s), 1);
      mbar_init(bar(BAR_S_EMPTY + s), kSoftmaxWarps);
      mbar_init(bar(BAR_P_FULL + s), kSoftmaxWarps);
      mbar_init(bar(BAR_PV_DONE + s), 1);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_DRAIN + 1), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (tid < 32) phaseF[tid] = a.phase.F[tid];
  if (warp == kMmaWarp) {
    tmem_alloc(sb + kOffTmemPtr, tmem_cols(H));
    tmem_relinquish();
    if (lane == 0) IRM_TL(TL_TMEM);
  }

  // ---- start-up work that needs no mbarrier: while the barriers and TMEM are being set up,
  //      the row-map warp builds tile 0's map and the loaders issue the copies of Q and of
  //      tile 0 (their landing is signalled after the block-wide barrier) ------------------
  const bool is_loader = warp >= kSoftmaxWarps && warp < kMmaWarp;
  const int tp = tid - kSoftmaxThreads;
  const int chk = tp & 7;    // loaders: 16-byte chunk of a 128-byte slab row
  const int rsub = tp >> 3;  // loaders: row within a pass
  const __nv_bfloat16* kvp = static_cast<const __nv_bfloat16*>(a.kv);
  ChunkWindow cw;
  cw.chunks = chunks;
  cw.c_end = c_end;
  cw.win = c_begin;
  if (warp == kMapWarp) {
    if (ntiles > 0) {
      if (c_first >= 0) {
        cw.win = c_first;  // the chunk holding the split's first row (launch hint)
        cw.load(lane);
      } else {
        cw.seek(c_begin, kb * kBN, lane);
      }
      cw.build_map(kb * kBN, ctx, a.n_rows, map_src, map_delta, a.status, lane);
    }
    __syncwarp();
    if (lane == 0) IRM_TL(TL_MAP);
    named_bar_arrive(2, kLoaderThreads + 32);  // tile 0's map is in slot 0
  } else if (is_loader) {
    named_bar_sync(2, kLoaderThreads + 32);
    if (ntiles > 0) {
      const __nv_bfloat16* ql = static_cast<const __nv_bfloat16*>(a.q_lat);
      const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(a.q_rope);
      // Q (H rows, all 576 columns, slab-major); it lands with tile 0 (same arrives)
      for (int h = rsub; h < H; h += kRowsPerPass) {
        const int64_t row = (int64_t)b * H + h;
        for (int slab = 0; slab < 9; ++slab) {
          const void* src = slab < 8 ? (const void*)(ql + row * kDLat + slab * 64 + chk * 8)
                                     : (const void*)(qr + row * kDRope + chk * 8);
          cp_async_16(sb + L.q + (uint32_t)slab * H * 128u + sw128_offset(h, chk), src, 16u);
        }
      }
      // tile 0 into k_r slot 0 and ring units 0-3 (all free at start)
      const __nv_bfloat16* rowp[kLoadPasses];
      uint32_t nb[kLoadPasses];
#pragma unroll
      for (int i = 0; i < kLoadPasses; ++i) {
        const int sr = map_src[kRowsPerPass * i + rsub];
        rowp[i] = kvp + (int64_t)(sr >= 0 ? sr : 0) * kDRow + chk * 8;
        nb[i] = sr >= 0 ? 16u : 0u;
      }
#pragma unroll
      for (int i = 0; i < kLoadPasses; ++i)
        cp_async_16(sb + L.kr + sw128_offset(kRowsPerPass * i + rsub, chk), rowp[i] + 8 * 64, nb[i]);
      for (int pr = 0; pr < 4; ++pr) {
        const uint32_t ub = sb + L.ring + (uint32_t)pr * kPairBytes;
#pragma unroll
        for (int i = 0; i < kLoadPasses; ++i) {
          const uint32_t r = (uint32_t)(kRowsPerPass * i + rsub);
          cp_async_16(ub + pair_offset(r, 0u, (uint32_t)chk), rowp[i] + (2 * pr) * 64, nb[i]);
          cp_async_16(ub + pair_offset(r, 1u, (uint32_t)chk), rowp[i] + (2 * pr + 1) * 64, nb[i]);
        }
      }
      if (tp == 0) IRM_TL(TL_ISSUED);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);
  if (threadIdx.x == 0) IRM_TL(TL_SETUP);

  if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
    // ======================= loaders: row gather with cp.async =========================
    const int pw = warp - kSoftmaxWarps;
    // tile 0 (and Q) went out before the block-wide barrier: signal its landing now (each
    // arrive fires once all of this thread's earlier copies have landed)
    if (ntiles > 0) {
      cp_async_arrive_noinc(bar(BAR_KR_LANDED + 0));
      for (int pr = 0; pr < 4; ++pr) cp_async_arrive_noinc(bar(BAR_PAIR_FULL + pr));
    }

    // k_r rotation, in tile order: this warp's 8 rows of every slot whose bytes have landed
    int rot = 0;
    int dprev = 0;
    float cs_c[8], cs_s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      cs_c[e] = 1.f;
      cs_s[e] = 0.f;
    }
    auto rotate_landed = [&](int upto) {
      while (rot < upto && __all_sync(kFullMask, mbar_test_wait(bar(BAR_KR_LANDED + rot % kKrSlots),
                                                                (uint32_t)(rot / kKrSlots) & 1u))) {
        const int rs = rot % kKrSlots;
#pragma unroll
        for (int r0 = 0; r0 < R::kRotRows; r0 += 8)
          rotate_krope_8rows(smem + L.kr + (uint32_t)rs * kSlab, map_delta + rs * kBN, phaseF, a.interleaved,
                             R::kRotRows * pw + r0,
                             lane, dprev, cs_c, cs_s);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_KR_FULL + rs));
        ++rot;
      }
    };
    // Wait for a ring barrier phase, rotating landed k_r slots meanwhile.
    auto wait_rotating = [&](uint32_t bb, uint32_t parity, int upto) -> bool {
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        rotate_landed(upto);
        if (__all_sync(kFullMask, mbar_test_wait(bb, parity))) break;
        __nanosleep(32);
        if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) return false;
      }
      return warp_wait(bb, parity, abort_flag);  // every lane acquires
    };

    bool ok = true;
    for (int j = 1; j < ntiles && ok; ++j) {
      const int ks = j % kKrSlots;
      const uint32_t kph = (uint32_t)(j / kKrSlots) & 1u;
      // k_r slot ks and its row map are free once the S^T of tile j - kKrSlots is done
      if (j >= kKrSlots && !(ok = wait_rotating(bar(BAR_KR_EMPTY + ks), kph ^ 1u, j))) break;
      if (!(ok = warp_wait(bar(BAR_MAP + ks), kph, abort_flag))) break;
      const __nv_bfloat16* rowp[kLoadPasses];
      uint32_t nb[kLoadPasses];
#pragma unroll
      for (int i = 0; i < kLoadPasses; ++i) {
        const int sr = map_src[ks * kBN + kRowsPerPass * i + rsub];
        rowp[i] = kvp + (int64_t)(sr >= 0 ? sr : 0) * kDRow + chk * 8;
        nb[i] = sr >= 0 ? 16u : 0u;
      }
      // k_r first: its rotation then overlaps the cKV copies
      const uint32_t kr = sb + L.kr + (uint32_t)ks * kSlab;
#pragma unroll
      for (int i = 0; i < kLoadPasses; ++i)
        cp_async_16(kr + sw128_offset(kRowsPerPass * i + rsub, chk), rowp[i] + 8 * 64, nb[i]);
      cp_async_arrive_noinc(bar(BAR_KR_LANDED + ks));
      for (int pr = 0; pr < 4; ++pr) {
        const int gu = 4 * j + pr;  // global unit sequence number
        const int u = gu % L.units, use = gu / L.units;
        if (use >= 1 && !(ok = wait_rotating(bar(BAR_PAIR_EMPTY + u), (uint32_t)(use - 1) & 1u, j))) break;
        const uint32_t ub = sb + L.ring + (uint32_t)u * kPairBytes;
#pragma unroll
        for (int i = 0; i < kLoadPasses; ++i) {
          const uint32_t r = (uint32_t)(kRowsPerPass * i + rsub);
          cp_async_16(ub + pair_offset(r, 0u, (uint32_t)chk), rowp[i] + (2 * pr) * 64, nb[i]);
          cp_async_16(ub + pair_offset(r, 1u, (uint32_t)chk), rowp[i] + (2 * pr + 1) * 64, nb[i]);
        }
        cp_async_arrive_noinc(bar(BAR_PAIR_FULL + u));
      }
      if (ok) rotate_landed(j + 1);
    }
    // rotate what is left (bounded waits for the last slots to land)
    while (ok && rot < ntiles) {
      if (!(ok = warp_wait(bar(BAR_KR_LANDED + rot % kKrSlots), (uint32_t)(rot / kKrSlots) & 1u, abort_flag))) break;
      rotate_landed(rot + 1);
    }
    cp_async_wait_all();
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
  } else if (warp == kMapWarp) {
    // ======================= row maps: tile t into slot t % 3 once tile t-3's S^T is done ======
    // (tile 0's map was built before the block-wide barrier; its arrive keeps the phases)
    bool ok = true;
    if (ntiles > 0 && lane == 0) mbar_arrive(bar(BAR_MAP + 0));
    for (int t = 1; t < ntiles && ok; ++t) {
      const int ks = t % kKrSlots;
      if (t >= kKrSlots &&
          !(ok = warp_wait(bar(BAR_KR_EMPTY + ks), ((uint32_t)(t / kKrSlots) & 1u) ^ 1u, abort_flag)))
        break;
      cw.build_map((kb + t) * kBN, ctx, a.n_rows, map_src + ks * kBN, map_delta + ks * kBN, a.status, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_MAP + ks));
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ======================= S^T issuer (one thread) =====================================
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdescS2 = idesc_bf16_f32(128, 2 * H, 0, 0);  // A = slab pair, B = Q slab pair
      constexpr uint32_t kIdescS1 = idesc_bf16_f32(64, H, 0, 0);       // A = k_r slab, B = Q k_r slab
      bool ok = true;
      for (int ns = 0; ns < ntiles && ok; ++ns) {
        const uint32_t tS = tmem + kTmemS + (uint32_t)((ns & 1) * 3 * H);
        // score buffer ns&1 is free once the softmax read tile ns-2's scores
        if (ns >= 2 && !(ok = mbar_wait(bar(BAR_S_EMPTY + (ns & 1)), ((ns >> 1) - 1) & 1, abort_flag))) break;
        for (int sq = 0; sq < 4; ++sq) {
          const int gu = 4 * ns + sq;
          const int u = gu % L.units, use = gu / L.units;
          if (!(ok = mbar_wait(bar(BAR_PAIR_FULL + u), (uint32_t)use & 1u, abort_flag))) break;
          // cp.async bytes observed through the barrier -> async proxy before the UMMA reads
          tc_fence_after();
          fence_proxy_async_smem();
          const uint32_t ub = sb + L.ring + (uint32_t)u * kPairBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(ub + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sb + L.q + (uint32_t)(2 * sq) * H * 128u + kk * 32, 16, 1024);
            umma_bf16(tS, ad, bd, kIdescS2, (sq | kk) ? 1u : 0u);
          }
        }
        if (!ok) break;
        const int ks = ns % kKrSlots;
        IRM_TL_TILE(ns, 0);
        if (!(ok = mbar_wait(bar(BAR_KR_FULL + ks), (uint32_t)(ns / kKrSlots) & 1u, abort_flag))) break;
        // rotated rows (generic-proxy writes of the loaders) -> async proxy
        tc_fence_after();
        fence_proxy_async_smem();
        const uint32_t kr = sb + L.kr + (uint32_t)ks * kSlab;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(kr + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + L.q + 8u * H * 128u + kk * 32, 16, 1024);
          umma_bf16(tS + 2u * H, ad, bd, kIdescS1, kk ? 1u : 0u);
        }
        umma_commit(bar(BAR_KR_EMPTY + ks));
        umma_commit(bar(BAR_S_FULL + (ns & 1)));
        IRM_TL_TILE(ns, 1);
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, kDevErrTimeout);
      }
      umma_commit(bar(BAR_DRAIN));
      if (!mbar_wait(bar(BAR_DRAIN), 0, nullptr)) set_status(a.status, kDevErrTimeout);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ======================= P.V issuer (one thread) =====================================
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, H, 1, 0);  // A = V^T (MN-major), B = P^T
      bool ok = true;
      for (int np = 0; np < ntiles && ok; ++np) {
        if (!(ok = mbar_wait(bar(BAR_P_FULL + (np & 1)), (np >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t pb = sb + L.p + (uint32_t)(np & 1) * H * 128u;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          // V^T block = slab pair blk: M atoms (64 columns) 1024 B apart, 8-row K groups
          // 2048 B apart, 16 KV rows per K-step; the unit is released as soon as its own
          // four UMMAs complete
          const uint32_t ub = sb + L.ring + (uint32_t)((4 * np + blk) % L.units) * kPairBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_sw128(pb + kk * 32, 16, 1024);
            const uint64_t ad = sdesc_sw128(ub + kk * 4096, 1024, 2048);
            umma_bf16(tmem + kTmemO + (uint32_t)(blk * H), ad, bd, kIdescPV, (np > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar(BAR_PAIR_EMPTY + (4 * np + blk) % L.units));
        }
        umma_commit(bar(BAR_PV_DONE + (np & 1)));
        IRM_TL_TILE(np, 2);
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, kDevErrTimeout);
      }
      umma_commit(bar(BAR_DRAIN + 1));
      if (!mbar_wait(bar(BAR_DRAIN + 1), 0, nullptr)) set_status(a.status, kDevErrTimeout);
    }
    __syncwarp();
  } else {
    // ======================= softmax: two lanes per KV row, each with half of the heads ====
    // Paired S^T: lane L of warp w holds, for local row rho = 8 (L / 16) + L % 8, the partial
    // over the even cKV slabs (L % 16 < 8, columns [0, H)) or over the odd ones (columns
    // [H, 2H)); the k_r part of local row rho sits in lane rho (M = 64 layout).
    constexpr int Hh = H / 2;
    const bool odd = (lane & 8) != 0;               // this lane takes heads [Hh, H)
    const int rho = ((lane >> 4) << 3) | (lane & 7);
    const int krow = 16 * warp + rho;               // KV row of the tile
    const int hbase = odd ? Hh : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c = a.scale_log2;
    float* wmax = reinterpret_cast<float*>(smem + kOffWmax);
    int* wfail = reinterpret_cast<int*>(smem + kOffWfail);
    float m_run[H], l_own[Hh];
#pragma unroll
    for (int h = 0; h < H; ++h) m_run[h] = -INFINITY;
#pragma unroll
    for (int k = 0; k < Hh; ++k) l_own[k] = 0.f;
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      const int T = (kb + j) * kBN;
      float x[Hh];
      if (warp_wait(bar(BAR_S_FULL + s), (j >> 1) & 1, abort_flag)) {
        tc_fence_after();
        const uint32_t tS = tmem + kTmemS + (uint32_t)(s * 3 * H) + lane_base;
        uint32_t r2[2 * H], u[H];
        if constexpr (H == 16) {
          tmem_ld32(tS, r2);
        } else {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r2[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r2[32]);
          tmem_ld32(tS, lo);
          tmem_ld32(tS + 32u, hi);
        }
        tmem_ld_h<H>(tS + 2u * H, u);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_S_EMPTY + s));
        // own heads: own half-sum + the partner lane's (8 lanes away) + the k_r part of the row
        const bool valid = T + krow < ctx;
#pragma unroll
        for (int k = 0; k < Hh; ++k) {
          const float own = __uint_as_float(odd ? r2[H + Hh + k] : r2[k]);
          const float give = __uint_as_float(odd ? r2[H + k] : r2[Hh + k]);
          const float ua = __shfl_sync(kFullMask, __uint_as_float(u[k]), rho);
          const float ub = __shfl_sync(kFullMask, __uint_as_float(u[Hh + k]), rho);
          const float v = own + __shfl_xor_sync(kFullMask, give, 8) + (odd ? ub : ua);
          x[k] = valid ? v * c : -INFINITY;
        }
      } else {
#pragma unroll
        for (int k = 0; k < Hh; ++k) x[k] = -INFINITY;
        bad = true;
      }
      bool exceed = false;
#pragma unroll
      for (int k = 0; k < Hh; ++k) exceed |= x[k] > (odd ? m_run[Hh + k] : m_run[k]) + 8.f;
      if (named_bar_red_or(1, kSoftmaxThreads, exceed || bad)) {
        // some score passed its head's running max by 2^8 (or a wait failed): tile max per
        // head over the 64 rows (the 16 lanes of a warp holding a head, then the 4 warps)
#pragma unroll
        for (int k = 0; k < Hh; ++k) {
          float v = x[k];
          v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 16));
          v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 4));
          v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 2));
          v = fmaxf(v, __shfl_xor_sync(kFullMask, v, 1));
          if ((lane & 23) == 0) wmax[warp * 32 + hbase + k] = v;  // lanes 0 and 8
        }
        if (lane == 0) wfail[warp] = bad ? 1 : 0;
        named_bar_sync(1, kSoftmaxThreads);
        if (wfail[0] | wfail[1] | wfail[2] | wfail[3]) break;  // every warp leaves here
        float corr[H];
        bool changed = false;
#pragma unroll
        for (int h = 0; h < H; ++h) {
          const float tm = fmaxf(fmaxf(wmax[h], wmax[32 + h]), fmaxf(wmax[64 + h], wmax[96 + h]));
          const bool want = tm > m_run[h] + 8.f;
          corr[h] = want ? fast_exp2(m_run[h] - tm) : 1.f;
          if (want) {
            changed |= m_run[h] != -INFINITY;
            m_run[h] = tm;
          }
        }
#pragma unroll
        for (int k = 0; k < Hh; ++k) l_own[k] *= odd ? corr[Hh + k] : corr[k];
        if (changed && j > 0) {
          // rescale O^T (every lane holds one cKV column of each block) once the previous
          // tile's P.V has landed
          if (!warp_wait(bar(BAR_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag)) {
            bad = true;
          } else {
            tc_fence_after();
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t r[H];
              tmem_ld_h<H>(tmem + kTmemO + (uint32_t)(blk * H) + lane_base, r);
              tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < H; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * corr[h]);
              tmem_st_h<H>(tmem + kTmemO + (uint32_t)(blk * H) + lane_base, r);
            }
            tmem_st_wait();
          }
        }
      }
      // P^T buffer s is free once the P.V of tile j-2 completed
      if (j >= 2 && !warp_wait(bar(BAR_PV_DONE + s), ((j - 2) >> 1) & 1, abort_flag)) bad = true;
      {
        // P^T row h (K-major, 64 KV rows = 128 bytes, 128-byte swizzle), element krow
        uint8_t* pbuf = smem + L.p + (uint32_t)s * H * 128u;
        const uint32_t ck = (uint32_t)krow >> 3, wo = ((uint32_t)krow & 7u) * 2u;
#pragma unroll
        for (int k = 0; k < Hh; ++k) {
          const int h = hbase + k;
          const float p = fast_exp2(x[k] - (odd ? m_run[Hh + k] : m_run[k]));
          l_own[k] += p;
          *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + ((ck ^ (uint32_t)(h & 7)) << 4) + wo) =
              __float2bfloat16_rn(p);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + s));
    }
    bool ok = !bad;
    if (ntiles > 0 && ok)
      ok = warp_wait(bar(BAR_PV_DONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, abort_flag);
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
    // per-head sums over the 64 rows (the 16 lanes holding a head, then the 4 warps)
    float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
#pragma unroll
    for (int k = 0; k < Hh; ++k) {
      float v = l_own[k];
      v += __shfl_xor_sync(kFullMask, v, 16);
      v += __shfl_xor_sync(kFullMask, v, 4);
      v += __shfl_xor_sync(kFullMask, v, 2);
      v += __shfl_xor_sync(kFullMask, v, 1);
      if ((lane & 23) == 0) lsum[warp * 32 + hbase + k] = v;
    }
    named_bar_sync(1, kSoftmaxThreads);
    if (tid < H) {
      float mv = -INFINITY;
#pragma unroll
      for (int h = 0; h < H; ++h)
        if (h == tid) mv = m_run[h];
      ml[tid] = mv;
      ml[32 + tid] = (lsum[tid] + lsum[32 + tid]) + (lsum[64 + tid] + lsum[96 + tid]);
    }
  }

  // ---- park this split's unnormalised O^T [H][512] (fp32) in the drained KV stages ------
  __syncthreads();
  if (threadIdx.x == 0) IRM_TL(TL_PIPE_END);
  const bool cta_ok = *abort_flag == 0 && ntiles > 0;
  float* opart = reinterpret_cast<float*>(smem + L.ring);
  if (warp < kSoftmaxWarps) {
    tc_fence_after();
    if (!cta_ok && tid < H) {
      ml[tid] = -INFINITY;
      ml[32 + tid] = 0.f;
    }
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t r[H];
      if (cta_ok) {
        tmem_ld_h<H>(tmem + kTmemO + (uint32_t)(blk * H) + ((uint32_t)(warp * 32) << 16), r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int h = 0; h < H; ++h) r[h] = 0u;
      }
      const int col = blk * 128 + warp * 32 + lane;
#pragma unroll
      for (int h = 0; h < H; ++h) opart[h * kDLat + col] = __uint_as_float(r[h]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) IRM_TL(TL_PARKED);
  cluster_arrive();  // every split of the request has parked its partial
  cluster_wait();
  if (threadIdx.x == 0) IRM_TL(TL_CLUSTER);

  // ---- merge the C splits of this cluster through distributed shared memory: CTA crank
  //      takes items [crank * per, (crank + 1) * per) of the H x 64 items (at most one per
  //      thread for 16 heads and C >= 4).  Item (h, q) is 8 columns of head h in two groups of
  //      4, columns c0 = 256 (q / 32) + 4 (q % 32) and c0 + 128: a warp's 16-byte loads of one
  //      group are contiguous (512 B), which the cluster's shared-memory network serves about
  //      twice as fast as 16-byte pieces 32 B apart ------------------------------------------
  const int per = H * 64 / C;
  float4* gpart = reinterpret_cast<float4*>(a.gpart);
  for (int it = tid; it < per; it += kThreads) {
    const int item = crank * per + it;
    const int h = item >> 6, q = item & 63;
    const int c0 = 256 * (q >> 5) + 4 * (q & 31);
    // online merge over the splits, 8 at a time: every remote load of a batch is issued before
    // any is used, so a batch costs one round trip through the cluster
    float M = -INFINITY, den = 0.f;
    float4 acc_a = make_float4(0.f, 0.f, 0.f, 0.f), acc_b = acc_a;
    for (int q0 = 0; q0 < C; q0 += 8) {
      float mq[8], lq[8];
      float4 va[8], vb[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (q0 + k < C) {
          const uint32_t base = mapa_shared(sb, (uint32_t)(q0 + k));
          const uint32_t vaddr = base + L.ring + (uint32_t)(h * kDLat + c0) * 4u;
          mq[k] = ld_cluster_f32(base + kOffML + 4u * h);
          lq[k] = ld_cluster_f32(base + kOffML + 128u + 4u * h);
          va[k] = ld_cluster_v4(vaddr);
          vb[k] = ld_cluster_v4(vaddr + 512u);
        } else {
          mq[k] = -INFINITY;
          lq[k] = 0.f;
          va[k] = vb[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      merge_batch2(mq, lq, va, vb, M, den, acc_a, acc_b);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const float lse2 = den > 0.f ? M + __log2f(den) : -INFINITY;  // log2 units
    const int64_t orow = (int64_t)b * H + h;
    if (G == 1) {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + orow * kDLat + c0;
      *reinterpret_cast<uint2*>(o) = pack_bf16x4(acc_a, inv);
      *reinterpret_cast<uint2*>(o + 128) = pack_bf16x4(acc_b, inv);
      if (q == 0 && a.lse != nullptr) a.lse[orow] = lse2 * kLn2;
    } else {
      float4* dst = gpart + ((int64_t)b * G + g) * (H * 128) + h * 128 + (c0 >> 2);
      dst[0] = make_float4(acc_a.x * inv, acc_a.y * inv, acc_a.z * inv, acc_a.w * inv);
      dst[32] = make_float4(acc_b.x * inv, acc_b.y * inv, acc_b.z * inv, acc_b.w * inv);
      if (q == 0) a.glse[((int64_t)b * G + g) * H + h] = lse2;
    }
  }
  cluster_arrive();  // this CTA has finished reading its peers' shared memory (waited for at exit)
  if (threadIdx.x == 0) IRM_TL(TL_MERGED);
  if (G > 1) {
    // the last of the G clusters to finish slice crank merges it (threadfence reduction; the
    // counter resets itself so the workspace stays reusable)
    int* last_sh = reinterpret_cast<int*>(smem + kOffWfail);
    __syncthreads();
    if (tid == 0) {
      __threadfence();  // cumulative: the CTA's partial stores, ordered before it by the barrier
      int* cnt = a.counters + (int64_t)b * C + crank;
      const int done = atomicAdd(cnt, 1);
      *last_sh = done == G - 1;
      if (done == G - 1) *cnt = 0;
    }
    __syncthreads();
    if (*last_sh) {
      __threadfence();
      for (int it = tid; it < per; it += kThreads) {
        const int item = crank * per + it;
        const int h = item >> 6, q = item & 63;
        const int c0 = 256 * (q >> 5) + 4 * (q & 31);
        const float* gl = a.glse + (int64_t)b * G * H + h;
        float M = -INFINITY, den = 0.f;
        float4 acc_a = make_float4(0.f, 0.f, 0.f, 0.f), acc_b = acc_a;
        for (int q0 = 0; q0 < G; q0 += 8) {
          float mq[8], lq[8];
          float4 va[8], vb[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (q0 + k < G) {
              const float4* src = gpart + ((int64_t)b * G + q0 + k) * (H * 128) + h * 128 + (c0 >> 2);
              mq[k] = __ldcg(gl + (int64_t)(q0 + k) * H);  // log2-sum-exp of a normalised partial
              lq[k] = 1.f;
              va[k] = __ldcg(src);
              vb[k] = __ldcg(src + 32);
            } else {
              mq[k] = -INFINITY;
              lq[k] = 0.f;
              va[k] = vb[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          merge_batch2(mq, lq, va, vb, M, den, acc_a, acc_b);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        const int64_t orow = (int64_t)b * H + h;
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + orow * kDLat + c0;
        *reinterpret_cast<uint2*>(o) = pack_bf16x4(acc_a, inv);
        *reinterpret_cast<uint2*>(o + 128) = pack_bf16x4(acc_b, inv);
        if (q == 0 && a.lse != nullptr) a.lse[orow] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
      }
    }
  }
  if (threadIdx.x == 0) IRM_TL(TL_END);
  cluster_wait();  // peers are done reading this CTA's shared memory
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols(H));
  }
}

template <int H>
cudaLaunchConfig_t decode_config(const DecodeArgs& a, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(a.C * a.G), (unsigned)a.B, 1);
  cfg.blockDim = dim3(Roles<H>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = make_dlayout(H).total;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Kernel attributes belong to the device: they are set once per device (not per launch).
template <int H>
cudaError_t prepare_decode() {
  static std::mutex mu;
  static bool done[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 128;
  std::lock_guard<std::mutex> lk(mu);
  if (cached && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(mla_decode_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)make_dlayout(H).total);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mla_decode_kernel<H>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess && cached) done[dev] = true;
  return e;
}

template <int H>
cudaError_t launch_decode_h(const DecodeArgs& a, cudaStream_t stream) {
  cudaError_t e = prepare_decode<H>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = decode_config<H>(a, stream, attr);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<H>, a);
}

template <int H>
int max_clusters_h(int C) {
  if (prepare_decode<H>() != cudaSuccess) return 0;
  DecodeArgs a{};
  a.C = C;
  a.G = 1;
  a.B = 1;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = decode_config<H>(a, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<H>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

bool decode_supported(int H) { return H == 16 || H == 32; }

int decode_max_active_clusters(int H, int C) {
  if (C < 1 || C > kMaxDecodeCluster) return 0;
  return H == 16 ? max_clusters_h<16>(C) : H == 32 ? max_clusters_h<32>(C) : 0;
}

#ifdef IRM_TIMELINE
// Timeline build only: copies out (and clears) the stamps of the last decode.
extern "C" int irm_timeline_read(unsigned long long* cta, unsigned long long* tile) {
  cudaError_t e = cudaMemcpyFromSymbol(cta, g_tl_cta, sizeof(g_tl_cta));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(tile, g_tl_tile, sizeof(g_tl_tile));
  static unsigned long long zero[kTlCtas * kTlTiles * 3];
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tl_cta, zero, sizeof(g_tl_cta));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_tl_tile, zero, sizeof(g_tl_tile));
  return (int)e;
}
#endif

cudaError_t launch_mla_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.C < 1 || a.C > kMaxDecodeCluster || (a.C & (a.C - 1)) != 0 || a.G < 1 ||
      (a.G > 1 && (a.gpart == nullptr || a.glse == nullptr || a.counters == nullptr)))
    return cudaErrorInvalidConfiguration;
  if (a.H == 16) return launch_decode_h<16>(a, stream);
  if (a.H == 32) return launch_decode_h<32>(a, stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace irm
