// Fused delta-rotate + absorbed MLA attention (decode and causal prefill), sm_103a.
//
// What is computed ("Irminsul论文详解" §4; technical summary §2.2): for every query row
// (query token, head) of a request whose KV is rebuilt from a chunk pool,
//   s_t = scale * (q_lat . cKV_t + q_rope . R(delta_t) k_r,t),  O = softmax(s) . cKV,
// where cKV_t and k_r,t come from the row store at the chunk table's source row, and the
// rotation R(delta_t) is applied while the tile sits in shared memory, between the HBM
// load and the tensor-core read, so rotated keys are never written back to HBM.
//
// Structure (one 2-CTA cluster per 128-row query tile and KV split):
//   - The [cKV | k_r] contraction of Q K^T is split by columns: CTA r owns cKV[256r, 256r+256)
//     and the NeoX pairs j = 16r .. 16r+15 of k_r (columns j and 32 + j), and rotates them.
//     The two CTAs thus load, rotate and multiply equal shares, and each loads only its own
//     columns of every KV row, so each row is read from memory exactly once.
//   - Each CTA computes its partial scores S_r = Q_r K_r^T (tcgen05, M=128, N=64) into
//     TMEM and ships them to the peer with st.async, as fp16 (half the bytes and stores of
//     the exchange; the rounding, ~5e-4 of a partial, is well below P's own bf16 rounding).
//     Both form round_f32(fp16 own + fp16 peer) and run the identical online softmax, so P
//     is bit-identical in both CTAs.
//   - The output is split the same way: CTA r accumulates O[:, 256r:256r+256) += P V_r
//     (tcgen05, M=128, N=256) in TMEM, with V_r = the cKV columns it already holds.
//   - TMEM holds O (256 columns), one score buffer (64 columns), a double buffer for P
//     (2 x 32 columns of bf16 pairs) and the CTA's four cKV slabs of Q as bf16 pairs (128
//     columns); both Q.K^T and P.V take their A operand from TMEM.  The softmax warps load
//     a tile's scores into registers and release the score buffer at once, so the next
//     Q.K^T never waits for a P.V.  Both issuers build their operand descriptors once per
//     tile and step them by constants (a thread issues one UMMA per ~50 cycles at best, so
//     small UMMAs are issue-bound).  Only the CTA's half of q_rope sits in shared memory,
//     so nearly all of shared memory is KV pipeline stages.
//   - The softmax is software-pipelined: iteration j combines tile j's own and peer
//     partials, loads tile j+1's scores, ships them to the peer once the peer has read tile
//     j's, and then runs tile j's exponentials, so the exchange of one tile overlaps the
//     softmax of the previous one.
//   - Warp roles: 0-7 softmax, two warps per TMEM lane quadrant (thread = TMEM lane = query
//     row; warps 0-3 take keys 0-31 of every tile, warps 4-7 keys 32-63, and the two warps
//     of a quadrant agree on their rows' running max through one 64-thread barrier
//     reduction per tile); 8-9 gather KV
//     rows with cp.async (completion tracked by an mbarrier, so they run ahead across
//     stages); 10-11 rotate each landed tile's k_r by R(delta) and publish it; 12 allocates
//     TMEM; 13 issues P.V and 15 Q.K^T (one issuing thread per product); 14 turns the chunk
//     table into per-tile row maps, up to the stage count ahead of the copies.
//   - Only the first Mv rows (valid query rows rounded up to 8) of the q_rope slab and the
//     score exchange are stored: the UMMA still reads 128 rows, and the rows past Mv read
//     whatever follows in shared memory (or TMEM lanes nobody wrote).  Those rows only
//     ever produce rows of S / O that are never read.
// Every pipeline wait is bounded (2 s) and reports a timeout in the status word.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>
#include <mutex>

#include "irm_internal.h"
#include "irm_pipeline.cuh"

namespace irm {
namespace {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 64;   // KV rows per tile
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quadrant: keys 0-31 / 32-63 of a tile
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kLoaderWarps = 4;   // 2 copy warps + 2 publishers
constexpr int kCopyWarps = 2;
constexpr int kCopyThreads = kCopyWarps * 32;
constexpr int kPubWarps = kLoaderWarps - kCopyWarps;
constexpr int kMmaWarp = kSoftmaxWarps + kLoaderWarps;  // 12: TMEM allocation
constexpr int kPvWarp = kMmaWarp + 1;                    // 13: P.V issue
constexpr int kMapWarp = kPvWarp + 1;                    // 14: row maps, ahead of the copies
constexpr int kSWarp = kMapWarp + 1;                     // 15: Q.K^T issue
constexpr int kThreads = (kSWarp + 1) * 32;              // 512
constexpr int kCopyRowsPerPass = kCopyThreads / 8;       // rows one pass of the copy warps covers
constexpr int kCopyPasses = (kBN + kCopyRowsPerPass - 1) / kCopyRowsPerPass;
constexpr int kMaxStages = 6;
constexpr uint32_t kSlabKV = kBN * 128;  // one 64-column slab of a KV tile
constexpr uint32_t kSmemLimit = 232448 - 128;  // opt-in maximum, less room for static shared memory

// Fixed area at the start of shared memory.
constexpr uint32_t kOffBars = 0;                                   // 64 mbarriers
constexpr uint32_t kOffMapSrc = kOffBars + 64 * 8;                 // int32 [kMaxStages][64]
constexpr uint32_t kOffMapDelta = kOffMapSrc + kMaxStages * kBN * 4;
constexpr uint32_t kOffPhase = kOffMapDelta + kMaxStages * kBN * 4;  // uint64 [32]
constexpr uint32_t kOffTmemPtr = kOffPhase + 32 * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kOffHalfMax = kOffAbort + 12;          // float [2 halves][128 rows]: tile max
constexpr uint32_t kOffHalfL = kOffHalfMax + 2 * 128 * 4;   // float [2 halves][128 rows]: row sum
constexpr uint32_t kFixedBytes = 6144;
static_assert(kOffHalfL + 2 * 128 * 4 <= kFixedBytes, "fixed area overflow");

// Named barriers (0 is __syncthreads): the split-KV completion count, the softmax warps'
// final row sums, and per TMEM lane quadrant (the two warps that share its rows) the per-tile
// reduction and the rare second round of it.
constexpr int kBarSmMerge = 1;
constexpr int kBarSmRed2 = 3;
constexpr int kBarPairRed = 4;   // 4 .. 7
constexpr int kBarPairRed2 = 8;  // 8 .. 11

enum : int {
  BAR_KV_FULL = 0,                      // [kMaxStages] publishers published the tile (count 2)
  BAR_KV_EMPTY = BAR_KV_FULL + kMaxStages,  // [kMaxStages] UMMA commit after P.V of the stage
  BAR_LANDED = BAR_KV_EMPTY + kMaxStages,   // [kMaxStages] every copy thread's copies landed
  BAR_MAP = BAR_LANDED + kMaxStages,        // [kMaxStages] row map of the stage published
  BAR_S_FULL = BAR_MAP + kMaxStages,        // UMMA commit after Q.K^T into the score buffer
  BAR_S_EMPTY = BAR_S_FULL + 1,             // softmax warps loaded the score buffer (count 8)
  BAR_PV_DONE = BAR_S_EMPTY + 1,            // [2] UMMA commit after P.V of P buffer
  BAR_P_FULL = BAR_PV_DONE + 2,             // [2] softmax wrote P buffer (and rescaled O) (count 8)
  BAR_Q_FULL = BAR_P_FULL + 2,              // softmax warps stored Q in TMEM (count 8)
  BAR_X_FULL = BAR_Q_FULL + 1,              // peer's partial scores landed (1 arrive + tx)
  BAR_X_EMPTY = BAR_X_FULL + 1,             // peer's 8 softmax warps consumed our scores (remote)
  BAR_DRAIN = BAR_X_EMPTY + 1,              // [2] all UMMAs of the Q.K^T / P.V issuer done
  NUM_BARS = BAR_DRAIN + 2,
};
static_assert(NUM_BARS <= 64, "barrier area");

constexpr uint32_t kTmemO = 0;    // O half: 256 fp32 columns
constexpr uint32_t kTmemS = 256;  // score buffer: 64 fp32 columns
constexpr uint32_t kTmemP = 320;  // P double buffer: 2 x 32 columns of bf16 pairs
constexpr uint32_t kTmemQ = 384;  // Q, cKV slabs 0-3: 4 x 32 columns of bf16 pairs
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);   // A, B K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, 256, 0, 1);  // B (cKV tile) MN-major
constexpr float kLn2 = 0.6931471805599453f;

// Two fp32 values in one 64-bit register pair, and the paired fp32 FMA / add of sm_100 and
// later (each lane rounds exactly as fmaf / + would).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
constexpr uint32_t FULL = kFullMask;

// Shared-memory layout for a given number of stored query rows (Mv, multiple of 8), the same
// in both CTAs (the peer addresses the score exchange buffer through its own layout): the
// exchange buffer, the CTA's q_rope half (Mv rows x 128 B, first 64 B used), the KV stages'
// cKV slabs (4 per stage), then their k_r halves: stage s owns chunks 4 (s & 1) .. 4 (s & 1) + 3
// of k_r slab s / 2.
struct Layout {
  uint32_t x, qr, kv, kr, stage, total;
  int stages;
};
__host__ __device__ inline Layout make_layout(int Mv, int rank) {
  Layout L;
  L.x = kFixedBytes;                                // 8 x Mv 16-byte words (8 fp16 scores each)
  L.qr = L.x + (uint32_t)Mv * 128u;                 // Mv rows x 128 B
  (void)rank;
  const uint32_t end = L.qr + (uint32_t)Mv * 128u;
  L.kv = (end + 1023u) & ~1023u;
  L.stage = 4u * kSlabKV;  // cKV slabs of a stage; the k_r halves of stages 2i, 2i+1 share a slab
  const uint32_t avail = kSmemLimit - 1024u - L.kv;  // 1024: base alignment slack
  int st = kMaxStages;
  while (st > 0 && (uint32_t)st * L.stage + (uint32_t)((st + 1) / 2) * kSlabKV > avail) --st;
  L.stages = st;
  L.kr = L.kv + (uint32_t)st * L.stage;
  L.total = L.kr + (uint32_t)((st + 1) / 2) * kSlabKV + 1024u;
  return L;
}
__host__ __device__ inline uint32_t launch_smem(int Mv) {
  const uint32_t t0 = make_layout(Mv, 0).total, t1 = make_layout(Mv, 1).total;
  return t0 > t1 ? t0 : t1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_attn_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int last_sh;  // this CTA merges the split-KV partials of its query tile
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int col0 = (int)rank * 256;
  const int Mv = a.Mv;
  const Layout L = make_layout(Mv, (int)rank);
  const int NS = L.stages;
  auto kr_slab = [&](int st) -> uint32_t { return L.kr + (uint32_t)(st >> 1) * kSlabKV; };  // smem offset

  // ---- work unit: request b, query tile, KV split --------------------------------------
  // Split launch: grid (2 n_qtiles S, B), cluster x / 2 = qtile S + split.  Long-first launch
  // (one query tile per request, S = 2): grid (2 B, 2), split = y, so that every long split 0
  // precedes every short split 1 in the grid and the short ones fill the cluster slots left.
  const int b = a.long_first ? (int)(blockIdx.x >> 1) : (int)blockIdx.y;
  const int unit = a.long_first ? (int)blockIdx.y : (int)(blockIdx.x >> 1);
  const int qtile = unit / a.S, split = unit % a.S;
  // the chunk table: in the parameter block (small tables) or in the workspace
  const irm_chunk* chunks = a.inline_table ? a.tab.chunks : a.chunks;
  const int32_t* indptr = a.inline_table ? a.tab.indptr : a.indptr;
  int c_begin = indptr[b], c_end = indptr[b + 1];
  int ctx = 0;
  const bool table_ok = c_begin >= 0 && c_end > c_begin && c_end <= a.n_chunks;
  if (table_ok) {
    const irm_chunk last = chunks[c_end - 1];
    ctx = last.p_tgt + last.len;
  } else {
    c_begin = c_end = 0;
  }
  const int q0 = qtile * a.qpt;
  const int nq_tile = min(a.qpt, a.n_q - q0);
  const int rows_valid = nq_tile * a.H;
  const int pos_last = ctx - a.n_q + q0 + nq_tile - 1;
  const int kv_tiles = (table_ok && pos_last >= 0) ? (pos_last + kBN) / kBN : 0;
  // split boundaries at split * kv_tiles * num / den (the last one at kv_tiles): num / den = 1 / S,
  // or for the long-first launch the cut (in 1/4096)
  const int kb = (int)((int64_t)split * kv_tiles * a.split_num / a.split_den);
  const int ke = split == a.S - 1 ? kv_tiles : (int)((int64_t)(split + 1) * kv_tiles * a.split_num / a.split_den);
  const int ntiles = ke - kb;

  auto bar = [&](int i) -> uint32_t { return sb + kOffBars + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  int32_t* map_src = reinterpret_cast<int32_t*>(smem + kOffMapSrc);
  int32_t* map_delta = reinterpret_cast<int32_t*>(smem + kOffMapDelta);
  uint64_t* phaseF = reinterpret_cast<uint64_t*>(smem + kOffPhase);


  if (tid == 0) {
    last_sh = 0;
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), kPubWarps);
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
      mbar_init(bar(BAR_LANDED + s), kCopyThreads);
      mbar_init(bar(BAR_MAP + s), 1);
    }
    mbar_init(bar(BAR_S_FULL), 1);
    mbar_init(bar(BAR_S_EMPTY), kSoftmaxWarps);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_PV_DONE + s), 1);
      mbar_init(bar(BAR_P_FULL + s), kSoftmaxWarps);
    }
    mbar_init(bar(BAR_X_FULL), 1);
    mbar_init(bar(BAR_X_EMPTY), kSoftmaxWarps);
    mbar_init(bar(BAR_Q_FULL), kSoftmaxWarps);
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_DRAIN + 1), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (tid < 32) phaseF[tid] = a.phase.F[tid];
  if (warp == kMmaWarp) {
    tmem_alloc(sb + kOffTmemPtr, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // the peer's barriers exist before any remote traffic
  cluster_wait();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemPtr);
  // (checked only now, so that the set-up above does not wait for the chunk-table reads)
  if (tid == 0 && !table_ok) set_status(a.status, kDevErrBounds);

  // The softmax branch comes first: its loop is the hottest code of the kernel, and its place
  // in the binary measurably matters (instruction fetch is a top stall reason).
  if (warp < kSoftmaxWarps) {
    // ======================= softmax + epilogue (thread = query row) ===================
    // Warps w and w + 4 share TMEM lane quadrant w & 3; `half` 0 takes keys 0-31 of every
    // tile and O columns [0, 128) of this CTA's 256, half 1 keys 32-63 and columns [128, 256).
    const int half = warp >> 2;
    const int m = tid & (kBM - 1);
    const int wq = warp & 3;
    const bool warp_live = wq * 32 < Mv;       // this warp holds stored query rows
    const bool row_live = m < Mv;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + kTmemO + lane_base + 128u * (uint32_t)half;
    const int pos_m = (m < rows_valid) ? ctx - a.n_q + q0 + m / a.H : pos_last;
    const int pos_first = ctx - a.n_q + q0;  // position of the tile's first query
    float* half_max = reinterpret_cast<float*>(smem + kOffHalfMax);  // [2][128]
    float* half_l = reinterpret_cast<float*>(smem + kOffHalfL);      // [2][128]
    float m_run = -INFINITY, l_run = 0.f;  // m_run agrees in both halves; l_run is this half's
    // score exchange buffer, transposed ([8 words][Mv rows], word = 8 fp16 scores; words 0-3
    // hold keys 0-31, 4-7 keys 32-63) so that consecutive rows are consecutive 16-byte words:
    // conflict-free for both the peer's stores and our loads
    const uint32_t rX = mapa_shared(sb + L.x, peer);
    const uint32_t rXfull = mapa_shared(bar(BAR_X_FULL), peer);
    const uint32_t rXempty = mapa_shared(bar(BAR_X_EMPTY), peer);
    const uint4* X = reinterpret_cast<const uint4*>(smem + L.x);
    bool ok = true;
    // Q, this CTA's cKV columns, into TMEM: half h stores cKV slabs 2h, 2h + 1 of row m as
    // bf16 pairs (rows past the valid ones are zero; warps holding no stored rows leave their
    // lanes)
    if (ntiles > 0 && warp_live) {
      const bool valid = m < rows_valid;
      const int64_t row = valid ? ((int64_t)b * a.n_q + q0) * a.H + m : 0;
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_lat) +
                                                         row * kDLat + col0);
#pragma unroll 1
      for (int slab = 2 * half; slab < 2 * half + 2; ++slab) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = valid ? __ldg(qsrc + slab * 8 + i) : make_uint4(0u, 0u, 0u, 0u);
          r[4 * i] = v.x;
          r[4 * i + 1] = v.y;
          r[4 * i + 2] = v.z;
          r[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + kTmemQ + 32u * slab + lane_base, r);
      }
      tmem_st_wait();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(BAR_Q_FULL));
    // This half's partial scores of one tile (the CTA's share of the contraction), loaded from
    // the score buffer, which is released at once, and rounded to fp16 pairs exactly as the
    // peer receives them.
    auto load_scores = [&](int t, uint32_t (&w)[16]) -> bool {
      if (!warp_wait(bar(BAR_S_FULL), (uint32_t)t & 1u, abort_flag)) return false;
      tc_fence_after();
      uint32_t r[32];
      if (warp_live) {
        tmem_ld32(tmem + kTmemS + 32u * (uint32_t)half + lane_base, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_S_EMPTY));
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        w[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      return true;
    };
    // Ship them to the peer's exchange buffer (transposed: word (4 half + i) of row m).
    auto send_scores = [&](const uint32_t (&w)[16]) {
      if (row_live) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_async_v4_b32(rX + (uint32_t)((4 * half + i) * Mv + m) * 16u,
                          make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]), rXfull);
      }
    };
    // Software pipeline: iteration j combines tile j's own and peer partials, loads tile
    // j+1's scores (freeing the score buffer for the next Q.K^T), ships them once the peer
    // has read tile j's (normally long since), and runs tile j's softmax.  P goes to its own
    // double buffer, so the score buffer never waits for a P.V.
    uint32_t own[16];  // this half's partial scores of the tile in flight (fp16 pairs)
    if (ntiles > 0) {
      if (m == 0 && half == 0) mbar_arrive_expect_tx(bar(BAR_X_FULL), (uint32_t)Mv * kBN * 2u);
      ok = load_scores(0, own);
      if (ok) send_scores(own);
    }
    // Every softmax warp runs every iteration up to the tile's barrier reduction, also after a
    // failed wait (it then skips its work): the reduction tells both warps of a quadrant of a
    // failure, and they leave the loop together, so no warp is left waiting at a named
    // barrier; the abort flag they raise makes the other quadrants' waits give up as well.
    for (int j = 0; j < ntiles; ++j) {
      const int T = (kb + j) * kBN + 32 * half;  // position of this half's first key
      const bool more = j + 1 < ntiles;
      // the peer's partial scores of tile j
      if (ok) ok = warp_wait_cluster(bar(BAR_X_FULL), (uint32_t)j & 1u, abort_flag);
      float sv[32];
      float lmx = -INFINITY;
      bool need = false;
      if (ok) {
        // the barrier's next phase expects the peer's tile j+1 bytes
        if (more && m == 0 && half == 0) mbar_arrive_expect_tx(bar(BAR_X_FULL), (uint32_t)Mv * kBN * 2u);
        if (row_live) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = X[(4 * half + i) * Mv + m];
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = add_f16x2_f16x2_f32(own[4 * i + k], vv[k]);
              sv[8 * i + 2 * k] = f.x;
              sv[8 * i + 2 * k + 1] = f.y;
            }
          }
        }
        __syncwarp();
        // this warp is done with the peer's scores (the values are in registers and used, so
        // a relaxed arrive suffices; a release would stall on this lane's outstanding st.async)
        if (lane == 0) mbar_arrive_remote_relaxed(rXempty);
        // tile j+1's scores (own[] is free again), shipped once the peer has read tile j's
        if (more) {
          ok = load_scores(j + 1, own);
          if (ok) ok = warp_wait_cluster(bar(BAR_X_EMPTY), (uint32_t)j & 1u, abort_flag);
          if (ok) send_scores(own);
        }
      }
      if (ok) {
        if (row_live) {
          // causal mask t <= pos_m, only on tiles that reach past the tile's first query
          if (T + 31 > pos_first) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (T + i > pos_m) sv[i] = -INFINITY;
          }
          // this half's row max, three-input max tree (scale > 0, so max(s) * scale =
          // max(s * scale))
          float t[11];
#pragma unroll
          for (int i = 0; i < 10; ++i) t[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          t[10] = fmaxf(sv[30], sv[31]);
          const float u0 = fmax3(t[0], t[1], t[2]), u1 = fmax3(t[3], t[4], t[5]);
          const float u2 = fmax3(t[6], t[7], t[8]), u3 = fmaxf(t[9], t[10]);
          lmx = fmaxf(fmax3(u0, u1, u2), u3) * a.scale_log2;  // log2 units
          // The running max only moves when it grows by more than 2^8: P stays <= 256 and O
          // is rescaled rarely (the final 1/l uses the same max, so the result is exact).
          need = (m < rows_valid) && (lmx > m_run + 8.f);
        }
      }
      // One reduction per tile over the quadrant's two warps (both halves of its rows): it
      // flags the rare tile where a row's max moves or a wait failed (and a second one agrees
      // on the new max or on leaving).
      if (named_bar_red_or(kBarPairRed + wq, 64, need || !ok)) {
        half_max[half * kBM + m] = lmx;
        if (named_bar_red_or(kBarPairRed2 + wq, 64, !ok)) {
          ok = false;
          *abort_flag = 1;  // the other quadrants' waits give up too
          break;
        }
        lmx = fmaxf(lmx, half_max[(half ^ 1) * kBM + m]);  // the row's max over both halves
      }
      const bool want = (m < rows_valid) && (lmx > m_run + 8.f);  // same in both halves
      const float corr = want ? fast_exp2(m_run - lmx) : 1.f;
      if (j > 0 && __any_sync(FULL, want)) {
        // rescale this half's O columns once the previous tile's P.V is complete
        if (warp_wait(bar(BAR_PV_DONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
            tmem_st32(tO + c, r);
          }
          tmem_st_wait();
        } else {
          ok = false;  // reported at the next tile's reduction (or after the loop)
        }
      }
      if (want) {
        l_run *= corr;
        m_run = lmx;
      }
      uint32_t pk[16];
      if (row_live) {
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t c2 = f2_pack(a.scale_log2, a.scale_log2), m2 = f2_pack(-m_use, -m_use);
        uint64_t part[2] = {0ull, 0ull};  // paired partial sums
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = f2_unpack(f2_fma(f2_pack(sv[i], sv[i + 1]), c2, m2));
          const float p0 = fast_exp2(x.x);
          const float p1 = fast_exp2(x.y);
          part[(i >> 1) & 1] = f2_add(part[(i >> 1) & 1], f2_pack(p0, p1));
          const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
          pk[i >> 1] = *reinterpret_cast<const uint32_t*>(&h);
        }
        const float2 s01 = f2_unpack(f2_add(part[0], part[1]));
        l_run += s01.x + s01.y;
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
      }
      // P buffer j&1 is free once the P.V of tile j-2 has completed; this half's 32 keys are
      // its columns 16 * half .. 16 * half + 15 (bf16 pairs)
      if (ok && j >= 2) ok = warp_wait(bar(BAR_PV_DONE + (j & 1)), ((j - 2) >> 1) & 1, abort_flag);
      if (ok && warp_live) {
        tc_fence_after();
        tmem_st16(tmem + kTmemP + 32u * (uint32_t)(j & 1) + 16u * (uint32_t)half + lane_base, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + (j & 1)));
    }
    if (ok && ntiles > 0)
      ok = warp_wait(bar(BAR_PV_DONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, abort_flag);
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
    tc_fence_after();
    // the row's sum over both halves
    half_l[half * kBM + m] = l_run;
    named_bar_sync(kBarSmRed2, kSoftmaxThreads);
    const float l_tot = l_run + half_l[(half ^ 1) * kBM + m];
    // ---- epilogue: O / l for this half's 128 of the CTA's 256 columns -------------------
    if (warp_live) {
      const bool have = ntiles > 0 && ok && l_tot > 0.f;
      const float inv_l = have ? 1.f / l_tot : 0.f;
      const float lse_v = have ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
      const bool write_row = m < rows_valid;
      const int qi = q0 + (write_row ? m / a.H : 0), hh = write_row ? m % a.H : 0;
      const int64_t orow = ((int64_t)b * a.n_q + qi) * a.H + hh;
      const int64_t prow = ((int64_t)b * a.n_qtiles * a.S + unit) * kBM + m;
      const int cbase = col0 + 128 * half;
      for (int c = 0; c < 128; c += 32) {
        uint32_t r[32];
        if (ntiles > 0) {
          tmem_ld32(tO + c, r);  // warp-collective: every lane executes it
          tmem_ld_wait();
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = have ? __uint_as_float(r[i]) * inv_l : 0.f;
        if (!write_row) continue;
        if (a.S == 1) {
          uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * kDLat +
                                              cbase + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * q + 0], v[8 * q + 1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * q + 2], v[8 * q + 3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * q + 4], v[8 * q + 5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * q + 6], v[8 * q + 7]);
            w.x = *reinterpret_cast<uint32_t*>(&h0);
            w.y = *reinterpret_cast<uint32_t*>(&h1);
            w.z = *reinterpret_cast<uint32_t*>(&h2);
            w.w = *reinterpret_cast<uint32_t*>(&h3);
            o[q] = w;
          }
        } else {
          float4* o = reinterpret_cast<float4*>(a.opart + prow * kDLat + cbase + c);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      if (write_row && half == 0) {
        if (a.S == 1) {
          if (a.lse != nullptr && rank == 0) a.lse[orow] = lse_v;
        } else {
          a.lsepart[(int64_t)rank * a.B * a.n_qtiles * a.S * kBM + prow] = lse_v;
        }
      }
    }
    if (a.S > 1) {
      // Split-KV merge, fused: the last CTA (per rank) to finish a query tile merges the S
      // partials of its 256 columns after teardown (threadfence-reduction pattern; the
      // counter resets itself, so the workspace stays reusable).
      __threadfence();
      named_bar_sync(kBarSmMerge, kSoftmaxThreads);
      if (tid == 0) {
        int* cnt = a.counters + ((int64_t)b * a.n_qtiles + qtile) * 2 + rank;
        last_sh = (atomicAdd(cnt, 1) == a.S - 1) ? 1 : 0;
      }
    }
  
  } else if (warp < kMmaWarp) {
    // ======================= loaders =====================================================
    // Warps 8-9 gather KV rows with cp.async following the row maps that warp 14 builds from
    // the chunk table; warps 10-11 wait for each tile's bytes to land, rotate this CTA's k_r pairs by
    // R(delta) in shared memory and publish the tile.  Every role blocks in mbarrier waits, so
    // no loader warp spins for issue slots the softmax warps need, and the copies run up to NS
    // tiles ahead.  The Q.K^T issuer fences the bytes for the async proxy after acquiring
    // KV_FULL (a writer's own fence would also wait for its copies of later tiles in flight).
    const int lw = warp - kSoftmaxWarps;  // 0-1 copy warps, 2-3 publishers
    bool ok = true;
    if (lw < kCopyWarps) {
      const int tp = tid - kSoftmaxWarps * 32;  // 0 .. kCopyThreads - 1
      const int chk = tp & 7;     // 16-byte chunk of a 128-byte slab row
      const int rsub = tp >> 3;   // row within a group of kCopyThreads / 8
      const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(a.q_rope);
      const __nv_bfloat16* kvp = static_cast<const __nv_bfloat16*>(a.kv);
      // Stored chunk c (0..3) of this CTA's k_r / q_rope half: the 16-byte chunk
      // half_chunk(c) of the 64 rope columns (NeoX: its pairs' first then second halves;
      // interleaved: four contiguous chunks).
      const int kr_col = chk < 4 ? 8 * half_chunk(a.interleaved, (int)rank, chk) : 0;
      // The CTA's q_rope half: Mv rows (rows past the tile's valid rows are zero filled); it
      // lands with the first KV tile (same cp.async group).
      if (ntiles > 0 && chk < 4) {
        // tile row m is (query q0 + m / H, head m % H): global row (b n_q + q0) H + m
        const int64_t row0 = ((int64_t)b * a.n_q + q0) * a.H;
        for (int m = rsub; m < Mv; m += kCopyThreads / 8) {
          const bool valid = m < rows_valid;
          const int64_t row = valid ? row0 + m : 0;
          const void* src = valid ? (const void*)(qr + row * kDRope + kr_col) : a.q_rope;
          cp_async_16(sb + L.qr + sw128_offset(m, chk), src, valid ? 16u : 0u);
        }
      }
      int s = 0;
      uint32_t ph = 0;
      for (int j = 0; j < ntiles; ++j) {
        // stage s is free once the P.V of tile j-NS completed
        if (j >= NS && !(ok = warp_wait(bar(BAR_KV_EMPTY + s), ph ^ 1u, abort_flag))) break;
        if (!(ok = warp_wait(bar(BAR_MAP + s), ph, abort_flag))) break;
        const uint32_t stage = sb + L.kv + (uint32_t)s * L.stage;
        // all of this thread's source rows first, then every copy of the tile back to back
        int srs[kCopyPasses];
#pragma unroll
        for (int p = 0; p < kCopyPasses; ++p) {
          const int row = p * kCopyRowsPerPass + rsub;
          srs[p] = row < kBN ? map_src[s * kBN + row] : -1;
        }
#pragma unroll
        for (int p = 0; p < kCopyPasses; ++p) {
          const int row = p * kCopyRowsPerPass + rsub;
          if (row >= kBN) break;
          const int sr = srs[p];
          const __nv_bfloat16* kvrow = kvp + (int64_t)(sr >= 0 ? sr : 0) * kDRow;
          const __nv_bfloat16* rowp = kvrow + col0 + chk * 8;
          const uint32_t dst = stage + sw128_offset(row, chk);
          const uint32_t nb = sr >= 0 ? 16u : 0u;
#pragma unroll
          for (int slab = 0; slab < 4; ++slab) cp_async_16(dst + slab * kSlabKV, rowp + slab * 64, nb);
          if (chk < 4)
            cp_async_16(sb + kr_slab(s) + sw128_offset(row, chk + 4 * (s & 1)), kvrow + kDLat + kr_col, nb);
        }
        cp_async_arrive_noinc(bar(BAR_LANDED + s));
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
      cp_async_wait_all();
    } else {
      // publisher pb owns rows 32 pb .. 32 pb + 31 of every tile; each 16-row half keeps its
      // lane's last (cos, sin) (recomputed only when the row's delta changes)
      const int pb = lw - kCopyWarps;
      int dprev[2] = {0, 0};
      float cs_c[2][8], cs_s[2][8];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cs_c[h][e] = 1.f;
          cs_s[h][e] = 0.f;
        }
      int s = 0;
      uint32_t ph = 0;
      for (int j = 0; j < ntiles; ++j) {
        if (!(ok = warp_wait(bar(BAR_LANDED + s), ph, abort_flag))) break;
        if (!(ok = warp_wait(bar(BAR_MAP + s), ph, abort_flag))) break;  // orders the map's deltas
#pragma unroll
        for (int h = 0; h < 2; ++h)
          rotate_krope_half_16rows(smem + kr_slab(s), map_delta + s * kBN, phaseF, a.interleaved, (int)rank,
                                   32 * pb + 16 * h,
                                   4 * (s & 1), lane, dprev[h], cs_c[h], cs_s[h]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_KV_FULL + s));
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
  } else if (warp == kSWarp) {
    // ======================= Q.K^T issuer (one thread) ===================================
    // (warp 15, the only one of its SM sub-partition besides two softmax warps and a
    // publisher: its issue slots are the least contended)
    if (lane == 0 && ntiles > 0) {
      bool ok = mbar_wait(bar(BAR_Q_FULL), 0, abort_flag);
      tc_fence_after();
      int ss = 0;
      uint32_t phs = 0;  // kv_full parity of stage ss
      const uint64_t aq = sdesc_sw128(sb + L.qr, 16, 1024);  // the q_rope half (A, K-major)
      for (int ns = 0; ns < ntiles && ok; ++ns) {
        if (!(ok = mbar_wait(bar(BAR_KV_FULL + ss), phs, abort_flag))) break;
        // the score buffer is free once the softmax warps have loaded tile ns-1's scores
        if (ns >= 1 && !(ok = mbar_wait(bar(BAR_S_EMPTY), (ns - 1) & 1, abort_flag))) break;
        // the tile's bytes (cp.async-written and rotated) -> async proxy before the UMMA reads
        tc_fence_after();
        fence_proxy_async_smem();
        const uint64_t bd = sdesc_sw128(sb + L.kv + (uint32_t)ss * L.stage, 16, 1024);
        const uint64_t bk = sdesc_sw128(sb + kr_slab(ss) + (ss & 1) * 64, 16, 1024);
        const uint32_t tS = tmem + kTmemS;
#pragma unroll
        for (int slab = 0; slab < 4; ++slab) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_ts(tS, tmem + kTmemQ + 32u * slab + 8u * kk, sdesc_add(bd, slab * kSlabKV + kk * 32),
                         kIdescS, (slab | kk) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)  // the half k_r slab: 32 columns, 2 K-steps
          umma_bf16(tS, sdesc_add(aq, kk * 32), sdesc_add(bk, kk * 32), kIdescS, 1u);
        umma_commit(bar(BAR_S_FULL));
        if (++ss == NS) {
          ss = 0;
          phs ^= 1u;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, kDevErrTimeout);
      }
      umma_commit(bar(BAR_DRAIN));
      if (!mbar_wait(bar(BAR_DRAIN), 0, nullptr)) set_status(a.status, kDevErrTimeout);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // TMEM allocation and release only
  } else if (warp == kMapWarp) {
    // ======================= row maps ====================================================
    // A window of 32 chunk records (one per lane) turned into each tile's row map: source
    // row (-1 = outside the context, zero filled) and delta.  The map of tile j goes into
    // slot j % NS once tile j-NS has been published (its copies issued and its k_r rotated),
    // so maps are ready up to NS tiles ahead of the copies.
    ChunkWindow cw;
    cw.chunks = chunks;
    cw.c_end = c_end;
    cw.win = c_begin;
    bool ok = true;
    if (ntiles > 0) {
      if (kb == 0) {
        cw.load(lane);  // the request's first chunk starts at position 0
      } else {
        cw.seek(c_begin, kb * kBN, lane);
      }
    }
    int s = 0;
    uint32_t ph = 0;
    for (int j = 0; j < ntiles; ++j) {
      if (j >= NS && !(ok = warp_wait(bar(BAR_KV_FULL + s), ph ^ 1u, abort_flag))) break;
      cw.build_map((kb + j) * kBN, ctx, a.n_rows, map_src + s * kBN, map_delta + s * kBN, a.status, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_MAP + s));
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
  } else if (warp == kPvWarp) {
    // ======================= P.V issuer (one thread) =====================================
    if (lane == 0 && ntiles > 0) {
      const uint32_t tO = tmem + kTmemO;
      bool ok = true;
      int sp = 0;
      for (int np = 0; np < ntiles && ok; ++np) {
        if (!(ok = mbar_wait(bar(BAR_P_FULL + (np & 1)), (np >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t bv = sdesc_sw128(sb + L.kv + (uint32_t)sp * L.stage, kSlabKV, 1024);
        const uint32_t tP = tmem + kTmemP + 32u * (uint32_t)(np & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ts(tO, tP + 8u * kk, sdesc_add(bv, kk * 2048), kIdescPV, (np > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(BAR_KV_EMPTY + sp));
        umma_commit(bar(BAR_PV_DONE + (np & 1)));
        if (++sp == NS) sp = 0;
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, kDevErrTimeout);
      }
      umma_commit(bar(BAR_DRAIN + 1));
      if (!mbar_wait(bar(BAR_DRAIN + 1), 0, nullptr)) set_status(a.status, kDevErrTimeout);
    }
    __syncwarp();
  }
  // ---- teardown ---------------------------------------------------------------------
  __syncthreads();
  cluster_arrive();  // the peer no longer sends to this CTA's shared memory
  cluster_wait();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (a.S > 1 && last_sh) {
    // Merge, staged through shared memory (the pipeline is done): for a block of rows, every
    // partial's 256 columns of this rank are fetched with one burst of cp.async, then each
    // (row, 4-column group) item is merged from shared memory.
    __threadfence();
    const float* lse_r = a.lsepart + (int64_t)rank * a.B * a.n_qtiles * a.S * kBM;
    const int64_t ubase = ((int64_t)b * a.n_qtiles + qtile) * a.S;  // first unit of the tile
    const uint32_t per_row = (uint32_t)a.S * (1024u + 4u);           // partial O row half + lse
    const int rows_blk = max(1, min(rows_valid, (int)((L.total - 1024u) / per_row)));
    float* so = reinterpret_cast<float*>(smem);                       // [S][rows_blk][256]
    float* sl = so + (size_t)a.S * rows_blk * 256;                    // [S][rows_blk]
    for (int r0 = 0; r0 < rows_valid; r0 += rows_blk) {
      const int nr = min(rows_blk, rows_valid - r0);
      const int n16 = a.S * nr * 64;
      for (int it = tid; it < n16; it += kThreads) {
        const int c16 = it & 63, rr = (it >> 6) % nr, sp = (it >> 6) / nr;
        const float* src = a.opart + ((ubase + sp) * kBM + r0 + rr) * kDLat + col0 + c16 * 4;
        cp_async_16(smem_u32(so + ((size_t)(sp * rows_blk + rr) * 256 + c16 * 4)), src, 16u);
      }
      cp_async_commit();
      for (int it = tid; it < a.S * nr; it += kThreads) {
        const int rr = it % nr, sp = it / nr;
        sl[sp * rows_blk + rr] = lse_r[(ubase + sp) * kBM + r0 + rr];
      }
      cp_async_wait_all();
      __syncthreads();
      for (int it = tid; it < nr * 64; it += kThreads) {
        const int rr = it >> 6, c4 = it & 63;
        float mx = -INFINITY;
        for (int sp = 0; sp < a.S; ++sp) mx = fmaxf(mx, sl[sp * rows_blk + rr]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (mx != -INFINITY) {
          for (int sp = 0; sp < a.S; ++sp) {
            const float l = sl[sp * rows_blk + rr];
            const float w = (l == -INFINITY) ? 0.f : __expf(l - mx);
            const float4 v = reinterpret_cast<const float4*>(so + (size_t)(sp * rows_blk + rr) * 256)[c4];
            wsum += w;
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
          }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        const int mm = r0 + rr;
        const int qi = q0 + mm / a.H, hh = mm % a.H;
        const int64_t orow = ((int64_t)b * a.n_q + qi) * a.H + hh;
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 w2;
        w2.x = *reinterpret_cast<const uint32_t*>(&h0);
        w2.y = *reinterpret_cast<const uint32_t*>(&h1);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * kDLat + col0 + c4 * 4) = w2;
        if (c4 == 0 && rank == 0 && a.lse != nullptr)
          a.lse[orow] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
      }
      __syncthreads();
    }
    __syncthreads();
    if (tid == 0) a.counters[((int64_t)b * a.n_qtiles + qtile) * 2 + rank] = 0;
  }
}

}  // namespace

size_t attn_smem_bytes(int Mv) { return launch_smem(Mv); }

namespace {
// The kernel's dynamic shared memory limit belongs to the device: raised when a launch needs
// more than what was set on this device before.
cudaError_t raise_smem_limit(uint32_t smem) {
  static std::mutex mu;
  static uint32_t set_to[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 0 || dev >= 128 || set_to[dev] < smem) {
    e = cudaFuncSetAttribute(mla_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) set_to[dev] = smem;
  }
  return cudaSuccess;
}
}  // namespace

int attn_max_active_clusters(int Mv) {
  const uint32_t smem = launch_smem(Mv);
  if (raise_smem_limit(smem) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_attn_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_mla_attn(const AttnArgs& a, cudaStream_t stream) {
  if (make_layout(a.Mv, 0).stages < 2 || make_layout(a.Mv, 1).stages < 2)
    return cudaErrorInvalidConfiguration;
  if (a.long_first && (a.S != 2 || a.n_qtiles != 1)) return cudaErrorInvalidConfiguration;
  const uint32_t smem = launch_smem(a.Mv);
  cudaError_t e = raise_smem_limit(smem);
  if (e != cudaSuccess) return e;
  const dim3 grid = a.long_first ? dim3(2 * a.B, 2) : dim3(2 * a.n_qtiles * a.S, a.B);
  mla_attn_kernel<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irm
