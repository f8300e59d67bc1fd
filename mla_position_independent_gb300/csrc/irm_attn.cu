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
//   - The [cKV | k_r] contraction of Q K^T is split by columns: CTA 0 owns cKV[0:256),
//     CTA 1 owns cKV[256:512) and k_r (and therefore the rotation).  Each CTA loads only
//     its own columns of every KV row, so each row is read from memory exactly once.
//   - Each CTA computes its partial scores S_r = Q_r K_r^T (tcgen05, M=128, N=64) into
//     TMEM and ships them to the peer with st.async; both add the two partials in the
//     same way and run the identical online softmax, so P is bit-identical in both.
//   - The output is split the same way: CTA r accumulates O[:, 256r:256r+256) += P V_r
//     (tcgen05, M=128, N=256) in TMEM, with V_r = the cKV columns it already holds.
//   - Warp roles: warps 0-3 softmax (thread = TMEM lane = query row), warps 4-7 load
//     tiles with cp.async (row gather following the chunk table) and rotate k_r, warp 8
//     allocates TMEM and issues the UMMAs.
// Every pipeline wait is bounded (2 s) and reports a timeout in the status word.
#include <cuda_runtime.h>
#include <climits>
#include <cmath>

#include "irm_common.cuh"
#include "irm_internal.h"

namespace irm {
namespace {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 64;   // KV rows per tile
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxSlabs = 5;                      // 64-column slabs per CTA (4 or 5)
constexpr uint32_t kSlabQ = kBM * 128;            // bytes of one Q slab
constexpr uint32_t kSlabKV = kBN * 128;           // bytes of one KV slab
constexpr uint32_t kStage = kMaxSlabs * kSlabKV;  // one KV pipeline stage
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kMaxSlabs * kSlabQ;
constexpr uint32_t kOffP = kOffKV + 2 * kStage;
constexpr uint32_t kOffX = kOffP + kBM * 128;
constexpr uint32_t kOffMisc = kOffX + kBM * kBN * 4;
constexpr uint32_t kOffMapSrc = kOffMisc + 32 * 8;
constexpr uint32_t kOffMapDelta = kOffMapSrc + 2 * kBN * 4;
constexpr uint32_t kOffPhase = kOffMapDelta + 2 * kBN * 4;
constexpr uint32_t kOffTmemPtr = kOffPhase + 32 * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kMiscBytes = 2048;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + base alignment slack
static_assert(kOffAbort + 4 <= kOffMisc + kMiscBytes, "misc area overflow");
static_assert(kSmemBytes <= 232448, "shared memory budget");

enum : int {
  BAR_KV_FULL = 0,   // [2] producers -> MMA (count 4: one arrive per producer warp)
  BAR_KV_EMPTY = 2,  // [2] MMA commit after P.V of the stage
  BAR_S_FULL = 4,    // [2] MMA commit after Q.K^T into S buffer
  BAR_S_EMPTY = 6,   // [2] softmax warps read S (count 4)
  BAR_P_FULL = 8,    // softmax wrote P (and rescaled O) (count 4)
  BAR_PV_DONE = 9,   // MMA commit after P.V
  BAR_X_FULL = 10,   // peer's partial scores landed (1 arrive + tx bytes)
  BAR_X_EMPTY = 11,  // peer consumed our partial scores (remote arrive)
  BAR_DRAIN = 12,    // all UMMAs done before TMEM is released
  BAR_MAP = 13,      // [2] producer warp 0 published the tile's row map (count 1)
  BAR_LANDED = 15,   // [2] every producer warp's copies of the tile landed (count 4)
  BAR_X_READ = 17,   // every softmax warp read the peer's partial scores (count 4)
  NUM_BARS = 18,
};

constexpr uint32_t kTmemO = 0;     // O half: 256 fp32 columns
constexpr uint32_t kTmemS = 256;   // S double buffer: 2 x 64 columns
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);    // A, B K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, 256, 0, 1);   // B (cKV tile) MN-major
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t FULL = 0xffffffffu;

// Warp-uniform bounded wait: every lane polls (and so acquires) the barrier, and the
// verdict is agreed with __all_sync so no lane leaves a loop its warp-mates stay in.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(FULL, ok);
}
__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort_flag) {
  const bool ok = mbar_wait_cluster(bar, parity, abort_flag);
  return __all_sync(FULL, ok);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_attn_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int nslab = rank == 0 ? 4 : 5;
  const int col0 = (int)rank * 256;

  // ---- work unit: request b, query tile, KV split --------------------------------------
  const int b = blockIdx.y;
  const int unit = blockIdx.x >> 1;
  const int qtile = unit / a.S, split = unit % a.S;
  int c_begin = a.indptr[b], c_end = a.indptr[b + 1];
  int ctx = 0;
  bool table_ok = c_begin >= 0 && c_end > c_begin && c_end <= a.n_chunks;
  if (table_ok) {
    const irm_chunk last = a.chunks[c_end - 1];
    ctx = last.p_tgt + last.len;
  } else {
    c_begin = c_end = 0;
  }
  const int q0 = qtile * a.qpt;
  const int nq_tile = min(a.qpt, a.n_q - q0);
  const int rows_valid = nq_tile * a.H;
  const int pos_last = ctx - a.n_q + q0 + nq_tile - 1;
  const int kv_tiles = (table_ok && pos_last >= 0) ? (pos_last + kBN) / kBN : 0;
  const int kb = (int)((int64_t)split * kv_tiles / a.S);
  const int ke = (int)((int64_t)(split + 1) * kv_tiles / a.S);
  const int ntiles = ke - kb;

  auto bar = [&](int i) -> uint32_t { return sb + kOffMisc + 8u * (uint32_t)i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  int32_t* map_src = reinterpret_cast<int32_t*>(smem + kOffMapSrc);
  int32_t* map_delta = reinterpret_cast<int32_t*>(smem + kOffMapDelta);
  uint64_t* phaseF = reinterpret_cast<uint64_t*>(smem + kOffPhase);

  if (tid == 0) {
    if (!table_ok) set_status(a.status, kDevErrBounds);
    mbar_init(bar(BAR_KV_FULL), kProducerWarps);
    mbar_init(bar(BAR_KV_FULL + 1), kProducerWarps);
    mbar_init(bar(BAR_KV_EMPTY), 1);
    mbar_init(bar(BAR_KV_EMPTY + 1), 1);
    mbar_init(bar(BAR_S_FULL), 1);
    mbar_init(bar(BAR_S_FULL + 1), 1);
    mbar_init(bar(BAR_S_EMPTY), kSoftmaxWarps);
    mbar_init(bar(BAR_S_EMPTY + 1), kSoftmaxWarps);
    mbar_init(bar(BAR_P_FULL), kSoftmaxWarps);
    mbar_init(bar(BAR_PV_DONE), 1);
    mbar_init(bar(BAR_X_FULL), 1);
    mbar_init(bar(BAR_X_EMPTY), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    mbar_init(bar(BAR_MAP), 1);
    mbar_init(bar(BAR_MAP + 1), 1);
    mbar_init(bar(BAR_LANDED), kProducerWarps);
    mbar_init(bar(BAR_LANDED + 1), kProducerWarps);
    mbar_init(bar(BAR_X_READ), kSoftmaxWarps);
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

  if (warp >= kSoftmaxWarps && warp < kMmaWarp) {
    // ======================= producers: gather, rotate, publish ========================
    const int tp = tid - kSoftmaxWarps * 32;
    const int pw = warp - kSoftmaxWarps;
    const __nv_bfloat16* ql = static_cast<const __nv_bfloat16*>(a.q_lat);
    const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(a.q_rope);
    const __nv_bfloat16* kvp = static_cast<const __nv_bfloat16*>(a.kv);
    const int per_row = nslab * 8;  // 16-byte chunks per row owned by this CTA

    // Q columns of this CTA, 128 rows (rows past the tile's valid rows are zero).
    for (int idx = tp; idx < kBM * per_row; idx += 128) {
      const int m = idx / per_row, rem = idx - m * per_row, slab = rem >> 3, chk = rem & 7;
      const void* src = a.q_lat;
      uint32_t nbytes = 0;
      if (m < rows_valid && ntiles > 0) {
        const int qi = q0 + m / a.H, h = m % a.H;
        const int64_t row = ((int64_t)b * a.n_q + qi) * a.H + h;
        src = (slab < 4) ? (const void*)(ql + row * kDLat + col0 + slab * 64 + chk * 8)
                         : (const void*)(qr + row * kDRope + chk * 8);
        nbytes = 16;
      }
      cp_async_16(sb + kOffQ + slab * kSlabQ + sw128_offset(m, chk), src, nbytes);
    }
    cp_async_commit();

    // Producer warp 0 keeps a window of 32 chunk records (one per lane) and turns it into
    // per-tile row maps: source row (-1 = outside the context, zero filled) and delta.
    int win = c_begin;
    int w_start = INT_MAX, w_end = INT_MAX, w_delta = 0;
    long long w_off = 0;
    auto load_window = [&]() {
      const int c = win + lane;
      if (c < c_end) {
        const irm_chunk ch = a.chunks[c];
        w_start = ch.p_tgt;
        w_end = ch.p_tgt + ch.len;
        w_off = ch.pool_offset;
        w_delta = ch.reused ? ch.p_tgt - ch.p_src : 0;
      } else {
        w_start = INT_MAX;
        w_end = INT_MAX;
        w_off = 0;
        w_delta = 0;
      }
    };
    if (pw == 0 && ntiles > 0) {
      const int T0 = kb * kBN;  // find the last chunk with p_tgt <= T0
      int lo = c_begin, hi = c_end;
      while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int c = lo + lane * step;
        const bool le = (c < hi) && (a.chunks[c].p_tgt <= T0);
        const unsigned msk = __ballot_sync(FULL, le);
        const int k = msk ? 31 - __clz((int)msk) : 0;
        lo = lo + k * step;
        hi = min(hi, lo + step);
      }
      win = lo;
      load_window();
    }
    auto build_map = [&](int T, int s) {
      const int t0 = T + lane, t1 = T + lane + 32;
      int src0 = -1, src1 = -1, d0 = 0, d1 = 0;
      bool need0 = t0 < ctx, need1 = t1 < ctx;
      for (int guard = 0; guard < kBN + 1; ++guard) {
        const int nvalid = min(32, c_end - win);
        if (!__any_sync(FULL, need0 || need1)) break;
        if (nvalid <= 0) {  // the device table does not cover the context
          if (lane == 0) set_status(a.status, kDevErrBounds);
          break;
        }
        const int last_end = __shfl_sync(FULL, w_end, nvalid - 1);
        int k0 = 0, k1 = 0;
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const int c0 = k0 + step, c1 = k1 + step;
          const int s0 = __shfl_sync(FULL, w_start, c0 & 31);
          const int s1 = __shfl_sync(FULL, w_start, c1 & 31);
          if (c0 < nvalid && s0 <= t0) k0 = c0;
          if (c1 < nvalid && s1 <= t1) k1 = c1;
        }
        const int st0 = __shfl_sync(FULL, w_start, k0), st1 = __shfl_sync(FULL, w_start, k1);
        const long long of0 = __shfl_sync(FULL, w_off, k0), of1 = __shfl_sync(FULL, w_off, k1);
        const int dd0 = __shfl_sync(FULL, w_delta, k0), dd1 = __shfl_sync(FULL, w_delta, k1);
        if (need0 && t0 < last_end) {
          const long long r = of0 + (t0 - st0);
          if (r < 0 || r >= a.n_rows) set_status(a.status, kDevErrBounds); else src0 = (int)r;
          d0 = dd0;
          need0 = false;
        }
        if (need1 && t1 < last_end) {
          const long long r = of1 + (t1 - st1);
          if (r < 0 || r >= a.n_rows) set_status(a.status, kDevErrBounds); else src1 = (int)r;
          d1 = dd1;
          need1 = false;
        }
        if (!__any_sync(FULL, need0 || need1)) break;
        win += nvalid;
        load_window();
      }
      map_src[s * kBN + lane] = src0;
      map_src[s * kBN + lane + 32] = src1;
      map_delta[s * kBN + lane] = d0;
      map_delta[s * kBN + lane + 32] = d1;
    };

    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      // stage s is free once the P.V of tile j-2 completed (that also means every producer
      // finished reading the row map of tile j-2, which shares buffer s)
      if (j >= 2 && !(ok = warp_wait(bar(BAR_KV_EMPTY + s), ph ^ 1u, abort_flag))) break;
      if (pw == 0) {
        build_map((kb + j) * kBN, s);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_MAP + s));
      }
      if (!(ok = warp_wait(bar(BAR_MAP + s), ph, abort_flag))) break;
      const uint32_t stage = sb + kOffKV + (uint32_t)s * kStage;
      for (int idx = tp; idx < kBN * per_row; idx += 128) {
        const int row = idx / per_row, rem = idx - row * per_row, slab = rem >> 3, chk = rem & 7;
        const int sr = map_src[s * kBN + row];
        const void* src = a.kv;
        uint32_t nbytes = 0;
        if (sr >= 0) {
          src = kvp + (int64_t)sr * kDRow + col0 + slab * 64 + chk * 8;
          nbytes = 16;
        }
        cp_async_16(stage + slab * kSlabKV + sw128_offset(row, chk), src, nbytes);
      }
      cp_async_commit();
      cp_async_wait_all();
      if (rank == 1) {
        // delta-rotation of k_r in shared memory (slab 4 holds k_r of the 64 rows), once
        // every producer warp's copies of the tile have landed
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_LANDED + s));
        if (!(ok = warp_wait(bar(BAR_LANDED + s), ph, abort_flag))) break;
        uint8_t* kr = smem + kOffKV + (uint32_t)s * kStage + 4 * kSlabKV;
        for (int it = tp; it < kBN * 4; it += 128) {
          const int row = it >> 2, pv = it & 3;
          const int d = map_delta[s * kBN + row];
          if (d != 0) {
            uint4* px = reinterpret_cast<uint4*>(kr + sw128_offset(row, pv));
            uint4* py = reinterpret_cast<uint4*>(kr + sw128_offset(row, pv + 4));
            uint4 x = *px, y = *py;
            float cc[8], ss[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) rope_cos_sin(d, phaseF[8 * pv + e], cc[e], ss[e]);
            rotate_pairs8(x, y, cc, ss);
            *px = x;
            *py = y;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_KV_FULL + s));
    }
    cp_async_wait_all();
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer (one thread) ===================================
    if (lane == 0 && ntiles > 0) {
      const uint32_t tO = tmem + kTmemO;
      bool ok = true;
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait(bar(BAR_P_FULL), jj & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t stage = sb + kOffKV + (uint32_t)(jj & 1) * kStage;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sdesc_sw128(sb + kOffP + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(stage + kk * 2048, kSlabKV, 1024);
          umma_bf16(tO, ad, bd, kIdescPV, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(BAR_KV_EMPTY + (jj & 1)));
        umma_commit(bar(BAR_PV_DONE));
        return true;
      };
      for (int j = 0; j < ntiles && ok; ++j) {
        const int s = j & 1;
        ok = mbar_wait(bar(BAR_KV_FULL + s), (j >> 1) & 1, abort_flag);
        if (ok && j >= 2) ok = mbar_wait(bar(BAR_S_EMPTY + s), ((j >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t stage = sb + kOffKV + (uint32_t)s * kStage;
        const uint32_t tS = tmem + kTmemS + 64u * (uint32_t)s;
        for (int slab = 0; slab < nslab; ++slab) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc_sw128(sb + kOffQ + slab * kSlabQ + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(stage + slab * kSlabKV + kk * 32, 16, 1024);
            umma_bf16(tS, ad, bd, kIdescS, (slab | kk) ? 1u : 0u);
          }
        }
        umma_commit(bar(BAR_S_FULL + s));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(ntiles - 1);
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, kDevErrTimeout);
      }
      umma_commit(bar(BAR_DRAIN));
      if (!mbar_wait(bar(BAR_DRAIN), 0, nullptr)) set_status(a.status, kDevErrTimeout);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue (thread = query row) ===================
    const int m = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + kTmemO + lane_base;
    const int pos_m = (m < rows_valid) ? ctx - a.n_q + q0 + m / a.H : pos_last;
    float m_run = -INFINITY, l_run = 0.f;
    const uint32_t rX = mapa_shared(sb + kOffX, peer);
    const uint32_t rXfull = mapa_shared(bar(BAR_X_FULL), peer);
    const uint32_t rXempty = mapa_shared(bar(BAR_X_EMPTY), peer);
    const float* X = reinterpret_cast<const float*>(smem + kOffX) + m * kBN;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int s = j & 1;
      const int T = (kb + j) * kBN;
      float sv[kBN];
      if (!(ok = warp_wait(bar(BAR_S_FULL + s), (j >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      {
        uint32_t r[32];
        tmem_ld32(tmem + kTmemS + 64u * (uint32_t)s + lane_base, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = __uint_as_float(r[i]);
        tmem_ld32(tmem + kTmemS + 64u * (uint32_t)s + 32u + lane_base, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_S_EMPTY + s));

      // exchange partial scores with the peer (each side owns half of the contraction)
      if (j >= 1 && !(ok = warp_wait_cluster(bar(BAR_X_EMPTY), (j - 1) & 1, abort_flag))) break;
      if (m == 0) mbar_arrive_expect_tx(bar(BAR_X_FULL), kBM * kBN * 4);
#pragma unroll
      for (int i = 0; i < kBN; i += 4)
        st_async_v4(rX + (uint32_t)(m * kBN + i) * 4u, sv[i], sv[i + 1], sv[i + 2], sv[i + 3],
                    rXfull);
      if (!(ok = warp_wait_cluster(bar(BAR_X_FULL), j & 1, abort_flag))) break;
#pragma unroll
      for (int i = 0; i < kBN; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(X + i);
        sv[i] += v.x;
        sv[i + 1] += v.y;
        sv[i + 2] += v.z;
        sv[i + 3] += v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_X_READ));
      if (m == 0) {  // all four warps read the peer's scores: it may send the next tile's
        if (mbar_wait(bar(BAR_X_READ), j & 1, abort_flag)) mbar_arrive_remote(rXempty);
        else *abort_flag = 1;
      }

      // online softmax in log2 units; causal mask t <= pos_m
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBN; ++i) {
        float x = sv[i] * a.scale_log2;
        if (T + i > pos_m) x = -INFINITY;
        sv[i] = x;
        mx = fmaxf(mx, x);
      }
      // The running max only moves when it grows by more than 2^8: P stays <= 256 and
      // O is rescaled rarely (the final 1/l uses the same max, so the result is exact).
      const bool want = mx > m_run + 8.f;
      float corr = 1.f;
      if (want) corr = fast_exp2(m_run - mx);
      bool pv_waited = false;
      if (j > 0 && __any_sync(FULL, want)) {
        if (!(ok = warp_wait(bar(BAR_PV_DONE), (j - 1) & 1, abort_flag))) break;
        pv_waited = true;
        tc_fence_after();
        for (int c = 0; c < 256; c += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
          tmem_st32(tO + c, r);
        }
        tmem_st_wait();
      }
      if (want) {
        l_run *= corr;
        m_run = mx;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float lsum = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int i = 0; i < kBN; i += 2) {
        const __nv_bfloat162 h =
            __floats2bfloat162_rn(fast_exp2(sv[i] - m_use), fast_exp2(sv[i + 1] - m_use));
        const float2 hf = __bfloat1622float2(h);  // sum what the tensor core will multiply
        lsum += hf.x + hf.y;
        pk[i >> 1] = *reinterpret_cast<const uint32_t*>(&h);
      }
      l_run += lsum;
      if (j > 0 && !pv_waited &&
          !(ok = warp_wait(bar(BAR_PV_DONE), (j - 1) & 1, abort_flag)))
        break;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(smem + kOffP + sw128_offset(m, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL));
    }
    if (ok && ntiles > 0) ok = warp_wait(bar(BAR_PV_DONE), (ntiles - 1) & 1, abort_flag);
    if (!ok) {
      *abort_flag = 1;
      set_status(a.status, kDevErrTimeout);
    }
    tc_fence_after();
    // ---- epilogue: O / l for this CTA's 256 columns ------------------------------------
    const bool have = ntiles > 0 && ok && l_run > 0.f;
    const float inv_l = have ? 1.f / l_run : 0.f;
    const float lse_v = have ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
    const bool write_row = m < rows_valid;
    const int qi = q0 + (write_row ? m / a.H : 0), hh = write_row ? m % a.H : 0;
    const int64_t orow = ((int64_t)b * a.n_q + qi) * a.H + hh;
    const int64_t prow = ((int64_t)b * a.n_qtiles * a.S + unit) * kBM + m;
    for (int c = 0; c < 256; c += 32) {
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
                                            col0 + c);
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
        float4* o = reinterpret_cast<float4*>(a.opart + prow * kDLat + col0 + c);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
    if (write_row && rank == 0) {
      if (a.S == 1) {
        if (a.lse != nullptr) a.lse[orow] = lse_v;
      } else {
        a.lsepart[prow] = lse_v;
      }
    }
  }

  // ---- teardown ---------------------------------------------------------------------
  __syncthreads();
  cluster_arrive();  // the peer no longer sends to this CTA's shared memory
  cluster_wait();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// LSE-weighted merge of the split-KV partials; one warp per (request, query, head) row.
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ AttnArgs a) {
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.B * a.n_q * a.H;
  if (gw >= total) return;
  const int h = (int)(gw % a.H);
  const int qi = (int)((gw / a.H) % a.n_q);
  const int b = (int)(gw / ((int64_t)a.H * a.n_q));
  const int qtile = qi / a.qpt;
  const int m = (qi - qtile * a.qpt) * a.H + h;
  const int64_t base = ((int64_t)b * a.n_qtiles * a.S + (int64_t)qtile * a.S) * kBM + m;
  float mx = -INFINITY;
  for (int s = 0; s < a.S; ++s) mx = fmaxf(mx, a.lsepart[base + (int64_t)s * kBM]);
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < a.S; ++s) {
      const float l = a.lsepart[base + (int64_t)s * kBM];
      if (l == -INFINITY) continue;
      const float w = __expf(l - mx);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(a.opart + (base + (int64_t)s * kBM) * kDLat);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[k * 32 + lane];
        acc[k].x += w * v.x;
        acc[k].y += w * v.y;
        acc[k].z += w * v.z;
        acc[k].w += w * v.w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int64_t orow = ((int64_t)b * a.n_q + qi) * a.H + h;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + orow * kDLat;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int col = (k * 32 + lane) * 4;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[k].x * inv, acc[k].y * inv);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[k].z * inv, acc[k].w * inv);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&h0);
    w.y = *reinterpret_cast<uint32_t*>(&h1);
    *reinterpret_cast<uint2*>(o + col) = w;
  }
  if (lane == 0 && a.lse != nullptr) a.lse[orow] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace

size_t attn_smem_bytes() { return kSmemBytes; }

cudaError_t launch_mla_attn(const AttnArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(mla_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * a.n_qtiles * a.S, a.B);
  mla_attn_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t stream) {
  const int64_t warps = (int64_t)a.B * a.n_q * a.H;
  const int64_t blocks = (warps * 32 + 255) / 256;
  combine_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irm
