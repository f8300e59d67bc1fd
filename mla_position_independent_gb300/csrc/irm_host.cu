// C ABI of the library: host-side validation of chunk tables, the copy of the validated
// tables into the caller's workspace, launch geometry, launches.  No allocation.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/irm.h"
#include "irm_internal.h"

namespace {

thread_local std::string g_last_error;

irm_status fail(irm_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

irm_status cuda_fail(cudaError_t e, const char* where) {
  return fail(IRM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// RoPE phase step of one pair: F = frac(theta / 2pi) * 2^64 (fp64 on the host), so that the
// device's (delta * F) mod 2^64 is the angle delta * theta reduced to one turn.
uint64_t phase_step(double theta) {
  const double two_pi = 6.283185307179586476925286766559;
  double turns = theta / two_pi;
  turns -= std::floor(turns);  // [0, 1]
  const double v = std::ldexp(turns, 64);
  return v >= 18446744073709551616.0 ? 0ull : (uint64_t)v;
}

// The default convention: NeoX half split, theta_j = 10000^(-2j/64).
const irm::RopePhaseHost& rope_phase() {
  static const irm::RopePhaseHost tab = [] {
    irm::RopePhaseHost t{};
    for (int j = 0; j < 32; ++j) t.F[j] = phase_step(std::pow(10000.0, -2.0 * j / 64.0));
    return t;
  }();
  return tab;
}

// Phase steps and pairing of a caller's RoPE variant (NULL: the default).
irm_status rope_select(const irm_rope* rope, uint64_t* F, int* interleaved) {
  if (rope == nullptr) {
    std::memcpy(F, rope_phase().F, 32 * sizeof(uint64_t));
    *interleaved = 0;
    return IRM_OK;
  }
  if (rope->pairing != IRM_ROPE_NEOX && rope->pairing != IRM_ROPE_INTERLEAVED)
    return fail(IRM_ERR_INVALID_ARG, "rope pairing %d is neither IRM_ROPE_NEOX nor IRM_ROPE_INTERLEAVED",
                rope->pairing);
  if (rope->reserved != 0) return fail(IRM_ERR_INVALID_ARG, "rope reserved field must be 0");
  for (int j = 0; j < 32; ++j) {
    if (!std::isfinite(rope->inv_freq[j])) return fail(IRM_ERR_INVALID_ARG, "rope inv_freq[%d] is not finite", j);
    F[j] = phase_step(rope->inv_freq[j]);
  }
  *interleaved = rope->pairing == IRM_ROPE_INTERLEAVED ? 1 : 0;
  return IRM_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

struct TableInfo {
  std::vector<int64_t> ctx;
  int64_t n_chunks = 0;
  int64_t max_ctx = 0;
  int64_t min_ctx = 0;
};

// Chunk-table rules [walkthrough §5 assembly loop, §7 carve-out]: per request the chunks
// tile [0, ctx) in target order with len > 0; source rows lie in the row store; a reused
// chunk never covers a position below 32; delta and positions fit in int32.
irm_status validate(const irm_chunk* chunks, const int32_t* indptr, int B, int64_t n_rows,
                    TableInfo* info) {
  if (B <= 0) return fail(IRM_ERR_INVALID_ARG, "B must be positive (got %d)", B);
  if (chunks == nullptr || indptr == nullptr)
    return fail(IRM_ERR_INVALID_ARG, "null chunk table pointer");
  if (indptr[0] != 0) return fail(IRM_ERR_CHUNK_TABLE, "indptr[0] must be 0");
  if (n_rows < 0 || n_rows >= (int64_t(1) << 31))
    return fail(IRM_ERR_INVALID_ARG, "n_rows %lld outside [0, 2^31)", (long long)n_rows);
  info->ctx.assign(B, 0);
  for (int b = 0; b < B; ++b) {
    const int32_t c0 = indptr[b], c1 = indptr[b + 1];
    if (c1 <= c0) return fail(IRM_ERR_CHUNK_TABLE, "request %d has no chunks", b);
    int64_t expect = 0;
    for (int32_t c = c0; c < c1; ++c) {
      const irm_chunk& ch = chunks[c];
      if (ch.len <= 0) return fail(IRM_ERR_CHUNK_TABLE, "chunk %d: len %d <= 0", c, ch.len);
      if ((int64_t)ch.p_tgt != expect)
        return fail(IRM_ERR_CHUNK_TABLE, "chunk %d: p_tgt %d, expected %lld (chunks must tile the context in order)",
                    c, ch.p_tgt, (long long)expect);
      if (ch.pool_offset < 0 || ch.pool_offset + ch.len > n_rows)
        return fail(IRM_ERR_CHUNK_TABLE, "chunk %d: rows [%lld, %lld) outside the row store of %lld rows", c,
                    (long long)ch.pool_offset, (long long)(ch.pool_offset + ch.len), (long long)n_rows);
      if (ch.reused > 1) return fail(IRM_ERR_CHUNK_TABLE, "chunk %d: reused must be 0 or 1", c);
      if (ch.reused && ch.p_tgt < IRM_CARVE_OUT)
        return fail(IRM_ERR_CARVEOUT, "chunk %d: reused chunk covers position %d < %d (first-chunk carve-out)",
                    c, ch.p_tgt, IRM_CARVE_OUT);
      if (ch.reused) {
        const int64_t d = (int64_t)ch.p_tgt - (int64_t)ch.p_src;
        if (d > INT32_MAX || d < INT32_MIN) return fail(IRM_ERR_CHUNK_TABLE, "chunk %d: delta overflows int32", c);
      }
      expect += ch.len;
      if (expect > INT32_MAX) return fail(IRM_ERR_CHUNK_TABLE, "request %d: context exceeds int32", b);
    }
    info->ctx[b] = expect;
  }
  info->n_chunks = indptr[B];
  info->max_ctx = info->min_ctx = info->ctx[0];
  for (int b = 1; b < B; ++b) {
    info->max_ctx = std::max(info->max_ctx, info->ctx[b]);
    info->min_ctx = std::min(info->min_ctx, info->ctx[b]);
  }
  return IRM_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Table area of a workspace, right after the status header: indptr [B+1] int32 (padded to
// 8 bytes), then the chunk records.  The kernels read the table from here only.
size_t indptr_area(int B) { return align_up((size_t)(B + 1) * sizeof(int32_t), 8); }
size_t table_bytes(int B, int64_t n_chunks) {
  return align_up(indptr_area(B) + (size_t)n_chunks * sizeof(irm_chunk), 256);
}

// Page-locked host memory: `locked`, and the address the device reads it through (nullptr
// when the memory is locked but not mapped for the device).
struct HostMem {
  bool locked;
  const void* dev;
};
HostMem host_mem(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return {false, nullptr};
  }
  if (at.type != cudaMemoryTypeHost) return {false, nullptr};
  return {true, at.devicePointer};
}

// A host array and where it goes inside the destination block.
struct HostPart {
  const void* src;
  size_t off, bytes;
};

// Copies host arrays into a device block on `stream`.  Page-locked arrays that the device can
// address are read by one small kernel straight from host memory (cheaper inside a step than
// copy-engine transfers, whose latency dominates for tables of a few hundred KB); other
// page-locked arrays are copied by one cudaMemcpyAsync each; pageable ones are packed into a
// host staging buffer and copied once, which the runtime has read when cudaMemcpyAsync returns
// (pageable copies cannot be captured into a graph).
irm_status stage_to_device(const HostPart* parts, int n, uint8_t* dst, cudaStream_t stream) {
  const void* dev_src[3] = {nullptr, nullptr, nullptr};
  bool locked = true, mapped = n <= 3;
  for (int i = 0; i < n && locked; ++i) {
    const HostMem m = host_mem(parts[i].src);
    locked = m.locked;
    if (i < 3) dev_src[i] = m.dev;
    mapped = mapped && m.dev != nullptr && parts[i].bytes % 4 == 0 && parts[i].off % 4 == 0 &&
             reinterpret_cast<uintptr_t>(m.dev) % 4 == 0;
  }
  cudaError_t e = cudaSuccess;
  if (locked && mapped) {
    irm::HostCopyArgs c{};
    c.dst = dst;
    c.n = n;
    for (int i = 0; i < n; ++i) {
      c.src[i] = dev_src[i];
      c.off[i] = parts[i].off;
      c.bytes[i] = parts[i].bytes;
    }
    e = irm::launch_host_copy(c, stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying the chunk table to the workspace");
    return IRM_OK;
  }
  if (locked) {
    for (int i = 0; i < n && e == cudaSuccess; ++i)
      e = cudaMemcpyAsync(dst + parts[i].off, parts[i].src, parts[i].bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "copying the chunk table to the workspace");
    return IRM_OK;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone)
    return fail(IRM_ERR_INVALID_ARG,
                "a chunk table in pageable host memory cannot be captured into a CUDA graph; "
                "pass page-locked host memory");
  thread_local std::vector<uint8_t> staging;
  const size_t end = parts[n - 1].off + parts[n - 1].bytes;
  staging.resize(end - parts[0].off);
  for (int i = 0; i < n; ++i) std::memcpy(staging.data() + (parts[i].off - parts[0].off), parts[i].src, parts[i].bytes);
  e = cudaMemcpyAsync(dst + parts[0].off, staging.data(), staging.size(), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copying the chunk table to the workspace");
  return IRM_OK;
}

// Copies a validated chunk table into the workspace's table area; returns the device
// addresses the kernels read.
irm_status stage_table(const irm_chunk* chunks_host, const int32_t* indptr_host, int B, int64_t n_chunks,
                       void* workspace, cudaStream_t stream, const irm_chunk** chunks_dev,
                       const int32_t** indptr_dev) {
  uint8_t* tab = static_cast<uint8_t*>(workspace) + IRM_WORKSPACE_HEADER;
  const HostPart parts[2] = {{indptr_host, 0, (size_t)(B + 1) * sizeof(int32_t)},
                             {chunks_host, indptr_area(B), (size_t)n_chunks * sizeof(irm_chunk)}};
  irm_status st = stage_to_device(parts, 2, tab, stream);
  if (st != IRM_OK) return st;
  *indptr_dev = reinterpret_cast<const int32_t*>(tab);
  *chunks_dev = reinterpret_cast<const irm_chunk*>(tab + indptr_area(B));
  return IRM_OK;
}

constexpr int kBM = 128;
constexpr int kBN = 64;

// Decode split-KV factor: the attention runs one 2-CTA cluster per (request, split); pick the
// split count that minimises waves x (tiles per split + the fixed cost of a split) plus the
// merge of the splits' partials.  In tile times (measured on the V3-shaped decode): a split's
// pipeline fill and epilogue cost ~12 tiles, and the merge reads each split's fp32 partial,
// ~3.6 tiles per split for 128 query rows (fewer rows, proportionally less).
int choose_splits(int B, int64_t max_ctx, int H, int sms, double* cost_out = nullptr) {
  const int pairs = std::max(1, sms / 2);
  const int64_t tiles = (max_ctx + kBN - 1) / kBN;
  const double split_cost = 12.0;
  const double merge_per_split = 3.6 * std::min(H, kBM) / kBM;
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= 64 && S <= tiles; ++S) {
    const int64_t units = (int64_t)B * S;
    const int64_t waves = (units + pairs - 1) / pairs;
    const double cost = (double)waves * ((double)((tiles + S - 1) / S) + split_cost) +
                        (S > 1 ? merge_per_split * S : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  if (cost_out != nullptr) *cost_out = best_cost;
  return best;
}

// Co-resident clusters of the attention kernel for Mv stored query rows, cached per device.
int attn_clusters(int Mv) {
  static std::mutex mu;
  static int cache[64][17];
  static bool have[64][17];
  int dev = 0;
  const int mi = std::min(16, std::max(0, Mv / 8));
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev][mi]) {
    cache[dev][mi] = irm::attn_max_active_clusters(Mv);
    have[dev][mi] = true;
  }
  return cache[dev][mi];
}

// Long-first split of U query tiles of `tiles` KV tiles each over P co-resident clusters, when
// U < P: split 0 (the leading L tiles of every query tile) takes U clusters at once, the P - U
// clusters left run the U short splits one after another (R = ceil(U / (P - U)) each).  L
// balances the two, L + 12 = R (tiles - L + 12) (12: a split's fill and epilogue, in tile
// times as in choose_splits), plus the merge of two partials.  Returns the cost (1e30 when it
// does not apply) and the cut L / tiles in 1/4096.
double choose_long_first(int U, int64_t tiles, int H, int P, int* cut_q12) {
  *cut_q12 = 0;
  if (P <= 0 || U >= P || tiles < 2) return 1e30;
  const int64_t R = (U + (P - U) - 1) / (P - U);
  const double L = std::min((double)tiles - 1.0, std::max(1.0, ((double)R * ((double)tiles + 12.0) - 12.0) / (1.0 + R)));
  *cut_q12 = (int)std::lround(L / (double)tiles * 4096.0);
  const double merge = 2.0 * 3.6 * std::min(H, kBM) / kBM;
  return std::max(L + 12.0, (double)R * ((double)tiles - L + 12.0)) + merge;
}

// Split-KV scratch: fp32 partial O, per-rank partial LSE, finished-split counters.
size_t partial_o_bytes(int B, int units) {
  return align_up((size_t)B * units * kBM * IRM_D_LAT * sizeof(float), 256);
}
size_t partial_lse_bytes(int B, int units) {
  return align_up((size_t)2 * B * units * kBM * sizeof(float), 256);
}
size_t counter_bytes(int B, int n_qtiles) { return align_up((size_t)B * n_qtiles * 2 * sizeof(int), 256); }
size_t partial_bytes(int B, int n_qtiles, int S) {
  return partial_o_bytes(B, n_qtiles * S) + partial_lse_bytes(B, n_qtiles * S) + counter_bytes(B, n_qtiles);
}

struct AttnPlan {
  int qpt, n_qtiles, S;
  bool few_heads;  // decode with H in {16, 32}: the split-KV decode kernel
  int C, G;        // its cluster size and clusters per request
  int long_first, cut_q12;  // attention kernel: long-first split (S == 2) and its cut
  size_t scratch_off;  // workspace offset of the split-KV scratch (after header and table)
  size_t ws_bytes;
};

// Largest number of co-resident clusters of the decode kernel per cluster size, cached per
// device (the query needs the device; it is made once).
int decode_clusters(int H, int C) {
  static std::mutex mu;
  static int cache[64][2][5];
  static bool have[64][2][5];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return irm::decode_max_active_clusters(H, C);
  const int hi = H == 16 ? 0 : 1, ci = C == 1 ? 0 : C == 2 ? 1 : C == 4 ? 2 : C == 8 ? 3 : 4;
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev][hi][ci]) {
    cache[dev][hi][ci] = irm::decode_max_active_clusters(H, C);
    have[dev][hi][ci] = true;
  }
  return cache[dev][hi][ci];
}

// Split of a decode over the decode kernel's clusters: C CTAs per cluster (a power of two
// up to 16), G clusters per request.  Minimises, in tile times, waves x (tiles per split +
// pipeline fill) plus the merge of G cluster partials (a fixed cost and the slice each
// last cluster CTA reads: G x H x 2 KiB / C).
void choose_decode_split(int B, int64_t max_ctx, int H, int* C_out, int* G_out) {
  const int64_t tiles = std::max<int64_t>(1, (max_ctx + kBN - 1) / kBN);
  int bestC = 1, bestG = 1;
  double best_cost = 1e30;
  for (int C = 1; C <= irm::kMaxDecodeCluster; C *= 2) {
    if (C > 1 && C > tiles) break;
    const int n = decode_clusters(H, C);
    if (n <= 0) continue;
    for (int G = 1; G <= 64; ++G) {
      const int64_t S = (int64_t)C * G;
      if (S > tiles && G > 1) break;
      const int64_t waves = ((int64_t)B * G + n - 1) / n;
      const double cost = (double)waves * ((double)((tiles + S - 1) / S) + 2.0) +
                          (G > 1 ? 0.5 + 0.01 * G * H / C : 0.0);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        bestC = C;
        bestG = G;
      }
    }
  }
  *C_out = bestC;
  *G_out = bestG;
}

size_t decode_gpart_bytes(int B, int G, int H) { return ((size_t)B * G * H * IRM_D_LAT * 4 + 255) / 256 * 256; }
size_t decode_glse_bytes(int B, int G, int H) { return ((size_t)B * G * H * 4 + 255) / 256 * 256; }
size_t decode_counter_bytes(int B, int C) { return ((size_t)B * C * 4 + 255) / 256 * 256; }

// ws_cap: the most scratch the caller can offer for a long-first split (the usual split is
// planned instead when that one needs more).
irm_status plan_attn(const TableInfo& info, int B, int n_q, int H, bool decode, AttnPlan* p,
                     size_t ws_cap = SIZE_MAX) {
  if (H < 1 || H > IRM_MAX_HEADS) return fail(IRM_ERR_UNSUPPORTED, "H=%d outside [1, %d]", H, IRM_MAX_HEADS);
  if (n_q < 1) return fail(IRM_ERR_INVALID_ARG, "n_q must be >= 1");
  if (n_q > info.min_ctx)
    return fail(IRM_ERR_INVALID_ARG, "n_q=%d exceeds the shortest context (%lld)", n_q, (long long)info.min_ctx);
  p->qpt = kBM / H;
  p->n_qtiles = (n_q + p->qpt - 1) / p->qpt;
  if (p->n_qtiles > 32767) return fail(IRM_ERR_UNSUPPORTED, "too many query tiles (%d)", p->n_qtiles);
  if (B > 65535) return fail(IRM_ERR_UNSUPPORTED, "B=%d exceeds 65535", B);
  p->few_heads = decode && n_q == 1 && irm::decode_supported(H);
  p->scratch_off = IRM_WORKSPACE_HEADER + table_bytes(B, info.n_chunks);
  if (p->few_heads) {
    p->S = 1;
    choose_decode_split(B, info.max_ctx, H, &p->C, &p->G);
    p->ws_bytes = p->scratch_off;
    if (p->G > 1)
      p->ws_bytes += decode_gpart_bytes(B, p->G, H) + decode_glse_bytes(B, p->G, H) + decode_counter_bytes(B, p->C);
    return IRM_OK;
  }
  double split_cost = 0.0;
  p->S = decode ? choose_splits(B, info.max_ctx, H, num_sms(), &split_cost) : 1;
  p->long_first = 0;
  p->cut_q12 = 0;
  p->ws_bytes = p->scratch_off + (p->S > 1 ? partial_bytes(B, p->n_qtiles, p->S) : 0);
  if (decode && p->n_qtiles == 1) {
    const int Mv = std::min(kBM, (std::min(p->qpt, n_q) * H + 7) / 8 * 8);
    int cut = 0;
    const double lf_cost = choose_long_first(B * p->n_qtiles, (info.max_ctx + kBN - 1) / kBN, H,
                                             attn_clusters(Mv), &cut);
    const size_t lf_ws = p->scratch_off + partial_bytes(B, p->n_qtiles, 2);
    if (lf_cost < split_cost - 1e-9 && lf_ws <= ws_cap) {
      p->long_first = 1;
      p->cut_q12 = cut;
      p->S = 2;
      p->ws_bytes = lf_ws;
    }
  }
  return IRM_OK;
}

irm_status run_attn(const void* q_lat, const void* q_rope, int B, int n_q, int H,
                    const irm_chunk* chunks_host, const int32_t* indptr_host, const void* kv_rows,
                    int64_t n_rows, float softmax_scale, void* out, float* lse, const irm_rope* rope,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream, bool decode,
                    size_t ws_cap = SIZE_MAX) {
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, n_rows, &info);
  if (st != IRM_OK) return st;
  uint64_t phaseF[32];
  int interleaved = 0;
  if ((st = rope_select(rope, phaseF, &interleaved)) != IRM_OK) return st;
  AttnPlan pl{};
  if ((st = plan_attn(info, B, n_q, H, decode, &pl, ws_cap)) != IRM_OK) return st;
  if (!q_lat || !q_rope || !kv_rows || !out) return fail(IRM_ERR_INVALID_ARG, "null device pointer");
  if (!aligned(q_lat, 16) || !aligned(q_rope, 16) || !aligned(kv_rows, 16) || !aligned(out, 16))
    return fail(IRM_ERR_INVALID_ARG, "q_lat, q_rope, kv_rows and out must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(IRM_ERR_INVALID_ARG, "misaligned lse pointer");
  if (!std::isfinite(softmax_scale)) return fail(IRM_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.ws_bytes)
    return fail(IRM_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes (got %zu)",
                pl.ws_bytes, workspace_bytes);
  // The validated table reaches the kernel in its parameter block when it is small (the
  // launch copies it), else through the workspace (one host-to-device copy before the launch).
  const bool inline_tab = info.n_chunks <= irm::kInlineChunks && B + 1 <= irm::kInlineIndptr;
  const irm_chunk* chunks_dev = nullptr;
  const int32_t* indptr_dev = nullptr;
  if (!inline_tab &&
      (st = stage_table(chunks_host, indptr_host, B, info.n_chunks, workspace, stream, &chunks_dev, &indptr_dev)) !=
          IRM_OK)
    return st;
  auto fill_inline = [&](int* flag, irm::InlineTable* tab) {
    *flag = inline_tab ? 1 : 0;
    if (inline_tab) {
      std::memcpy(tab->chunks, chunks_host, (size_t)info.n_chunks * sizeof(irm_chunk));
      std::memcpy(tab->indptr, indptr_host, (size_t)(B + 1) * sizeof(int32_t));
    }
  };
  if (pl.few_heads) {
    // ~30 KB with the inline table: kept off the stack; every field before the table is reset
    // (the table is written up to its length, and the kernel reads no further)
    thread_local irm::DecodeArgs d;
    std::memset(static_cast<void*>(&d), 0, offsetof(irm::DecodeArgs, tab));
    d.q_lat = q_lat;
    d.q_rope = q_rope;
    d.kv = kv_rows;
    d.chunks = chunks_dev;
    d.indptr = indptr_dev;
    fill_inline(&d.inline_table, &d.tab);
    d.n_rows = n_rows;
    d.n_chunks = info.n_chunks;
    d.B = B;
    d.H = H;
    d.C = pl.C;
    d.G = pl.G;
    if (pl.G > 1) {
      uint8_t* ws = static_cast<uint8_t*>(workspace) + pl.scratch_off;
      d.gpart = reinterpret_cast<float*>(ws);
      d.glse = reinterpret_cast<float*>(ws + decode_gpart_bytes(B, pl.G, H));
      d.counters = reinterpret_cast<int*>(ws + decode_gpart_bytes(B, pl.G, H) + decode_glse_bytes(B, pl.G, H));
    }
    d.scale_log2 = softmax_scale * 1.4426950408889634f;
    d.out = out;
    d.lse = lse;
    d.status = static_cast<int*>(workspace);
    std::memcpy(d.phase.F, phaseF, sizeof d.phase.F);
    d.interleaved = interleaved;
    const int splits = pl.C * pl.G;
    if ((int64_t)B * splits <= irm::kDecodeHints) {
      // each split's start, from the validated host table (the kernels use the same split
      // boundaries: split sp of a request starts at tile sp * tiles / splits)
      d.n_hints = B * splits;
      for (int b = 0; b < B; ++b) {
        const int cb = indptr_host[b], ce = indptr_host[b + 1];
        const int64_t ctx = info.ctx[b];
        const int64_t tiles = (ctx + kBN - 1) / kBN;
        int c = cb;
        for (int sp = 0; sp < splits; ++sp) {
          const int64_t t0 = (int64_t)sp * tiles / splits * kBN;
          while (c + 1 < ce && chunks_host[c + 1].p_tgt <= t0) ++c;
          d.hint[b * splits + sp] = irm::DecodeHint{cb, ce, (int32_t)ctx, c};
        }
      }
    }
    cudaError_t e = irm::launch_mla_decode(d, stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla decode launch");
    return IRM_OK;
  }
  thread_local irm::AttnArgs a;  // ~25 KB with the inline table (see above)
  std::memset(static_cast<void*>(&a), 0, offsetof(irm::AttnArgs, tab));
  a.q_lat = q_lat;
  a.q_rope = q_rope;
  a.kv = kv_rows;
  a.chunks = chunks_dev;
  a.indptr = indptr_dev;
  fill_inline(&a.inline_table, &a.tab);
  a.n_rows = n_rows;
  a.n_chunks = info.n_chunks;
  a.B = B;
  a.n_q = n_q;
  a.H = H;
  a.qpt = pl.qpt;
  a.n_qtiles = pl.n_qtiles;
  a.S = pl.S;
  a.long_first = pl.long_first;
  a.split_num = pl.long_first ? pl.cut_q12 : 1;
  a.split_den = pl.long_first ? 4096 : pl.S;
  // query rows a tile really holds (decode: H); Q, P and the score exchange store only these
  a.Mv = std::min(kBM, (std::min(pl.qpt, n_q) * H + 7) / 8 * 8);
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = out;
  a.lse = lse;
  a.status = static_cast<int*>(workspace);
  uint8_t* ws = static_cast<uint8_t*>(workspace) + pl.scratch_off;
  if (pl.S > 1) {
    const int units = pl.n_qtiles * pl.S;
    a.opart = reinterpret_cast<float*>(ws);
    a.lsepart = reinterpret_cast<float*>(ws + partial_o_bytes(B, units));
    a.counters = reinterpret_cast<int*>(ws + partial_o_bytes(B, units) + partial_lse_bytes(B, units));
  }
  std::memcpy(a.phase.F, phaseF, sizeof a.phase.F);
  a.interleaved = interleaved;
  cudaError_t e = irm::launch_mla_attn(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "mla attention launch");
  return IRM_OK;
}

// Scratch for irm_mla_attn_decode_noalloc: a fixed device array in this library, so that
// callers that cannot allocate device memory still get split-KV decode.  It exists once
// per device that loads the library and lives until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[128] = {};

// Device address of the scratch array for the current device.  In host code the array's
// name is only a host-side stand-in, so the address comes from cudaGetSymbolAddress, once
// per device, with that device current.
irm_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 128) return fail(IRM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return IRM_OK;
}

// Workspace of irm_cdc_chunk: status header, the copied stream offsets [S + 1], slot and
// segment bases [S + 1] each (used when the batch is too large for the kernel parameters),
// the candidate bitmask, then per speculative segment its chunk ends [spec_cap], count and
// exit, and its chunks' fingerprints [spec_cap].
struct CdcLayout {
  size_t offsets, base, seg_base, words, spec_ends, spec_count, spec_exit, spec_hash, total;
  int64_t n_segs, spec_cap;
};
irm_status cdc_check(const int64_t* offsets_host, int n_streams, const irm_cdc_params* params,
                     irm_cdc_params* p, int64_t* slots, int64_t* max_len, size_t* bytes,
                     CdcLayout* lay = nullptr) {
  if (n_streams <= 0 || offsets_host == nullptr) return fail(IRM_ERR_INVALID_ARG, "need n_streams > 0 and offsets");
  *p = params ? *params : irm_cdc_params{32, 512, 7, IRM_CDC_THRESHOLD, 0, 0};
  if (p->min_len < 1 || p->max_len < p->min_len || p->max_len > 65536)
    return fail(IRM_ERR_INVALID_ARG, "need 1 <= min_len <= max_len <= 65536 (got %d, %d)", p->min_len, p->max_len);
  if (p->bits < 1 || p->bits > 63) return fail(IRM_ERR_INVALID_ARG, "bits must lie in [1, 63]");
  if (p->mode != IRM_CDC_THRESHOLD && p->mode != IRM_CDC_LOW_BITS)
    return fail(IRM_ERR_INVALID_ARG, "mode must be IRM_CDC_THRESHOLD or IRM_CDC_LOW_BITS");
  if (offsets_host[0] != 0) return fail(IRM_ERR_INVALID_ARG, "offsets[0] must be 0");
  int64_t sl = 0, mx = 0;
  for (int s = 0; s < n_streams; ++s) {
    const int64_t len = offsets_host[s + 1] - offsets_host[s];
    if (len < 0 || len > INT32_MAX) return fail(IRM_ERR_INVALID_ARG, "stream %d has length %lld", s, (long long)len);
    sl += len / p->min_len + 1;
    mx = std::max(mx, len);
  }
  *slots = sl;
  *max_len = mx;
  CdcLayout L{};
  const int64_t seg = irm::cdc_segment_len();
  for (int s = 0; s < n_streams; ++s) L.n_segs += (offsets_host[s + 1] - offsets_host[s] + seg - 1) / seg;
  L.spec_cap = (seg + p->max_len) / p->min_len + 2;  // chunk ends in [seg start, seg end + max_len)
  const size_t words = (size_t)(offsets_host[n_streams] >> 5) + (size_t)n_streams + 1;
  const size_t bases = align_up((size_t)(n_streams + 1) * sizeof(int64_t), 256);
  L.offsets = IRM_WORKSPACE_HEADER;
  L.base = L.offsets + bases;
  L.seg_base = L.base + bases;
  L.words = L.seg_base + bases;
  L.spec_ends = L.words + align_up(words * sizeof(uint32_t), 256);
  L.spec_count = L.spec_ends + align_up((size_t)L.n_segs * (size_t)L.spec_cap * sizeof(int32_t), 256);
  L.spec_exit = L.spec_count + align_up((size_t)(L.n_segs + 1) * sizeof(int32_t), 256);
  L.spec_hash = L.spec_exit + align_up((size_t)(L.n_segs + 1) * sizeof(int32_t), 256);
  L.total = L.spec_hash + align_up((size_t)L.n_segs * (size_t)L.spec_cap * sizeof(uint64_t), 256);
  *bytes = L.total;
  if (lay) *lay = L;
  return IRM_OK;
}

}  // namespace

namespace irm {
// Sets the calling thread's last-error text (used by the registry's translation unit).
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace irm

extern "C" {

const char* irm_status_string(int status) {
  switch (status) {
    case IRM_OK: return "ok";
    case IRM_ERR_INVALID_ARG: return "invalid argument";
    case IRM_ERR_CHUNK_TABLE: return "invalid chunk table";
    case IRM_ERR_CARVEOUT: return "reused chunk inside the first-chunk carve-out";
    case IRM_ERR_UNSUPPORTED: return "unsupported shape";
    case IRM_ERR_CUDA: return "CUDA error";
    case IRM_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case IRM_ERR_DEVICE_BOUNDS: return "device saw a source row or page outside its buffer";
    case IRM_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

const char* irm_last_error(void) { return g_last_error.c_str(); }

const char* irm_version(void) { return "irm 0.1 sm_103a"; }

irm_status irm_validate_chunks(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                               int64_t n_rows, int64_t* ctx_out) {
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, n_rows, &info);
  if (st == IRM_OK && ctx_out != nullptr)
    for (int b = 0; b < B; ++b) ctx_out[b] = info.ctx[b];
  return st;
}

irm_status irm_device_status(void* workspace, cudaStream_t stream) {
  if (workspace == nullptr) return fail(IRM_ERR_INVALID_ARG, "null workspace");
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  if (word != 0) {
    e = cudaMemsetAsync(workspace, 0, sizeof word, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  }
  if (word & 1) return fail(IRM_ERR_DEVICE_TIMEOUT, "a device pipeline wait exceeded its limit");
  if (word & 2) return fail(IRM_ERR_DEVICE_BOUNDS, "a kernel met a source row or page outside its buffer");
  return IRM_OK;
}

irm_status irm_assemble_kv_workspace_size(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                                          size_t* bytes) {
  if (bytes == nullptr) return fail(IRM_ERR_INVALID_ARG, "bytes is null");
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, INT32_MAX, &info);
  if (st != IRM_OK) return st;
  // header, table, row starts [B+1] int64
  *bytes = IRM_WORKSPACE_HEADER + table_bytes(B, info.n_chunks) + align_up((size_t)(B + 1) * sizeof(int64_t), 256);
  return IRM_OK;
}

irm_status irm_assemble_kv(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                           const void* kv_rows, int64_t n_rows, void* paged_out, int64_t n_pages,
                           const int32_t* page_table, int max_pages, int32_t* out_src_row,
                           int32_t* out_delta, int32_t* out_pos_src, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  return irm_assemble_kv_rope(chunks_host, indptr_host, B, kv_rows, n_rows,
                              paged_out, n_pages, page_table, max_pages, out_src_row, out_delta,
                              out_pos_src, nullptr, workspace, workspace_bytes, stream);
}

irm_status irm_assemble_kv_rope(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                                const void* kv_rows, int64_t n_rows, void* paged_out,
                                int64_t n_pages, const int32_t* page_table, int max_pages,
                                int32_t* out_src_row, int32_t* out_delta, int32_t* out_pos_src,
                                const irm_rope* rope, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, n_rows, &info);
  if (st != IRM_OK) return st;
  uint64_t phaseF[32];
  int interleaved = 0;
  if ((st = rope_select(rope, phaseF, &interleaved)) != IRM_OK) return st;
  const bool plan_out = out_src_row || out_delta || out_pos_src;
  if (plan_out && !(out_src_row && out_delta && out_pos_src))
    return fail(IRM_ERR_INVALID_ARG, "out_src_row, out_delta and out_pos_src go together");
  if (paged_out) {
    if (!kv_rows || !page_table) return fail(IRM_ERR_INVALID_ARG, "paged output needs kv_rows and page_table");
    if (!aligned(kv_rows, 16) || !aligned(paged_out, 16))
      return fail(IRM_ERR_INVALID_ARG, "kv_rows and paged_out must be 16-byte aligned");
    if (n_pages <= 0 || max_pages <= 0) return fail(IRM_ERR_INVALID_ARG, "n_pages and max_pages must be positive");
    if ((info.max_ctx + IRM_PAGE_ROWS - 1) / IRM_PAGE_ROWS > max_pages)
      return fail(IRM_ERR_INVALID_ARG, "a context of %lld rows needs more than max_pages=%d pages",
                  (long long)info.max_ctx, max_pages);
  }
  const size_t tab_bytes = table_bytes(B, info.n_chunks);
  const size_t need = IRM_WORKSPACE_HEADER + tab_bytes + align_up((size_t)(B + 1) * sizeof(int64_t), 256);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(IRM_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
  if (!paged_out && !plan_out) return IRM_OK;
  const irm_chunk* chunks_dev = nullptr;
  const int32_t* indptr_dev = nullptr;
  if ((st = stage_table(chunks_host, indptr_host, B, info.n_chunks, workspace, stream, &chunks_dev, &indptr_dev)) !=
      IRM_OK)
    return st;
  irm::GatherArgs g{};
  g.chunks = chunks_dev;
  g.indptr = indptr_dev;
  g.B = B;
  g.n_chunks = info.n_chunks;
  g.kv = kv_rows;
  g.n_rows = n_rows;
  g.paged_out = paged_out;
  g.n_pages = n_pages;
  g.page_table = page_table;
  g.max_pages = max_pages;
  g.status = static_cast<int*>(workspace);
  g.out_src = out_src_row;
  g.out_delta = out_delta;
  g.out_pos_src = out_pos_src;
  std::memcpy(g.phase.F, phaseF, sizeof g.phase.F);
  g.interleaved = interleaved;
  // rows of the requests before each one: in the launch parameters for up to 256 requests,
  // else computed on the device from the copied table
  g.total_rows = 0;
  for (int b = 0; b < B; ++b) g.total_rows += info.ctx[b];
  g.inline_rows = B + 1 <= irm::kInlineIndptr ? 1 : 0;
  if (g.inline_rows) {
    int64_t t = 0;
    for (int b = 0; b < B; ++b) {
      g.rows[b] = t;
      t += info.ctx[b];
    }
    g.rows[B] = t;
  } else {
    int64_t* row_start =
        reinterpret_cast<int64_t*>(static_cast<uint8_t*>(workspace) + IRM_WORKSPACE_HEADER + tab_bytes);
    g.row_start = row_start;
    cudaError_t e = irm::launch_row_start(chunks_dev, indptr_dev, B, row_start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "row-start launch");
  }
  cudaError_t e = irm::launch_rotate_gather(g, num_sms(), stream);
  if (e != cudaSuccess) return cuda_fail(e, "rotate+gather launch");
  return IRM_OK;
}

irm_status irm_mla_attn_decode_workspace_size(const irm_chunk* chunks_host, const int32_t* indptr_host,
                                              int B, int H, size_t* bytes) {
  if (bytes == nullptr) return fail(IRM_ERR_INVALID_ARG, "bytes is null");
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, INT32_MAX, &info);
  if (st != IRM_OK) return st;
  AttnPlan pl{};
  if ((st = plan_attn(info, B, 1, H, true, &pl)) != IRM_OK) return st;
  *bytes = pl.ws_bytes;
  return IRM_OK;
}

irm_status irm_mla_attn_decode(const void* q_lat, const void* q_rope, int B, int H,
                               const irm_chunk* chunks_host, const int32_t* indptr_host,
                               const void* kv_rows, int64_t n_rows, float softmax_scale, void* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  return run_attn(q_lat, q_rope, B, 1, H, chunks_host, indptr_host, kv_rows,
                  n_rows, softmax_scale, out, lse, nullptr, workspace, workspace_bytes, stream, true);
}

irm_status irm_mla_attn_decode_rope(const void* q_lat, const void* q_rope, int B, int H,
                                    const irm_chunk* chunks_host, const int32_t* indptr_host,
                                    const void* kv_rows, int64_t n_rows, float softmax_scale,
                                    void* out, float* lse, const irm_rope* rope, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  return run_attn(q_lat, q_rope, B, 1, H, chunks_host, indptr_host, kv_rows,
                  n_rows, softmax_scale, out, lse, rope, workspace, workspace_bytes, stream, true);
}

irm_status irm_mla_attn_decode_noalloc(const void* q_lat, const void* q_rope, int B, int H,
                                       const irm_chunk* chunks_host, const int32_t* indptr_host,
                                       const void* kv_rows, int64_t n_rows, float softmax_scale,
                                       void* out, float* lse, cudaStream_t stream) {
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, n_rows, &info);
  if (st != IRM_OK) return st;
  AttnPlan pl{};
  if ((st = plan_attn(info, B, 1, H, true, &pl, kNoAllocScratchBytes)) != IRM_OK) return st;
  if (pl.ws_bytes > kNoAllocScratchBytes)
    return fail(IRM_ERR_WORKSPACE,
                "this decode needs %zu bytes of table and scratch, more than the %zu bytes the no-allocation "
                "entry point holds; use irm_mla_attn_decode with a workspace",
                pl.ws_bytes, kNoAllocScratchBytes);
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != IRM_OK) return st;
  // The array keeps the last call's contents: clear the split-KV completion counters, which
  // must start at zero.  The status word is left alone, so that a device error of any call
  // stays readable through irm_decode_noalloc_status().
  cudaError_t e = cudaSuccess;
  if (pl.few_heads && pl.G > 1) {
    const size_t off = pl.scratch_off + decode_gpart_bytes(B, pl.G, H) + decode_glse_bytes(B, pl.G, H);
    e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + off, 0, decode_counter_bytes(B, pl.C), stream);
  }
  if (e == cudaSuccess && !pl.few_heads && pl.S > 1) {
    const int units = pl.n_qtiles * pl.S;
    const size_t off = pl.scratch_off + partial_o_bytes(B, units) + partial_lse_bytes(B, units);
    e = cudaMemsetAsync(static_cast<uint8_t*>(ws) + off, 0, counter_bytes(B, pl.n_qtiles), stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "clearing the no-allocation scratch");
  return run_attn(q_lat, q_rope, B, 1, H, chunks_host, indptr_host, kv_rows,
                  n_rows, softmax_scale, out, lse, nullptr, ws, kNoAllocScratchBytes, stream, true,
                  kNoAllocScratchBytes);
}

irm_status irm_decode_noalloc_status(cudaStream_t stream) {
  void* ws = nullptr;
  irm_status st = noalloc_scratch(&ws);
  if (st != IRM_OK) return st;
  return irm_device_status(ws, stream);
}

irm_status irm_cdc_sizes(const int64_t* offsets_host, int n_streams, const irm_cdc_params* params,
                         size_t* bytes, int64_t* slots) {
  if (bytes == nullptr || slots == nullptr) return fail(IRM_ERR_INVALID_ARG, "null output");
  irm_cdc_params p{};
  int64_t mx;
  return cdc_check(offsets_host, n_streams, params, &p, slots, &mx, bytes);
}

irm_status irm_cdc_chunk(const int32_t* tokens, const int64_t* offsets_host, int n_streams,
                         const uint64_t* gear, int32_t vocab,
                         const irm_cdc_params* params, int32_t* n_chunks, int32_t* chunk_start,
                         int32_t* chunk_len, uint64_t* chunk_hash, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
  irm_cdc_params p{};
  int64_t slots = 0, max_len = 0;
  size_t need = 0;
  CdcLayout lay{};
  irm_status st = cdc_check(offsets_host, n_streams, params, &p, &slots, &max_len, &need, &lay);
  if (st != IRM_OK) return st;
  if (vocab <= 0) return fail(IRM_ERR_INVALID_ARG, "vocab must be positive");
  if (!n_chunks || !chunk_start || !chunk_len ||
      (!tokens && offsets_host[n_streams] > 0))
    return fail(IRM_ERR_INVALID_ARG, "null device pointer");
  if (!aligned(tokens, 4) || !aligned(gear, 8) || !aligned(chunk_hash, 8))
    return fail(IRM_ERR_INVALID_ARG, "misaligned device pointer");
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(IRM_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // ~25 KB with the inline stream table: kept off the stack; the fields before it are reset
  thread_local irm::CdcArgs a;
  std::memset(static_cast<void*>(&a), 0, offsetof(irm::CdcArgs, ib));
  if (n_streams <= irm::kCdcInline) {
    // offsets and per-stream bases (output slots, speculative segments) travel in the launch
    a.inline_streams = 1;
    int64_t sb = 0, gb = 0;
    const int64_t seg = irm::cdc_segment_len();
    for (int s = 0; s <= n_streams; ++s) {
      a.ib.offsets[s] = offsets_host[s];
      a.ib.base[s] = sb;
      a.ib.seg_base[s] = gb;
      if (s < n_streams) {
        const int64_t len = offsets_host[s + 1] - offsets_host[s];
        sb += len / p.min_len + 1;
        gb += (len + seg - 1) / seg;
      }
    }
  } else {
    const HostPart part = {offsets_host, 0, (size_t)(n_streams + 1) * sizeof(int64_t)};
    if ((st = stage_to_device(&part, 1, ws + lay.offsets, stream)) != IRM_OK) return st;
  }
  a.tokens = tokens;
  a.offsets = reinterpret_cast<const int64_t*>(ws + lay.offsets);
  a.S = n_streams;
  a.gear = gear;
  a.gear_seed = p.gear_seed;
  a.vocab = vocab;
  a.min_len = p.min_len;
  a.max_len = p.max_len;
  a.bits = p.bits;
  a.mode = p.mode;
  a.seed = p.seed;
  a.status = reinterpret_cast<int*>(ws);
  a.base = reinterpret_cast<int64_t*>(ws + lay.base);
  a.seg_base = reinterpret_cast<int64_t*>(ws + lay.seg_base);
  a.words = reinterpret_cast<uint32_t*>(ws + lay.words);
  a.spec_ends = reinterpret_cast<int32_t*>(ws + lay.spec_ends);
  a.spec_count = reinterpret_cast<int32_t*>(ws + lay.spec_count);
  a.spec_exit = reinterpret_cast<int32_t*>(ws + lay.spec_exit);
  a.spec_hash = reinterpret_cast<uint64_t*>(ws + lay.spec_hash);
  a.spec_cap = lay.spec_cap;
  a.n_segs = lay.n_segs;
  a.n_chunks = n_chunks;
  a.chunk_start = chunk_start;
  a.chunk_len = chunk_len;
  a.chunk_hash = chunk_hash;
  cudaError_t e = irm::launch_cdc(a, max_len, slots, lay.n_segs, stream);
  if (e != cudaSuccess) return cuda_fail(e, "content-defined chunking launch");
  return IRM_OK;
}

irm_status irm_mla_attn_prefill_workspace_size(const irm_chunk* chunks_host, const int32_t* indptr_host,
                                               int B, int n_q, int H, size_t* bytes) {
  if (bytes == nullptr) return fail(IRM_ERR_INVALID_ARG, "bytes is null");
  TableInfo info;
  irm_status st = validate(chunks_host, indptr_host, B, INT32_MAX, &info);
  if (st != IRM_OK) return st;
  AttnPlan pl{};
  if ((st = plan_attn(info, B, n_q, H, false, &pl)) != IRM_OK) return st;
  *bytes = pl.ws_bytes;
  return IRM_OK;
}

irm_status irm_mla_attn_prefill(const void* q_lat, const void* q_rope, int B, int n_q, int H,
                                const irm_chunk* chunks_host, const int32_t* indptr_host,
                                const void* kv_rows, int64_t n_rows, float softmax_scale, void* out,
                                float* lse, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  return run_attn(q_lat, q_rope, B, n_q, H, chunks_host, indptr_host, kv_rows,
                  n_rows, softmax_scale, out, lse, nullptr, workspace, workspace_bytes, stream, false);
}

irm_status irm_mla_attn_prefill_rope(const void* q_lat, const void* q_rope, int B, int n_q, int H,
                                     const irm_chunk* chunks_host, const int32_t* indptr_host,
                                     const void* kv_rows, int64_t n_rows, float softmax_scale,
                                     void* out, float* lse, const irm_rope* rope, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  return run_attn(q_lat, q_rope, B, n_q, H, chunks_host, indptr_host, kv_rows,
                  n_rows, softmax_scale, out, lse, rope, workspace, workspace_bytes, stream, false);
}

}  // extern "C"
