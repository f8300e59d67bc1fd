// Internal launch interfaces between the C ABI (irm_host.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/irm.h"

namespace irm {

struct RopePhaseHost {
  uint64_t F[32];
};

struct GatherArgs {
  const irm_chunk* chunks;
  const int32_t* indptr;
  int B;
  int64_t n_chunks;
  const void* kv;
  int64_t n_rows;
  void* paged_out;
  int64_t n_pages;
  const int32_t* page_table;
  int max_pages;
  const int64_t* row_start;  // device [B+1]: rows of the requests before b (unused with inline_rows)
  int inline_rows;           // 1: row_start is `rows` below (B <= 256)
  int64_t rows[257];
  int64_t total_rows;        // rows of all requests: the CTAs share them in equal contiguous ranges
  int32_t* out_src;
  int32_t* out_delta;
  int32_t* out_pos_src;
  int* status;
  int interleaved;  // RoPE pairing: 0 NeoX (j, j+32), 1 interleaved (2j, 2j+1)
  struct {
    uint64_t F[32];
  } phase;
};

// A small chunk table travels inside the kernel's parameter block: the launch copies it from
// the validated host table, so no separate host-to-device copy (and no wait for one)
// precedes the kernel.  Kernels read it through the parameter's address (param space).
constexpr int kInlineChunks = 1024;
constexpr int kInlineIndptr = 257;  // B <= 256
struct InlineTable {
  irm_chunk chunks[kInlineChunks];
  int32_t indptr[kInlineIndptr];
};

// Fused attention (decode and prefill share one kernel).
struct AttnArgs {
  const void* q_lat;    // bf16 [B, n_q, H, 512]
  const void* q_rope;   // bf16 [B, n_q, H, 64]
  const void* kv;       // bf16 [n_rows, 576]
  const irm_chunk* chunks;
  const int32_t* indptr;
  int64_t n_rows;
  int64_t n_chunks;
  int B, n_q, H;
  int qpt;        // queries per 128-row tile = 128 / H
  int n_qtiles;   // ceil(n_q / qpt)
  int S;          // KV splits per query tile
  int Mv;         // stored query rows per tile (valid rows rounded up to 8)
  float scale_log2;
  void* out;      // bf16 [B, n_q, H, 512] (S == 1)
  float* lse;     // fp32 [B, n_q, H] or nullptr (S == 1)
  float* opart;   // fp32 [B, n_qtiles*S, 128, 512] (S > 1)
  float* lsepart; // fp32 [2 ranks][B, n_qtiles*S, 128] (S > 1)
  int* counters;  // int [B, n_qtiles, 2] finished-split counters, zero between calls (S > 1)
  int* status;
  int interleaved;  // RoPE pairing: 0 NeoX (j, j+32), 1 interleaved (2j, 2j+1)
  struct {
    uint64_t F[32];
  } phase;
  // Split boundaries: split s of a query tile starts at s * kv_tiles * split_num / split_den
  // (1 / S for equal splits).  Long-first launch (one query tile per request, S == 2): the cut
  // split_num / split_den is the long split's share, and the grid is (2 B, 2) so that every
  // long split precedes every short one.
  int long_first;
  int split_num, split_den;
  int inline_table;  // 1: the table is `tab` below (chunks / indptr unused)
  InlineTable tab;
};

// Split-KV decode for a few heads (one query token per request): one CTA per (request,
// split), the C splits of a request in one cluster that merges them in shared memory.
constexpr int kMaxDecodeCluster = 16;
// Where a decode split starts, taken from the validated host copy of the chunk table when
// the launch has at most kDecodeHints splits: its request's chunk range [c_begin, c_end) and
// context, and the chunk that holds the split's first row.  The kernel then starts without
// the dependent reads of indptr, the last chunk and the search for its first chunk.
struct DecodeHint {
  int32_t c_begin, c_end, ctx, c_first;
};
constexpr int kDecodeHints = 256;
struct DecodeArgs {
  const void* q_lat;    // bf16 [B, H, 512]
  const void* q_rope;   // bf16 [B, H, 64]
  const void* kv;       // bf16 [n_rows, 576]
  const irm_chunk* chunks;
  const int32_t* indptr;
  int64_t n_rows;
  int64_t n_chunks;
  int B, H;
  int C;          // CTAs per cluster (power of two, <= kMaxDecodeCluster)
  int G;          // clusters per request; the request's KV splits are C * G
  float scale_log2;
  void* out;      // bf16 [B, H, 512]
  float* lse;     // fp32 [B, H] or nullptr
  float* gpart;   // G > 1: fp32 [B, G, H, 512] normalised partial O of each cluster
  float* glse;    // G > 1: fp32 [B, G, H] its log2-sum-exp (scaled scores, log2 units)
  int* counters;  // G > 1: int [B, C] finished clusters per output slice, zero between calls
  int* status;
  int interleaved;  // RoPE pairing: 0 NeoX (j, j+32), 1 interleaved (2j, 2j+1)
  struct {
    uint64_t F[32];
  } phase;
  int n_hints;      // B * C * G when the hints below are filled in, else 0
  DecodeHint hint[kDecodeHints];  // [b * C * G + split]
  int inline_table;  // 1: the table is `tab` below (chunks / indptr unused)
  InlineTable tab;
};
// kernel parameter blocks are limited to 32764 bytes
static_assert(sizeof(DecodeArgs) <= 32764 && sizeof(AttnArgs) <= 32764, "kernel parameter block");

// Content-defined chunking of a batch of token streams.  A batch of at most kCdcInline
// streams carries its offsets and per-stream bases in the kernel parameters.
constexpr int kCdcInline = 1024;
struct CdcStreams {
  int64_t offsets[kCdcInline + 1];
  int64_t base[kCdcInline + 1];
  int64_t seg_base[kCdcInline + 1];
};
struct CdcArgs {
  const int32_t* tokens;    // [offsets[S]] token ids, streams concatenated
  const int64_t* offsets;   // device [S + 1] (unused with inline_streams)
  int S;
  const uint64_t* gear;     // device [vocab], or nullptr: SplitMix64 words from gear_seed
  uint64_t gear_seed;
  int vocab;
  int min_len, max_len, bits, mode;
  uint64_t seed;
  int64_t* base;            // workspace [S + 1]: first output slot of each stream
  int64_t* seg_base;        // workspace [S + 1]: first speculative segment of each stream
  uint32_t* words;          // workspace: candidate bitmask, stream s from word (offsets[s] >> 5) + s
  int32_t* spec_ends;       // workspace [segments][spec_cap]: speculative chunk ends
  int32_t* spec_count;      // workspace [segments]
  int32_t* spec_exit;       // workspace [segments]: first chunk start after the speculative walk
  uint64_t* spec_hash;      // workspace [segments][spec_cap]: fingerprints of the speculative chunks
  int64_t spec_cap;
  int64_t n_segs;           // speculative segments over all streams
  int32_t* n_chunks;        // [S]
  int32_t* chunk_start;     // [slots] stream-relative start of each chunk
  int32_t* chunk_len;       // [slots]
  uint64_t* chunk_hash;     // [slots] or nullptr
  int* status;
  int inline_streams;       // 1: offsets and bases are `ib` (S <= kCdcInline)
  CdcStreams ib;
};
static_assert(sizeof(CdcArgs) <= 32764, "kernel parameter block");
int cdc_segment_len();
cudaError_t launch_cdc(const CdcArgs& a, int64_t max_stream_len, int64_t slots, int64_t n_segs,
                       cudaStream_t stream);

// Copy of page-locked host arrays (device-accessible addresses) into a device block.
struct HostCopyArgs {
  const void* src[3];
  size_t off[3], bytes[3];
  uint8_t* dst;
  int n;
};
cudaError_t launch_host_copy(const HostCopyArgs& a, cudaStream_t stream);

cudaError_t launch_row_start(const irm_chunk* chunks, const int32_t* indptr, int B,
                             int64_t* row_start, cudaStream_t stream);
cudaError_t launch_rotate_gather(const GatherArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_mla_attn(const AttnArgs& a, cudaStream_t stream);
size_t attn_smem_bytes(int Mv);
int attn_max_active_clusters(int Mv);  // co-resident clusters of the attention kernel, 0 on error
bool decode_supported(int H);
int decode_max_active_clusters(int H, int C);  // 0 when C does not fit
cudaError_t launch_mla_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace irm
