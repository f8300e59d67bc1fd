/*
 * irm.h -- C ABI of the GB300 (sm_103a) reuse-time MLA KV reconstruction library.
 *
 * The method (Irminsul, position-independent caching for MLA models): a request's KV is
 * rebuilt from a content-addressed chunk pool.  Every KV row is [cKV (512 bf16,
 * position-free) | k_r (64 bf16, RoPE slice)].  A chunk cached at source position p_src
 * and reused at target position p_tgt keeps its cKV rows untouched and has its k_r rows
 * rotated in closed form by R(delta), delta = p_tgt - p_src, because
 * R(delta) R(p_src) = R(p_tgt).  Positions 0..31 are always freshly prefilled.
 *   Passages: "Irminsul论文详解：面向Agentic LLM Serving的MLA原生位置无关缓存"
 *   (gentlecold.top) §4 (row split, delta rule), §5 (assembly loop), §7 (carve-out),
 *   §15 (worked example); "Irminsul: MLA-Native Position-Independent Caching for Agentic
 *   LLM Serving" (gist.science technical summary) §2.1-2.2.
 *
 * Conventions fixed here where the pages are silent:
 *   - The default RoPE is the NeoX half split: pair j couples k_r[j] and k_r[j+32] and
 *     turns by angle delta * theta_j, theta_j = 10000^(-2j/64), j = 0..31.  The *_rope entry
 *     points take the model's own frequencies and pairing instead (irm_rope).  Rotation
 *     math is fp32, the rotated k_r is rounded to bf16 (round to nearest even) once.
 *   - A fresh chunk (reused = 0) has delta = 0; its p_src is ignored.
 *   - Query i of n_q sits at position ctx - n_q + i and sees keys t <= that position.
 *
 * Memory and streams.  Pointers named *_host are host memory, every other buffer is device
 * memory; the caller owns all of them, and the library keeps no allocation of its own.
 * Every call is asynchronous on `stream`.
 *
 * Chunk tables.  A call takes the batch's chunk tables in host memory only (chunks_host,
 * indptr_host, and for irm_cdc_chunk the stream offsets).  The library validates them,
 * plans the launch from them, and hands those same bytes to the kernels, so the kernels
 * always run on exactly the table that was validated:
 *   - The attention calls pass a table of at most 1024 records for at most 256 requests
 *     inside the kernel launch's parameter block, which the CUDA runtime copies when the
 *     kernel is launched: no separate copy, any host memory, and the caller may reuse the
 *     table as soon as the call returns (a captured graph replays the table as validated).
 *   - Otherwise the library copies the table into the table area of the caller's workspace
 *     on `stream` before the kernels that read it.
 *     Page-locked (pinned) host tables are read when `stream` reaches the call: by a small copy
 *     kernel of the library straight from host memory (memory mapped for the device, as
 *     cudaHostAlloc / cudaMallocHost give), else by cudaMemcpyAsync.  Keep them unchanged until
 *     `stream` has passed the call.  Under CUDA stream capture the copy becomes part of the
 *     graph and every replay reads the same host bytes again, so they must stay unchanged for
 *     as long as the graph is replayed (the launch geometry was planned from them).
 *     Pageable host tables are packed by the library and handed to the CUDA runtime
 *     (cudaMemcpyAsync, host to device), which has read them when the call returns, so the
 *     caller may reuse them at once; such a copy cannot be captured into a CUDA graph
 *     (IRM_ERR_INVALID_ARG during capture).
 * Kernels still re-check each source row against n_rows and each page index against
 * n_pages, and record (never fault on) a violation.
 *
 * Errors.  Calls return an irm_status.  No exception crosses the ABI and nothing aborts.
 * Host-side checks happen before any copy or launch.  Device-side problems (a page index
 * outside the paged output, a source row outside the row store, or a pipeline wait that
 * exceeded its 2 s limit) set bits in the status word at the start of the workspace; read
 * and clear it with irm_device_status().
 *
 * Workspace.  Each call takes a caller-owned device workspace, 256-byte aligned, of at
 * least the size its *_workspace_size function reports for the same tables.  Its first
 * IRM_WORKSPACE_HEADER bytes hold the device status word, the next ones the copied chunk
 * table, the rest the call's scratch.  Zero the whole workspace once before first use:
 * decode keeps split-KV completion counters in it, which every call leaves at zero again.
 * After a call that reported a device error, zero it again.  Calls that share one
 * workspace must not overlap on the GPU.
 */
#ifndef IRM_H_
#define IRM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t; /* identical to the CUDA runtime's typedef */

#define IRM_D_LAT 512        /* cKV width */
#define IRM_D_ROPE 64        /* k_r width */
#define IRM_D_ROW 576        /* KV row width, elements (1152 bytes in bf16) */
#define IRM_PAGE_ROWS 64     /* rows per page of the paged KV layout */
#define IRM_CARVE_OUT 32     /* positions 0..31 are always fresh */
#define IRM_MAX_HEADS 128
#define IRM_WORKSPACE_HEADER 256

typedef enum irm_status {
  IRM_OK = 0,
  IRM_ERR_INVALID_ARG = -1,    /* null/misaligned pointer, bad size or count */
  IRM_ERR_CHUNK_TABLE = -2,    /* chunks do not tile [0, ctx) in order, len <= 0, rows out of range */
  IRM_ERR_CARVEOUT = -3,       /* a reused chunk covers a position < 32 */
  IRM_ERR_UNSUPPORTED = -4,    /* shape outside what the kernels implement */
  IRM_ERR_CUDA = -5,           /* a CUDA runtime call failed (see irm_last_error) */
  IRM_ERR_DEVICE_TIMEOUT = -6, /* a device pipeline wait ran out (from irm_device_status) */
  IRM_ERR_DEVICE_BOUNDS = -7,  /* a kernel met a source row outside the row store */
  IRM_ERR_WORKSPACE = -8       /* workspace missing or smaller than required */
} irm_status;

/* One chunk of a request's table, listed in target order [walkthrough §5].
 * Rows pool_offset .. pool_offset+len-1 of the row store become target positions
 * p_tgt .. p_tgt+len-1.  24 bytes, naturally aligned. */
typedef struct irm_chunk {
  int64_t pool_offset; /* first row of the chunk in the row store */
  int32_t len;         /* rows, > 0 */
  int32_t p_src;       /* position the cached k_r rows were encoded at (reused chunks) */
  int32_t p_tgt;       /* target position of the first row; chunks tile [0, ctx) in order */
  uint8_t reused;      /* 1: cached chunk, k_r rotated by p_tgt - p_src; 0: fresh */
  uint8_t pad[3];
} irm_chunk;

/*
 * RoPE variant of the cached k_r slice.  The delta-rotation is only right when it uses the
 * model's own rotary class: the same inv_freq table and pairing as the prefill that wrote
 * the cache ["Irminsul论文详解" §11: with a plain base-10000 fallback instead of the model's
 * rotary class, reuse was worse than naive reuse].
 *   inv_freq[j]  theta_j, the angle per position of pair j in radians (any finite value;
 *                base-b RoPE has theta_j = b^(-2j/64); scaled tables such as YaRN's are
 *                passed as they are)
 *   pairing      IRM_ROPE_NEOX: pair j = dims (j, j+32) of k_r;
 *                IRM_ROPE_INTERLEAVED: pair j = dims (2j, 2j+1)
 * A RoPE attention scaling factor does not enter the delta-rotation: it is already part of
 * the cached k_r, and R(delta) only turns pairs.  The host turns theta_j into a 64-bit
 * fixed-point phase step (one turn = 2^64, theta_j / 2pi rounded in fp64), and the kernels
 * reduce delta * step to one turn exactly in integer arithmetic for every int32 delta.
 * Passing NULL selects the default convention above.
 */
#define IRM_ROPE_NEOX 0
#define IRM_ROPE_INTERLEAVED 1
typedef struct irm_rope {
  double inv_freq[32];
  int32_t pairing;
  int32_t reserved; /* 0 */
} irm_rope;

/* Text for a status code (static storage). */
const char* irm_status_string(int status);

/* Detail of the last error raised on the calling thread ("" if none). */
const char* irm_last_error(void);

/* Library build identifier: "irm <version> sm_103a". */
const char* irm_version(void);

/*
 * Host-only validation of a batch of chunk tables (no GPU needed).
 *   chunks_host  [indptr_host[B]] records; request b owns [indptr_host[b], indptr_host[b+1])
 *   indptr_host  [B+1], indptr_host[0] == 0, non-decreasing
 *   n_rows       rows in the row store (every source row must lie in [0, n_rows))
 *   ctx_out      [B] or NULL: receives each request's context length
 * Returns IRM_OK, IRM_ERR_CHUNK_TABLE, IRM_ERR_CARVEOUT or IRM_ERR_INVALID_ARG.
 */
irm_status irm_validate_chunks(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                               int64_t n_rows, int64_t* ctx_out);

/*
 * Reads and clears the device status word of a workspace (synchronizes `stream`).
 * Returns IRM_OK, IRM_ERR_DEVICE_TIMEOUT, IRM_ERR_DEVICE_BOUNDS or IRM_ERR_CUDA.
 */
irm_status irm_device_status(void* workspace, cudaStream_t stream);

/*
 * Self-test of the bounded pipeline wait (the pages have no counterpart; for tests).  Launches
 * one warp on `stream` that waits on a barrier nothing ever arrives on; the wait gives up after
 * its time limit (2 s), exactly as a stalled pipeline wait of the other kernels would, and sets
 * the timeout bit of the workspace status word.  irm_device_status() then returns
 * IRM_ERR_DEVICE_TIMEOUT, and the context stays usable.
 *   workspace  device, 256-byte aligned, >= IRM_WORKSPACE_HEADER bytes (its status word is used)
 * Returns IRM_OK (launched), IRM_ERR_WORKSPACE or IRM_ERR_CUDA.
 */
irm_status irm_selftest_wait_timeout(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Rotate+gather into a paged KV layout, and/or the per-row assembly plan.
 * [walkthrough §5 assembly loop: reused chunks contribute (cKV, R(delta) k_r,base)]
 *
 * For target row t of request b, with c its chunk:
 *   src_row = pool_offset_c + (t - p_tgt_c); delta = reused_c ? p_tgt_c - p_src_c : 0
 *   paged_out[page_table[b*max_pages + t/64]*64 + t%64] = [cKV(src_row) | R(delta) k_r(src_row)]
 * cKV bytes are copied unchanged; rows with delta = 0 are copied bit for bit.
 *
 *   chunks_host, indptr_host, B   host chunk tables (validated, then copied into the
 *                workspace; see "Chunk tables" above)
 *   kv_rows      device bf16 [n_rows, 576], 16-byte aligned
 *   paged_out    device bf16 [n_pages, 64, 576] or NULL (plan only); rows of a page that
 *                no target row maps to are left untouched
 *   page_table   device int32 [B, max_pages] (required when paged_out != NULL); every
 *                entry used must lie in [0, n_pages) -- the kernel skips a row whose page
 *                is out of range and records IRM_ERR_DEVICE_BOUNDS
 *   out_src_row, out_delta, out_pos_src   device int32 [sum ctx] or NULL; rows are listed
 *                request after request (pos_src = t - delta)
 * Workspace: irm_assemble_kv_workspace_size bytes for the same tables.
 */
irm_status irm_assemble_kv_workspace_size(const irm_chunk* chunks_host, const int32_t* indptr_host,
                                          int B, size_t* bytes);
irm_status irm_assemble_kv(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                           const void* kv_rows, int64_t n_rows, void* paged_out,
                           int64_t n_pages, const int32_t* page_table, int max_pages,
                           int32_t* out_src_row,
                           int32_t* out_delta, int32_t* out_pos_src, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);
/* Same, with the model's RoPE variant (rope == NULL: the default).  IRM_ERR_INVALID_ARG for a
 * pairing other than the two above, a non-zero reserved field or a non-finite frequency. */
irm_status irm_assemble_kv_rope(const irm_chunk* chunks_host, const int32_t* indptr_host, int B,
                                const void* kv_rows, int64_t n_rows, void* paged_out,
                                int64_t n_pages, const int32_t* page_table, int max_pages,
                                int32_t* out_src_row, int32_t* out_delta, int32_t* out_pos_src,
                                const irm_rope* rope, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * Fused delta-rotate + absorbed MLA decode attention (one query token per request).
 * [walkthrough §4: scores over [cKV | k_r], output P.cKV; the rotation is applied on the
 *  HBM -> shared memory load path, so rotated keys are never written back]
 *
 *   q_lat   device bf16 [B, H, 512]   absorbed query (W_UK folded in)
 *   q_rope  device bf16 [B, H, 64]    RoPE query slice, already encoded at position ctx-1
 *   H       1..128 heads
 *   kv_rows device bf16 [n_rows, 576]
 *   softmax_scale  scale applied to q.k (1/sqrt(192) for DeepSeek-V2/V3 shapes)
 *   out     device bf16 [B, H, 512]:  O = softmax(s) . cKV, s_t = scale * (q_lat.cKV_t +
 *           q_rope.R(delta_t) k_r,t)
 *   lse     device fp32 [B, H] or NULL: natural-log sum of exp(s_t)
 * Workspace: irm_mla_attn_decode_workspace_size bytes for the same tables and H (the copied
 * chunk table and the split-KV partials).
 */
irm_status irm_mla_attn_decode_workspace_size(const irm_chunk* chunks_host,
                                              const int32_t* indptr_host, int B, int H,
                                              size_t* bytes);
irm_status irm_mla_attn_decode(const void* q_lat, const void* q_rope, int B, int H,
                               const irm_chunk* chunks_host, const int32_t* indptr_host,
                               const void* kv_rows, int64_t n_rows, float softmax_scale,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);
/* Same, with the model's RoPE variant (rope == NULL: the default; errors as for
 * irm_assemble_kv_rope). */
irm_status irm_mla_attn_decode_rope(const void* q_lat, const void* q_rope, int B, int H,
                                    const irm_chunk* chunks_host, const int32_t* indptr_host,
                                    const void* kv_rows, int64_t n_rows, float softmax_scale,
                                    void* out, float* lse, const irm_rope* rope, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode without any device allocation by the caller.  The method's pages have no
 * counterpart to this entry point: it exists for callers that cannot call cudaMalloc --
 * for example a plugin that runs inside a host application which owns the device memory
 * pool, or code that must not allocate while a CUDA graph is being built -- and so cannot
 * provide the workspace that irm_mla_attn_decode wants.
 *
 * Same arguments and results as irm_mla_attn_decode, minus the workspace.  The split-KV
 * scratch and the copied chunk table live in a fixed 32 MiB device array inside this library
 * (every GPU that loads the library holds it until the process exits).  The split of the
 * decode is chosen within that scratch: where irm_mla_attn_decode would use a split whose
 * scratch does not fit, this call uses the split it would otherwise take (same results up to
 * rounding order).  A decode whose table and scratch would still exceed 32 MiB
 * (IRM_ERR_WORKSPACE) is rejected before anything is copied or launched; use
 * irm_mla_attn_decode then.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current and caches it per
 * device ordinal, which assumes the CUDA runtime's primary context of that device (a caller
 * that binds another context through the driver API must not use this entry point); make
 * that first call before any stream capture.  Each call clears the array's split-KV
 * completion counters on `stream` (cudaMemsetAsync) and allocates nothing.  All calls share
 * the one array: calls that overlap on the GPU (other streams, other threads) race and must
 * be serialized by the caller.  Device-side status (timeouts, out-of-range rows) collects in
 * the array's own status word across calls: read and clear it with
 * irm_decode_noalloc_status().
 */
irm_status irm_mla_attn_decode_noalloc(const void* q_lat, const void* q_rope, int B, int H,
                                       const irm_chunk* chunks_host, const int32_t* indptr_host,
                                       const void* kv_rows, int64_t n_rows, float softmax_scale,
                                       void* out, float* lse, cudaStream_t stream);
/* Reads and clears the status word of the no-allocation scratch array of the current device
 * (synchronizes `stream`).  Returns what irm_device_status() returns for a workspace. */
irm_status irm_decode_noalloc_status(cudaStream_t stream);

/*
 * Fused delta-rotate + absorbed MLA prefill attention (n_q causal query tokens per request,
 * the last n_q positions of each request's assembled context).
 *   q_lat [B, n_q, H, 512], q_rope [B, n_q, H, 64], out [B, n_q, H, 512] bf16,
 *   lse [B, n_q, H] fp32 or NULL; 1 <= n_q <= ctx_b for every request.
 * Workspace: irm_mla_attn_prefill_workspace_size bytes for the same tables.
 */
irm_status irm_mla_attn_prefill_workspace_size(const irm_chunk* chunks_host,
                                               const int32_t* indptr_host, int B, int n_q, int H,
                                               size_t* bytes);
irm_status irm_mla_attn_prefill(const void* q_lat, const void* q_rope, int B, int n_q, int H,
                                const irm_chunk* chunks_host, const int32_t* indptr_host,
                                const void* kv_rows, int64_t n_rows, float softmax_scale,
                                void* out, float* lse, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);
/* Same, with the model's RoPE variant (rope == NULL: the default; errors as for
 * irm_assemble_kv_rope). */
irm_status irm_mla_attn_prefill_rope(const void* q_lat, const void* q_rope, int B, int n_q, int H,
                                     const irm_chunk* chunks_host, const int32_t* indptr_host,
                                     const void* kv_rows, int64_t n_rows, float softmax_scale,
                                     void* out, float* lse, const irm_rope* rope, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/*
 * Content-defined chunking of token streams, the step that cuts a request's unmatched tail
 * into content-addressed chunks before the registry lookup ["Irminsul: MLA-Native
 * Position-Independent Caching for Agentic LLM Serving" technical summary §2.2: rolling Gear
 * hash over 64-token windows, xxHash64 fingerprints; "Irminsul论文详解" §6: 7-bit boundary
 * test, chunk length clipped to [32, 512]].
 *   h_i = sum_{k=0}^{min(i,63)} gear[x_{i-k}] * 2^k mod 2^64, gear either a caller table or,
 *   when gear == NULL, generated: gear[t] = the (t+1)-th output of SplitMix64 seeded with
 *   params->gear_seed (a published counter-based generator; no table lookups on the GPU)
 *   position i is a boundary candidate when the 7-bit test passes:
 *     IRM_CDC_THRESHOLD: h_i < 2^(64 - bits) (the hash "falls below a threshold"; this test
 *                        reads bits that depend on the whole 64-token window)
 *     IRM_CDC_LOW_BITS:  h_i mod 2^bits == 0 (the "low 7 bits" wording; with this hash those
 *                        bits depend only on the last `bits` tokens)
 *   a chunk starting at s ends at the first candidate i >= s + min_len - 1, else at
 *   s + max_len - 1, else at the end of the stream (the last chunk may be shorter);
 *   its fingerprint is xxHash64 (seed `seed`) of its token ids as little-endian int32 bytes.
 * params NULL: min_len 32, max_len 512, bits 7, IRM_CDC_THRESHOLD, seed 0, gear_seed 0.
 */
#define IRM_CDC_THRESHOLD 0
#define IRM_CDC_LOW_BITS 1
typedef struct irm_cdc_params {
  int32_t min_len; /* >= 1 */
  int32_t max_len; /* >= min_len, <= 65536 */
  int32_t bits;    /* 1 .. 63 */
  int32_t mode;    /* IRM_CDC_THRESHOLD or IRM_CDC_LOW_BITS */
  uint64_t seed;      /* xxHash64 seed of the fingerprints */
  uint64_t gear_seed; /* SplitMix64 seed of the generated Gear words (gear == NULL) */
} irm_cdc_params;

/*
 * Sizes for irm_cdc_chunk:
 *   offsets_host  [n_streams + 1] int64, offsets_host[0] == 0, non-decreasing; stream s is
 *                 tokens[offsets[s] .. offsets[s+1]), at most INT32_MAX tokens long
 *   bytes         workspace bytes
 *   slots         output slots: stream s owns slots [base_s, base_s + len_s / min_len + 1),
 *                 base_s = sum over earlier streams of (len / min_len + 1)
 */
irm_status irm_cdc_sizes(const int64_t* offsets_host, int n_streams, const irm_cdc_params* params,
                         size_t* bytes, int64_t* slots);

/*
 *   tokens       device int32 [offsets[n_streams]], ids in [0, vocab) (an id outside is
 *                read as gear = 0 and recorded as IRM_ERR_DEVICE_BOUNDS in the status word)
 *   offsets_host the stream offsets (validated, then copied into the workspace like a
 *                chunk table; see "Chunk tables" above)
 *   gear         device uint64 [vocab], the Gear table, or NULL for generated Gear words
 *   vocab        token ids lie in [0, vocab)
 *   n_chunks     device int32 [n_streams]: chunks of each stream
 *   chunk_start  device int32 [slots]: stream-relative first token of each chunk (see
 *                irm_cdc_sizes for the slot layout)
 *   chunk_len    device int32 [slots]
 *   chunk_hash   device uint64 [slots] or NULL (no fingerprints)
 * Workspace: irm_cdc_sizes bytes, 256-byte aligned (its status word as for the other calls).
 */
irm_status irm_cdc_chunk(const int32_t* tokens, const int64_t* offsets_host, int n_streams,
                         const uint64_t* gear, int32_t vocab,
                         const irm_cdc_params* params, int32_t* n_chunks, int32_t* chunk_start,
                         int32_t* chunk_len, uint64_t* chunk_hash, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * Content-addressed chunk registry and chunk-table assembler (host side): the step that turns a
 * request into the chunk table the kernels above consume ["Irminsul论文详解" §5: exact prefix
 * first; then per CDC segment of the tail at target position p: p < 32 is prefilled (first-chunk
 * carve-out), a registry hit on the segment's fingerprint is reused with delta = p - p_src, a
 * miss is prefilled and registered at p; §6: the S1 fallback looks a missed chunk up again as
 * fixed 128-token sub-windows].
 *   The registry keys chunks by (xxHash64 fingerprint, length) and keeps their rows in a ring of
 *   pool_rows rows starting at row pool_base of the row store: a newly prefilled chunk takes the
 *   next rows of the ring (a chunk never wraps around the ring's end), and an entry becomes stale
 *   once the ring has moved a full turn past its first row (eviction by age).  capacity is the
 *   expected number of live entries (the table grows when needed).  All calls on one registry are
 *   serialized by a mutex; the registry is host memory only.
 */
typedef struct irm_registry irm_registry;
irm_status irm_registry_create(int64_t pool_base, int64_t pool_rows, int64_t capacity, irm_registry** out);
void irm_registry_destroy(irm_registry* reg);
/* Live (not stale) entries and rows allocated so far. */
irm_status irm_registry_stats(irm_registry* reg, int64_t* live_entries, int64_t* rows_allocated);

#define IRM_ASSEMBLE_S1 1 /* flags: look missed chunks up again as 128-token sub-windows */
/*
 * Chunk table of one request.
 *   tokens_host   the request's n_tokens token ids (needed with IRM_ASSEMBLE_S1, else may be NULL)
 *   prefix_len    tokens matched exactly by a prefix cache; they are reused in place from row
 *                 prefix_row on (one chunk, delta 0, not prefilled)
 *   seg_*         the n_seg CDC segments of the tail (tokens prefix_len ..), in order: start
 *                 relative to the tail, length, fingerprint (e.g. irm_cdc_chunk's outputs)
 *   flags, seed   IRM_ASSEMBLE_S1 or 0; xxHash64 seed of the S1 sub-window fingerprints
 *   chunks_out    [chunks_cap] the chunk table (irm_chunk, target order, tiling [0, n_tokens));
 *                 1 + n_seg entries suffice, 1 + sum ceil(len / 128) with IRM_ASSEMBLE_S1
 *   prefill_out   [chunks_cap] 1 where the caller must prefill the chunk's rows (pool_offset ..
 *                 pool_offset + len - 1 of the row store, at positions p_tgt ..) before the next
 *                 request can reuse them; 0 for reused and prefix chunks
 *   n_chunks_out  entries written
 * A chunk registered while assembling a request is not reused by later segments of the same
 * request.  Errors: IRM_ERR_INVALID_ARG for segments that do not tile the tail, a segment longer
 * than the pool or too small a capacity (nothing is changed then).
 */
irm_status irm_registry_assemble(irm_registry* reg, const int32_t* tokens_host, int64_t n_tokens,
                                 int64_t prefix_len, int64_t prefix_row, const int32_t* seg_start,
                                 const int32_t* seg_len, const uint64_t* seg_hash, int32_t n_seg,
                                 int32_t flags, uint64_t seed, irm_chunk* chunks_out,
                                 uint8_t* prefill_out, int32_t chunks_cap, int32_t* n_chunks_out);

#ifdef __cplusplus
}
#endif

#endif /* IRM_H_ */
