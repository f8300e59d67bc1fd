/*
 * irm_oracle.c -- reference oracle for delta-rotated MLA KV reconstruction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the benchmark's CPU
 * baseline may load this library.  The product path never calls it, and it shares no
 * code, header, table or constant with the CUDA path.
 *
 * Plain fp64 loops; OpenMP only over independent query rows.  No blocking, fusion or
 * reordering beyond the definitions below, so each step can be read against the pages.
 *
 * Pages cited (the web pages describing the method):
 *   [walkthrough] "Irminsul论文详解：面向Agentic LLM Serving的MLA原生位置无关缓存"
 *                 (gentlecold.top), sections numbered as on the page;
 *   [summary]     "Irminsul: MLA-Native Position-Independent Caching for Agentic LLM
 *                 Serving" (gist.science, French and Korean technical summary), sections
 *                 numbered as on the page.
 *
 * What is computed:
 *   - a KV row is [cKV (512, position-free) | k_r (64, RoPE slice)]     [walkthrough §4],
 *                                                                        [summary §2.1]
 *   - a reused chunk at target position p_tgt, cached at p_src, has
 *     delta = p_tgt - p_src and k_r,rot = R(delta) k_r,base, because
 *     R(delta) R(p_src) = R(p_tgt); cKV is reused untouched            [walkthrough §4, §15],
 *                                                                        [summary §2.2]
 *   - the assembly loop appends, per segment, either freshly prefilled rows or the
 *     cached rows with rotated k_r; positions below 32 are always fresh [walkthrough §5, §7]
 *   - absorbed MLA attention: scores use [cKV | k_r] against [q_lat | q_rope], the output
 *     is the softmax-weighted sum of cKV (W_UV applied outside)          [walkthrough §4]
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - default RoPE convention: NeoX half split, pair j couples dims (j, j+32), frequency
 *     theta_j = 10000^(-2j/64), j = 0..31; R(p) turns pair j by angle +p*theta_j.
 *   - RoPE variants [walkthrough §11: the rotary class and inv_freq must match the model]:
 *     the *_ex functions take the 32 frequencies theta_j (radians per position) and the
 *     pairing (0: NeoX half split, pair j = dims (j, j+32); 1: interleaved, pair j = dims
 *     (2j, 2j+1)).  Attention scaling does not enter R(delta): the cached k_r already
 *     carries it and R(delta) only turns pairs.
 *   - a fresh row (reused = 0) has delta = 0 and is passed through unchanged.
 *   - softmax scale is a caller argument (1/sqrt(192) for the configurations used here).
 *   - query i of n_q sits at position ctx - n_q + i and sees keys t <= that position.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

#define D_LAT 512
#define D_ROPE 64
#define D_ROW 576
#define N_PAIRS 32
#define CARVE_OUT 32

/* bf16 bit pattern -> fp64, exact: the bf16 value is the top half of an IEEE float. */
static double bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* RoPE frequencies, NeoX half split: theta_j = 10000^(-2j/64).  (reading, see header) */
void oracle_rope_theta(double *theta) {
  for (int j = 0; j < N_PAIRS; ++j) theta[j] = pow(10000.0, -2.0 * (double)j / (double)D_ROPE);
}

/* The two dims of pair j: NeoX half split (j, j+32) or interleaved (2j, 2j+1). */
static void pair_dims(int pairing, int j, int *dx, int *dy) {
  if (pairing == 1) {
    *dx = 2 * j;
    *dy = 2 * j + 1;
  } else {
    *dx = j;
    *dy = j + N_PAIRS;
  }
}

/* R(steps) applied to one 64-d row: pair j = (x, y) is turned by angle steps * theta_j,
 * (x, y) -> (x cos - y sin, x sin + y cos).  Used both for R(delta) [walkthrough §4] and
 * for R(p). */
static void rotate_row(const double *k, i64 steps, const double *theta, int pairing, double *out) {
  for (int j = 0; j < N_PAIRS; ++j) {
    int dx, dy;
    pair_dims(pairing, j, &dx, &dy);
    double ang = (double)steps * theta[j];
    double c = cos(ang), s = sin(ang);
    double x = k[dx], y = k[dy];
    out[dx] = x * c - y * s;
    out[dy] = x * s + y * c;
  }
}

/* out[r] = R(steps[r]) k[r] for n rows of 64 values, with an explicit RoPE spec. */
void oracle_rotate_ex(const double *k, i64 n, const i64 *steps, const double *theta, int pairing,
                      double *out) {
  for (i64 r = 0; r < n; ++r) rotate_row(k + r * D_ROPE, steps[r], theta, pairing, out + r * D_ROPE);
}

/* Same with the default convention. */
void oracle_rotate(const double *k, i64 n, const i64 *steps, double *out) {
  double theta[N_PAIRS];
  oracle_rope_theta(theta);
  oracle_rotate_ex(k, n, steps, theta, 0, out);
}

/*
 * Assembly plan [walkthrough §5 pseudo-code, §4 delta rule].
 * Chunk table of all requests, concatenated; request b owns chunks [indptr[b], indptr[b+1])
 * listed in target order.  For target row t of chunk c:
 *   src_row = pool_offset_c + (t - p_tgt_c)
 *   delta   = reused_c ? p_tgt_c - p_src_c : 0
 *   pos_src = t - delta
 * Rows are written request after request (row offset of request b = sum of earlier ctx).
 * Returns 0, or -1 if a request's chunks do not tile [0, ctx) in order, or -2 if a reused
 * chunk covers a position below 32 (the carve-out is always prefilled [walkthrough §7]).
 */
int oracle_plan(i64 B, const i64 *indptr, const i64 *pool_offset, const i64 *len,
                const i64 *p_src, const i64 *p_tgt, const uint8_t *reused, i64 *ctx_out,
                i64 *src_row, i64 *delta, i64 *pos_src) {
  i64 row = 0;
  for (i64 b = 0; b < B; ++b) {
    i64 expect = 0;
    for (i64 c = indptr[b]; c < indptr[b + 1]; ++c) {
      if (p_tgt[c] != expect || len[c] <= 0) return -1;
      if (reused[c] && p_tgt[c] < CARVE_OUT) return -2;
      for (i64 i = 0; i < len[c]; ++i) {
        i64 t = p_tgt[c] + i;
        i64 d = reused[c] ? p_tgt[c] - p_src[c] : 0;
        src_row[row] = pool_offset[c] + i;
        delta[row] = d;
        pos_src[row] = t - d;
        ++row;
      }
      expect += len[c];
    }
    ctx_out[b] = expect;
  }
  return 0;
}

/*
 * Assembled KV rows in fp64: out[r] = [cKV(src_row[r]) | R(delta[r]) k_r(src_row[r])].
 * kv_rows is the bf16 row store [n_rows, 576]; cKV is only widened, never modified.
 * RoPE spec as in oracle_rotate_ex.
 */
void oracle_assemble_ex(const uint16_t *kv_rows, i64 n, const i64 *src_row, const i64 *delta,
                        const double *theta, int pairing, double *out) {
#pragma omp parallel for schedule(static)
  for (i64 r = 0; r < n; ++r) {
    const uint16_t *src = kv_rows + src_row[r] * D_ROW;
    double *dst = out + r * D_ROW;
    double kr[D_ROPE];
    for (int d = 0; d < D_LAT; ++d) dst[d] = bf16_to_f64(src[d]);
    for (int d = 0; d < D_ROPE; ++d) kr[d] = bf16_to_f64(src[D_LAT + d]);
    if (delta[r] == 0) {
      for (int d = 0; d < D_ROPE; ++d) dst[D_LAT + d] = kr[d];
    } else {
      rotate_row(kr, delta[r], theta, pairing, dst + D_LAT);
    }
  }
}

/* Same with the default convention. */
void oracle_assemble(const uint16_t *kv_rows, i64 n, const i64 *src_row, const i64 *delta,
                     double *out) {
  double theta[N_PAIRS];
  oracle_rope_theta(theta);
  oracle_assemble_ex(kv_rows, n, src_row, delta, theta, 0, out);
}

/*
 * Absorbed MLA attention for R query rows [walkthrough §4].
 *   q[r]    = [q_lat | q_rope] of row r, fp64 [576]
 *   K       = assembled rows of one request, fp64 [ctx, 576]
 *   visible = number of keys row r sees (keys 0..visible-1)
 *   s_t = scale * (q_lat . cKV_t + q_rope . k_r,t)
 *   O   = sum_t exp(s_t - m) cKV_t / sum_t exp(s_t - m),  m = max_t s_t
 *   lse = m + ln sum_t exp(s_t - m)
 */
void oracle_attn(const double *q, const i64 *visible, i64 R, const double *K, i64 ctx,
                 double scale, double *O, double *lse) {
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
#pragma omp for schedule(dynamic, 1)
    for (i64 r = 0; r < R; ++r) {
      const double *qr = q + r * D_ROW;
      i64 n = visible[r];
      double m = -INFINITY;
      for (i64 t = 0; t < n; ++t) {
        const double *kt = K + t * D_ROW;
        double acc = 0.0;
        for (int d = 0; d < D_ROW; ++d) acc += qr[d] * kt[d];
        s[t] = acc * scale;
        if (s[t] > m) m = s[t];
      }
      double *o = O + r * D_LAT;
      for (int d = 0; d < D_LAT; ++d) o[d] = 0.0;
      double l = 0.0;
      for (i64 t = 0; t < n; ++t) {
        double p = exp(s[t] - m);
        l += p;
        const double *kt = K + t * D_ROW;
        for (int d = 0; d < D_LAT; ++d) o[d] += p * kt[d];
      }
      for (int d = 0; d < D_LAT; ++d) o[d] /= l;
      lse[r] = m + log(l);
    }
    free(s);
  }
}

/* Widen bf16 bit patterns to fp64 (n values). */
void oracle_widen(const uint16_t *src, i64 n, double *dst) {
  for (i64 i = 0; i < n; ++i) dst[i] = bf16_to_f64(src[i]);
}

/* Number of threads OpenMP would use (reported with timings). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Sets the number of OpenMP threads of later calls (timing runs; results do not depend on it). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------------------
 * Content-defined chunking of a token stream [summary §2.2, walkthrough §6].
 *   Gear hash over a 64-token window: h_i = sum_{k=0}^{min(i,63)} G[x_{i-k}] * 2^k
 *   (mod 2^64), G a 64-bit table indexed by token id (an input).
 *   A position i is a boundary candidate when the hash passes the 7-bit test:
 *     mode 0 (threshold): h_i < 2^(64 - bits)    (reading: "falls below a threshold")
 *     mode 1 (low bits):  h_i mod 2^bits == 0    (the walkthrough's "low 7 bits" wording)
 *   A chunk starting at s ends at the first candidate i with i - s + 1 >= min_len, or at
 *   i = s + max_len - 1, or at the end of the stream; the next chunk starts at i + 1.
 * ------------------------------------------------------------------------------------ */

/* Window sum, written out term by term. */
void oracle_gear_hash(const int32_t *tokens, i64 n, const uint64_t *gear, uint64_t *h) {
  for (i64 i = 0; i < n; ++i) {
    uint64_t acc = 0;
    for (int k = 0; k < 64 && k <= i; ++k) acc += gear[tokens[i - k]] << k;
    h[i] = acc;
  }
}

static int cdc_candidate(uint64_t h, int bits, int mode) {
  if (mode == 1) return (h & ((1ull << bits) - 1ull)) == 0ull;
  return (h >> (64 - bits)) == 0ull;
}

/* Chunks of one stream; returns their count (starts / lens must hold n entries). */
i64 oracle_cdc(const int32_t *tokens, i64 n, const uint64_t *gear, int min_len, int max_len,
               int bits, int mode, i64 *starts, i64 *lens) {
  uint64_t *h = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(n > 0 ? n : 1));
  oracle_gear_hash(tokens, n, gear, h);
  i64 count = 0, s = 0;
  for (i64 i = 0; i < n; ++i) {
    i64 len = i - s + 1;
    int end = (len >= min_len && cdc_candidate(h[i], bits, mode)) || len == max_len || i == n - 1;
    if (end) {
      starts[count] = s;
      lens[count] = len;
      ++count;
      s = i + 1;
    }
  }
  free(h);
  return count;
}

/* ------------------------------------------------------------------------------------
 * xxHash64 of a byte string (Y. Collet's XXH64: four 64-bit lanes over 32-byte stripes,
 * lane merge, then 8-, 4- and 1-byte tails and the final avalanche), used as the chunk
 * fingerprint [summary §2.2].  The chunk's token ids are hashed as little-endian int32.
 * ------------------------------------------------------------------------------------ */
static const uint64_t XP1 = 11400714785074694791ull, XP2 = 14029467366897019727ull,
                      XP3 = 1609587929392839161ull, XP4 = 9650029242287828579ull,
                      XP5 = 2870177450012600261ull;

static uint64_t rotl64(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
static uint64_t rd64(const uint8_t *p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint32_t rd32(const uint8_t *p) {
  uint32_t v = 0;
  for (int i = 3; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}
static uint64_t xround(uint64_t acc, uint64_t input) {
  acc += input * XP2;
  acc = rotl64(acc, 31);
  return acc * XP1;
}
static uint64_t xmerge(uint64_t acc, uint64_t v) {
  acc ^= xround(0, v);
  return acc * XP1 + XP4;
}

uint64_t oracle_xxh64(const uint8_t *p, i64 len, uint64_t seed) {
  const uint8_t *end = p + len;
  uint64_t h;
  if (len >= 32) {
    uint64_t v1 = seed + XP1 + XP2, v2 = seed + XP2, v3 = seed, v4 = seed - XP1;
    while (p + 32 <= end) {
      v1 = xround(v1, rd64(p));
      v2 = xround(v2, rd64(p + 8));
      v3 = xround(v3, rd64(p + 16));
      v4 = xround(v4, rd64(p + 24));
      p += 32;
    }
    h = rotl64(v1, 1) + rotl64(v2, 7) + rotl64(v3, 12) + rotl64(v4, 18);
    h = xmerge(h, v1);
    h = xmerge(h, v2);
    h = xmerge(h, v3);
    h = xmerge(h, v4);
  } else {
    h = seed + XP5;
  }
  h += (uint64_t)len;
  while (p + 8 <= end) {
    h ^= xround(0, rd64(p));
    h = rotl64(h, 27) * XP1 + XP4;
    p += 8;
  }
  if (p + 4 <= end) {
    h ^= (uint64_t)rd32(p) * XP1;
    h = rotl64(h, 23) * XP2 + XP3;
    p += 4;
  }
  while (p < end) {
    h ^= (uint64_t)(*p) * XP5;
    h = rotl64(h, 11) * XP1;
    ++p;
  }
  h ^= h >> 33;
  h *= XP2;
  h ^= h >> 29;
  h *= XP3;
  h ^= h >> 32;
  return h;
}

/* Fingerprint of tokens[start .. start + len): xxHash64 of their little-endian int32 bytes. */
uint64_t oracle_chunk_fingerprint(const int32_t *tokens, i64 start, i64 len, uint64_t seed) {
  uint8_t *buf = (uint8_t *)malloc((size_t)(4 * len + 1));
  for (i64 i = 0; i < len; ++i) {
    uint32_t v = (uint32_t)tokens[start + i];
    for (int b = 0; b < 4; ++b) buf[4 * i + b] = (uint8_t)(v >> (8 * b));
  }
  uint64_t h = oracle_xxh64(buf, 4 * len, seed);
  free(buf);
  return h;
}

/* Gear words from SplitMix64 (Steele, Lea, Flood 2014): G[t] is the (t+1)-th output of the
 * generator seeded with `seed`, i.e. mix(seed + (t + 1) * gamma) with the generator's output
 * mix.  An alternative to a stored Gear table. */
void oracle_splitmix_gear(i64 vocab, uint64_t seed, uint64_t *out) {
  const uint64_t gamma = 0x9e3779b97f4a7c15ull;
  for (i64 t = 0; t < vocab; ++t) {
    uint64_t z = seed + (uint64_t)(t + 1) * gamma;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    out[t] = z ^ (z >> 31);
  }
}
