// Content-addressed chunk registry and chunk-table assembler, host side ("Irminsul论文详解"
// §5: a request's exact prefix is reused in place; each CDC segment of the tail below
// position 32 is prefilled (first-chunk carve-out), a registry hit is reused with
// delta = p - p_src, a miss is prefilled and registered; §6: the S1 fallback looks a missed
// chunk up again as fixed 128-token sub-windows).
//
// The registry maps (xxHash64 fingerprint, length) to the chunk's rows in a ring of pool rows
// and its base position.  A chunk takes the next `len` rows of the ring (skipping to the
// ring's start rather than wrapping a chunk around its end); an entry is stale once the ring
// has moved a full turn past its first row, which is how old chunks are evicted.  Open
// addressing with linear probing; slots are never emptied, only overwritten, and the table is
// rebuilt without stale entries when it fills up.  An entry inserted while assembling a
// request is not a hit for later segments of the same request (its rows are only written by
// that request's own prefill).  One mutex per registry.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/irm.h"

namespace irm {
void set_last_error(const char* msg);
}

namespace {

constexpr int kCarveOut = IRM_CARVE_OUT;
constexpr int kS1Window = 128;

// xxHash64 of a byte string (Y. Collet's XXH64), host side, for the S1 sub-window keys.
constexpr uint64_t H1 = 11400714785074694791ull, H2 = 14029467366897019727ull,
                   H3 = 1609587929392839161ull, H4 = 9650029242287828579ull,
                   H5 = 2870177450012600261ull;
inline uint64_t rl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
inline uint64_t get64(const uint8_t* p) {
  uint64_t v;
  std::memcpy(&v, p, 8);  // little-endian host (x86-64, aarch64)
  return v;
}
inline uint32_t get32(const uint8_t* p) {
  uint32_t v;
  std::memcpy(&v, p, 4);
  return v;
}
inline uint64_t rnd(uint64_t a, uint64_t v) { return rl(a + v * H2, 31) * H1; }

uint64_t xxh64_host(const uint8_t* p, size_t n, uint64_t seed) {
  const uint8_t* const e = p + n;
  uint64_t h;
  if (n >= 32) {
    uint64_t a = seed + H1 + H2, b = seed + H2, c = seed, d = seed - H1;
    for (; p + 32 <= e; p += 32) {
      a = rnd(a, get64(p));
      b = rnd(b, get64(p + 8));
      c = rnd(c, get64(p + 16));
      d = rnd(d, get64(p + 24));
    }
    h = rl(a, 1) + rl(b, 7) + rl(c, 12) + rl(d, 18);
    for (uint64_t v : {a, b, c, d}) h = (h ^ rnd(0, v)) * H1 + H4;
  } else {
    h = seed + H5;
  }
  h += (uint64_t)n;
  for (; p + 8 <= e; p += 8) h = rl(h ^ rnd(0, get64(p)), 27) * H1 + H4;
  if (p + 4 <= e) {
    h = rl(h ^ ((uint64_t)get32(p) * H1), 23) * H2 + H3;
    p += 4;
  }
  for (; p < e; ++p) h = rl(h ^ ((uint64_t)(*p) * H5), 11) * H1;
  h ^= h >> 33;
  h *= H2;
  h ^= h >> 29;
  h *= H3;
  return h ^ (h >> 32);
}

// Fingerprint of tokens[start, start + len): xxHash64 of the little-endian int32 bytes.
uint64_t token_fingerprint(const int32_t* tokens, int64_t start, int64_t len, uint64_t seed) {
  std::vector<uint8_t> b((size_t)(4 * len));
  for (int64_t i = 0; i < len; ++i) {
    const uint32_t v = (uint32_t)tokens[start + i];
    for (int k = 0; k < 4; ++k) b[(size_t)(4 * i + k)] = (uint8_t)(v >> (8 * k));
  }
  return xxh64_host(b.data(), b.size(), seed);
}

}  // namespace

struct irm_registry {
  struct Slot {
    uint64_t hash;
    int32_t len;       // 0: never used
    int32_t base_pos;
    int64_t cursor;    // ring cursor of the chunk's first row
    int64_t call;      // assemble call that inserted it
  };
  int64_t pool_base, pool_rows;
  int64_t cursor = 0;  // rows ever allocated
  int64_t call = 0;
  std::vector<Slot> slots;
  int64_t used = 0;    // slots ever filled since the last rebuild
  std::mutex mu;

  bool live(const Slot& s) const { return s.len > 0 && cursor <= s.cursor + pool_rows; }
  int64_t row(int64_t c) const { return pool_base + c % pool_rows; }
  size_t home(uint64_t h) const { return (size_t)((h * 0x9e3779b97f4a7c15ull) >> 20) & (slots.size() - 1); }

  const Slot* find(uint64_t h, int32_t len) const {
    for (size_t i = home(h), n = 0; n < slots.size(); i = (i + 1) & (slots.size() - 1), ++n) {
      const Slot& s = slots[i];
      if (s.len == 0) return nullptr;
      if (s.hash == h && s.len == len) return &s;
    }
    return nullptr;
  }
  // A live entry of another call, or nullptr.
  const Slot* lookup(uint64_t h, int32_t len) const {
    const Slot* s = find(h, len);
    return (s && live(*s) && s->call != call) ? s : nullptr;
  }
  void rebuild() {
    std::vector<Slot> old;
    old.swap(slots);
    size_t n = old.size();
    int64_t keep = 0;
    for (const Slot& s : old) keep += live(s) ? 1 : 0;
    while ((int64_t)n < 4 * keep) n *= 2;  // at most a quarter full after the rebuild
    slots.assign(n, Slot{0, 0, 0, 0, 0});
    used = 0;
    for (const Slot& s : old)
      if (live(s)) place(s);
  }
  void place(const Slot& e) {
    size_t stale = SIZE_MAX;
    for (size_t i = home(e.hash), n = 0; n < slots.size(); i = (i + 1) & (slots.size() - 1), ++n) {
      Slot& s = slots[i];
      if (s.len == 0) {
        Slot& d = stale != SIZE_MAX ? slots[stale] : s;
        if (&d == &s) ++used;
        d = e;
        return;
      }
      if (s.hash == e.hash && s.len == e.len) {
        s = e;
        return;
      }
      if (stale == SIZE_MAX && !live(s)) stale = i;
    }
    if (stale != SIZE_MAX) slots[stale] = e;
  }
  void insert(uint64_t h, int32_t len, int64_t c, int32_t base_pos) {
    if (4 * (used + 1) > 3 * (int64_t)slots.size()) rebuild();
    place(Slot{h, len, base_pos, c, call});
  }
  // Ring rows for n rows; returns the cursor of the first.
  int64_t alloc(int64_t n) {
    const int64_t pos = cursor % pool_rows;
    if (pos + n > pool_rows) cursor += pool_rows - pos;
    const int64_t c = cursor;
    cursor += n;
    return c;
  }
};

namespace {
irm_status reg_fail(irm_status st, const char* fmt, long long a = 0, long long b = 0) {
  char buf[256];
  std::snprintf(buf, sizeof buf, fmt, a, b);
  irm::set_last_error(buf);
  return st;
}
}  // namespace

extern "C" {

irm_status irm_registry_create(int64_t pool_base, int64_t pool_rows, int64_t capacity, irm_registry** out) {
  if (out == nullptr || pool_base < 0 || pool_rows <= 0 || capacity <= 0)
    return reg_fail(IRM_ERR_INVALID_ARG, "need out, pool_base >= 0, pool_rows > 0 and capacity > 0");
  irm_registry* r = new irm_registry();
  r->pool_base = pool_base;
  r->pool_rows = pool_rows;
  size_t n = 64;
  while ((int64_t)n < 2 * capacity) n *= 2;
  r->slots.assign(n, irm_registry::Slot{0, 0, 0, 0, 0});
  *out = r;
  return IRM_OK;
}

void irm_registry_destroy(irm_registry* reg) { delete reg; }

irm_status irm_registry_stats(irm_registry* reg, int64_t* live_entries, int64_t* rows_allocated) {
  if (reg == nullptr) return reg_fail(IRM_ERR_INVALID_ARG, "null registry");
  std::lock_guard<std::mutex> lk(reg->mu);
  int64_t n = 0;
  for (const auto& s : reg->slots) n += reg->live(s) ? 1 : 0;
  if (live_entries) *live_entries = n;
  if (rows_allocated) *rows_allocated = reg->cursor;
  return IRM_OK;
}

irm_status irm_registry_assemble(irm_registry* reg, const int32_t* tokens_host, int64_t n_tokens,
                                 int64_t prefix_len, int64_t prefix_row, const int32_t* seg_start,
                                 const int32_t* seg_len, const uint64_t* seg_hash, int32_t n_seg,
                                 int32_t flags, uint64_t seed, irm_chunk* chunks_out,
                                 uint8_t* prefill_out, int32_t chunks_cap, int32_t* n_chunks_out) {
  if (reg == nullptr || n_chunks_out == nullptr || chunks_out == nullptr || prefill_out == nullptr)
    return reg_fail(IRM_ERR_INVALID_ARG, "null registry or output");
  if (n_seg < 0 || prefix_len < 0 || (n_seg > 0 && (!seg_start || !seg_len || !seg_hash)))
    return reg_fail(IRM_ERR_INVALID_ARG, "bad segment arguments");
  const bool s1 = (flags & IRM_ASSEMBLE_S1) != 0;
  if (s1 && tokens_host == nullptr) return reg_fail(IRM_ERR_INVALID_ARG, "S1 needs the tokens");
  // segments must tile the tail [prefix_len, n_tokens) in order
  int64_t expect = 0, need = prefix_len > 0 ? 1 : 0;
  for (int32_t i = 0; i < n_seg; ++i) {
    if (seg_start[i] != expect || seg_len[i] <= 0)
      return reg_fail(IRM_ERR_INVALID_ARG, "segment %lld does not start where the previous ended", i);
    if (seg_len[i] > reg->pool_rows)
      return reg_fail(IRM_ERR_INVALID_ARG, "segment %lld is longer than the pool", i);
    expect += seg_len[i];
    need += s1 ? (seg_len[i] + kS1Window - 1) / kS1Window : 1;
  }
  if (prefix_len + expect != n_tokens)
    return reg_fail(IRM_ERR_INVALID_ARG, "prefix and segments cover %lld tokens, not %lld", prefix_len + expect,
                    n_tokens);
  if (prefix_len + expect > INT32_MAX) return reg_fail(IRM_ERR_INVALID_ARG, "context exceeds int32");
  if (need > chunks_cap)
    return reg_fail(IRM_ERR_INVALID_ARG, "the chunk table needs up to %lld entries (capacity %lld)", need, chunks_cap);

  std::lock_guard<std::mutex> lk(reg->mu);
  ++reg->call;
  int32_t k = 0;
  auto emit = [&](int64_t row, int64_t len, int64_t p_src, int64_t p_tgt, int reused, int prefill) {
    irm_chunk& c = chunks_out[k];
    c.pool_offset = row;
    c.len = (int32_t)len;
    c.p_src = (int32_t)p_src;
    c.p_tgt = (int32_t)p_tgt;
    c.reused = (uint8_t)reused;
    c.pad[0] = c.pad[1] = c.pad[2] = 0;
    prefill_out[k] = (uint8_t)prefill;
    ++k;
  };
  if (prefix_len > 0) emit(prefix_row, prefix_len, 0, 0, 0, 0);
  std::vector<const irm_registry::Slot*> hits;
  for (int32_t i = 0; i < n_seg; ++i) {
    const int64_t p = prefix_len + seg_start[i];
    const int64_t len = seg_len[i];
    if (p < kCarveOut) {  // first-chunk carve-out: always prefilled, never registered
      emit(reg->row(reg->alloc(len)), len, p, p, 0, 1);
      continue;
    }
    if (const auto* h = reg->lookup(seg_hash[i], (int32_t)len)) {
      emit(reg->row(h->cursor), len, h->base_pos, p, 1, 0);
      continue;
    }
    // a miss: with S1, look the 128-token windows up again
    const int64_t nw = s1 ? (len + kS1Window - 1) / kS1Window : 1;
    hits.assign((size_t)nw, nullptr);
    std::vector<uint64_t> wh((size_t)nw, 0);
    if (s1) {
      for (int64_t w = 0; w < nw; ++w) {
        const int64_t w0 = w * kS1Window, wl = std::min<int64_t>(kS1Window, len - w0);
        wh[(size_t)w] = token_fingerprint(tokens_host, p + w0, wl, seed);
        hits[(size_t)w] = reg->lookup(wh[(size_t)w], (int32_t)wl);
      }
    }
    const int64_t c = reg->alloc(len);  // rows for the whole segment
    bool any_hit = false;
    for (int64_t w = 0; w < nw;) {
      const int64_t w0 = s1 ? w * kS1Window : 0;
      if (hits[(size_t)w]) {
        const int64_t wl = std::min<int64_t>(kS1Window, len - w0);
        emit(reg->row(hits[(size_t)w]->cursor), wl, hits[(size_t)w]->base_pos, p + w0, 1, 0);
        any_hit = true;
        ++w;
        continue;
      }
      int64_t w1 = w;
      while (w1 < nw && !hits[(size_t)w1]) ++w1;
      const int64_t a1 = s1 ? std::min<int64_t>(w1 * kS1Window, len) : len;
      emit(reg->row(c + w0), a1 - w0, p + w0, p + w0, 0, 1);
      w = w1;
    }
    if (!any_hit) reg->insert(seg_hash[i], (int32_t)len, c, (int32_t)p);
    if (s1) {
      for (int64_t w = 0; w < nw; ++w) {
        if (hits[(size_t)w]) continue;
        const int64_t w0 = w * kS1Window, wl = std::min<int64_t>(kS1Window, len - w0);
        reg->insert(wh[(size_t)w], (int32_t)wl, c + w0, (int32_t)(p + w0));
      }
    }
  }
  *n_chunks_out = k;
  return IRM_OK;
}

}  // extern "C"
