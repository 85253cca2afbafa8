// block_manager.cpp -- host block manager with a hash-chained prefix cache.
//
// Semantics (reference counts, chained block hashes, first-miss lookup capped at
// num_tokens - 1 tokens, LRU eviction among blocks nobody holds, immutable cached blocks)
// are stated with their sources in include/pkv_block_manager.h.  Host code only.
//
// Layout: one record per physical block (count, hash, free-queue links) in a flat vector;
// the free queue is an intrusive doubly linked list over those records with a sentinel at
// index num_blocks, so taking a block out of the middle (a cache hit on a freed block) is
// O(1); the hash table is an unordered_map from the 32-byte hash to the block id.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv_block_manager.h"

extern "C" void pkv_internal_set_error(const char* msg);

namespace {

pkv_status bm_fail(pkv_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pkv_status bm_fail(pkv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  pkv_internal_set_error(buf);
  return s;
}

// ------------------------------------------------------------------ SHA-256 (FIPS 180-4)
//
// The round constants are the first 32 bits of the fractional parts of the cube roots of
// the first 64 primes, the initial hash value those of the square roots of the first 8
// primes (FIPS 180-4, sections 4.2.2 and 5.3.3).  They are derived here from that
// definition with exact integer roots: floor(root(p) * 2^32) is the largest x with
// x^k <= p * 2^(32k), and its low 32 bits are the constant.

using u128 = unsigned __int128;

uint64_t iroot(u128 v, int k) {  // largest x with x^k <= v, for k in {2, 3}
  uint64_t lo = 0, hi = (k == 2) ? (1ull << 40) : (1ull << 36);  // p <= 311 fits below
  while (lo < hi) {
    const uint64_t mid = lo + (hi - lo + 1) / 2;
    u128 p = 1;
    for (int i = 0; i < k; ++i) p *= mid;
    if (p <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Sha256Constants {
  uint32_t k[64];
  uint32_t h0[8];
  Sha256Constants() {
    int primes[64], n = 0;
    for (int c = 2; n < 64; ++c) {
      bool prime = true;
      for (int d = 2; d * d <= c; ++d) if (c % d == 0) { prime = false; break; }
      if (prime) primes[n++] = c;
    }
    for (int i = 0; i < 64; ++i) k[i] = static_cast<uint32_t>(iroot(static_cast<u128>(primes[i]) << 96, 3));
    for (int i = 0; i < 8; ++i) h0[i] = static_cast<uint32_t>(iroot(static_cast<u128>(primes[i]) << 64, 2));
  }
};

const Sha256Constants& sha_constants() {
  static const Sha256Constants c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

class Sha256 {
 public:
  Sha256() : c_(sha_constants()) { std::memcpy(h_, c_.h0, sizeof h_); }

  void update(const void* data, size_t len) {
    const uint8_t* p = static_cast<const uint8_t*>(data);
    total_ += len;
    while (len > 0) {
      const size_t take = (64 - fill_) < len ? (64 - fill_) : len;
      std::memcpy(buf_ + fill_, p, take);
      fill_ += take;
      p += take;
      len -= take;
      if (fill_ == 64) {
        compress(buf_);
        fill_ = 0;
      }
    }
  }

  void finish(uint8_t out[32]) {
    const uint64_t bits = static_cast<uint64_t>(total_) * 8;
    const uint8_t one = 0x80, zero = 0;
    update(&one, 1);
    while (fill_ != 56) update(&zero, 1);
    uint8_t len_be[8];
    for (int i = 0; i < 8; ++i) len_be[i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
    update(len_be, 8);
    for (int i = 0; i < 8; ++i)
      for (int j = 0; j < 4; ++j) out[4 * i + j] = static_cast<uint8_t>(h_[i] >> (24 - 8 * j));
  }

 private:
  void compress(const uint8_t* blk) {
    uint32_t w[64];
    for (int t = 0; t < 16; ++t)
      w[t] = (uint32_t(blk[4 * t]) << 24) | (uint32_t(blk[4 * t + 1]) << 16) | (uint32_t(blk[4 * t + 2]) << 8) |
             uint32_t(blk[4 * t + 3]);
    for (int t = 16; t < 64; ++t) {
      const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
      const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
      w[t] = w[t - 16] + s0 + w[t - 7] + s1;
    }
    uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6], h = h_[7];
    for (int t = 0; t < 64; ++t) {
      const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
      const uint32_t ch = (e & f) ^ (~e & g);
      const uint32_t t1 = h + S1 + ch + c_.k[t] + w[t];
      const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
      const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
      const uint32_t t2 = S0 + maj;
      h = g; g = f; f = e; e = d + t1; d = c; c = b; b = a; a = t1 + t2;
    }
    h_[0] += a; h_[1] += b; h_[2] += c; h_[3] += d; h_[4] += e; h_[5] += f; h_[6] += g; h_[7] += h;
  }

  const Sha256Constants& c_;
  uint32_t h_[8];
  uint8_t buf_[64];
  size_t fill_ = 0;
  size_t total_ = 0;
};

// ------------------------------------------------------------------ block hashes

struct Hash {
  uint8_t b[32];
  bool operator==(const Hash& o) const { return std::memcmp(b, o.b, 32) == 0; }
};

struct HashHasher {
  size_t operator()(const Hash& h) const {
    size_t v;
    std::memcpy(&v, h.b, sizeof v);  // SHA-256 output bits are already uniform
    return v;
  }
};

void put_u32le(Sha256& s, uint32_t v) {
  const uint8_t b[4] = {uint8_t(v), uint8_t(v >> 8), uint8_t(v >> 16), uint8_t(v >> 24)};
  s.update(b, 4);
}

// h = SHA-256(parent || u32le(bs) || bs x i32le(token) || u32le(len(extra)) || extra)
Hash block_hash(const Hash& parent, int32_t bs, const int32_t* toks, const uint8_t* extra, int64_t extra_len) {
  Sha256 s;
  s.update(parent.b, 32);
  put_u32le(s, static_cast<uint32_t>(bs));
  for (int32_t i = 0; i < bs; ++i) put_u32le(s, static_cast<uint32_t>(toks[i]));
  put_u32le(s, static_cast<uint32_t>(extra_len));
  if (extra_len > 0) s.update(extra, static_cast<size_t>(extra_len));
  Hash h;
  s.finish(h.b);
  return h;
}

void chain(const Hash& seed, int32_t bs, const int32_t* tokens, int64_t num_tokens, const uint8_t* salt,
           int64_t salt_len, int64_t max_blocks, std::vector<Hash>* out) {
  const int64_t full = num_tokens / bs;
  const int64_t n = full < max_blocks ? full : max_blocks;
  out->resize(static_cast<size_t>(n));
  Hash parent = seed;
  for (int64_t i = 0; i < n; ++i) {
    parent = block_hash(parent, bs, tokens + i * bs, i == 0 ? salt : nullptr, i == 0 ? salt_len : 0);
    (*out)[static_cast<size_t>(i)] = parent;
  }
}

}  // namespace

// ------------------------------------------------------------------ the manager

struct pkv_block_manager {
  struct Block {
    int32_t ref = 0;
    bool cached = false;
    Hash hash{};
    int32_t prev = -1, next = -1;  // free-queue links (valid while ref == 0)
  };
  int64_t num_blocks = 0;
  int32_t block_size = 16;
  Hash seed{};
  std::vector<Block> blk;  // num_blocks records + the sentinel
  int64_t num_free = 0;
  std::unordered_map<Hash, int32_t, HashHasher> table;

  int32_t sentinel() const { return static_cast<int32_t>(num_blocks); }
  void queue_push_tail(int32_t id) {
    const int32_t s = sentinel(), last = blk[s].prev;
    blk[id].prev = last;
    blk[id].next = s;
    blk[last].next = id;
    blk[s].prev = id;
    ++num_free;
  }
  void queue_remove(int32_t id) {
    blk[blk[id].prev].next = blk[id].next;
    blk[blk[id].next].prev = blk[id].prev;
    blk[id].prev = blk[id].next = -1;
    --num_free;
  }
  bool valid(int32_t id) const { return id >= 0 && id < num_blocks; }
};

extern "C" {

void pkv_sha256(const void* data, int64_t len, uint8_t out[32]) {
  Sha256 s;
  if (len > 0) s.update(data, static_cast<size_t>(len));
  s.finish(out);
}

pkv_status pkv_bm_chain_hashes(const uint8_t seed[32], int32_t block_size, const int32_t* tokens, int64_t num_tokens,
                               const uint8_t* salt, int64_t salt_len, uint8_t* out_hashes) {
  if (!seed || block_size < 1 || num_tokens < 0 || salt_len < 0 || (salt_len > 0 && !salt) ||
      (num_tokens >= block_size && (!tokens || !out_hashes)))
    return bm_fail(PKV_ERR_INVALID_ARG, "chain_hashes: bad arguments");
  Hash s;
  std::memcpy(s.b, seed, 32);
  std::vector<Hash> hs;
  chain(s, block_size, tokens, num_tokens, salt, salt_len, INT64_MAX, &hs);
  for (size_t i = 0; i < hs.size(); ++i) std::memcpy(out_hashes + 32 * i, hs[i].b, 32);
  return PKV_OK;
}

pkv_status pkv_bm_create(int64_t num_blocks, int32_t block_size, const uint8_t* seed, pkv_block_manager** out) {
  if (!out) return bm_fail(PKV_ERR_INVALID_ARG, "create: out is NULL");
  *out = nullptr;
  if (num_blocks < 0 || num_blocks > INT32_MAX - 1)
    return bm_fail(PKV_ERR_INVALID_ARG, "create: num_blocks %lld outside [0, 2^31 - 2]",
                   static_cast<long long>(num_blocks));
  if (block_size < 1) return bm_fail(PKV_ERR_INVALID_ARG, "create: block_size must be >= 1");
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager;
  if (!bm) return bm_fail(PKV_ERR_WORKSPACE, "create: out of host memory");
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  if (seed) std::memcpy(bm->seed.b, seed, 32);
  bm->blk.resize(static_cast<size_t>(num_blocks) + 1);
  const int32_t s = bm->sentinel();
  bm->blk[s].prev = bm->blk[s].next = s;
  for (int32_t i = 0; i < num_blocks; ++i) bm->queue_push_tail(i);
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t n, int32_t* out_blocks) {
  if (!bm || n < 0 || (n > 0 && !out_blocks)) return bm_fail(PKV_ERR_INVALID_ARG, "allocate: bad arguments");
  if (n > bm->num_free)
    return bm_fail(PKV_ERR_WORKSPACE, "allocate: %lld blocks asked, %lld free", static_cast<long long>(n),
                   static_cast<long long>(bm->num_free));
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = bm->blk[bm->sentinel()].next;
    bm->queue_remove(id);
    auto& b = bm->blk[id];
    if (b.cached) {  // evict: the least recently freed cached block
      bm->table.erase(b.hash);
      b.cached = false;
    }
    b.ref = 1;
    out_blocks[i] = id;
  }
  return PKV_OK;
}

pkv_status pkv_bm_get_computed_blocks(pkv_block_manager* bm, const int32_t* tokens, int64_t num_tokens,
                                      const uint8_t* salt, int64_t salt_len, int32_t* out_blocks, int64_t max_out,
                                      int64_t* num_hit) {
  if (!bm || !num_hit || num_tokens < 0 || salt_len < 0 || (salt_len > 0 && !salt) || max_out < 0 ||
      (max_out > 0 && !out_blocks) || (num_tokens > 0 && !tokens))
    return bm_fail(PKV_ERR_INVALID_ARG, "get_computed_blocks: bad arguments");
  *num_hit = 0;
  const int64_t cap_tokens = num_tokens > 0 ? num_tokens - 1 : 0;  // keep one token to compute
  int64_t max_blocks = cap_tokens / bm->block_size;
  if (max_blocks > max_out) max_blocks = max_out;
  std::vector<Hash> hs;
  chain(bm->seed, bm->block_size, tokens, num_tokens, salt, salt_len, max_blocks, &hs);
  int64_t hits = 0;
  for (const Hash& h : hs) {
    auto it = bm->table.find(h);
    if (it == bm->table.end()) break;  // first miss: nothing after it can have been cached
    const int32_t id = it->second;
    auto& b = bm->blk[id];
    if (b.ref == 0) bm->queue_remove(id);
    ++b.ref;
    out_blocks[hits++] = id;
  }
  *num_hit = hits;
  return PKV_OK;
}

pkv_status pkv_bm_cache_full_blocks(pkv_block_manager* bm, const int32_t* tokens, int64_t num_tokens,
                                    const uint8_t* salt, int64_t salt_len, const int32_t* block_table,
                                    int64_t table_len, int64_t* num_cached) {
  if (!bm || num_tokens < 0 || salt_len < 0 || (salt_len > 0 && !salt) || table_len < 0 ||
      (table_len > 0 && !block_table) || (num_tokens > 0 && !tokens))
    return bm_fail(PKV_ERR_INVALID_ARG, "cache_full_blocks: bad arguments");
  int64_t full = num_tokens / bm->block_size;
  if (full > table_len)
    return bm_fail(PKV_ERR_INVALID_ARG, "cache_full_blocks: %lld full blocks but a table of %lld",
                   static_cast<long long>(full), static_cast<long long>(table_len));
  std::vector<Hash> hs;
  chain(bm->seed, bm->block_size, tokens, num_tokens, salt, salt_len, full, &hs);
  for (int64_t i = 0; i < full; ++i) {  // validate everything before changing anything
    const int32_t id = block_table[i];
    if (!bm->valid(id) || bm->blk[id].ref <= 0)
      return bm_fail(PKV_ERR_INVALID_ARG, "cache_full_blocks: block %d is not held", id);
    if (bm->blk[id].cached && !(bm->blk[id].hash == hs[static_cast<size_t>(i)]))
      return bm_fail(PKV_ERR_INVALID_ARG, "cache_full_blocks: block %d already holds another prefix's hash", id);
  }
  int64_t count = 0;
  for (int64_t i = 0; i < full; ++i) {
    const int32_t id = block_table[i];
    auto& b = bm->blk[id];
    const Hash& h = hs[static_cast<size_t>(i)];
    if (!b.cached) {
      auto ins = bm->table.emplace(h, id);
      if (ins.second) {
        b.cached = true;
        b.hash = h;
      }
    }
    count += b.cached ? 1 : 0;
  }
  if (num_cached) *num_cached = count;
  return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, const int32_t* blocks, int64_t n) {
  if (!bm || n < 0 || (n > 0 && !blocks)) return bm_fail(PKV_ERR_INVALID_ARG, "free: bad arguments");
  std::unordered_map<int32_t, int32_t> drops;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t id = blocks[i];
    if (!bm->valid(id)) return bm_fail(PKV_ERR_INVALID_ARG, "free: block id %d outside the pool", id);
    if (++drops[id] > bm->blk[id].ref)
      return bm_fail(PKV_ERR_INVALID_ARG, "free: block %d released more often than held", id);
  }
  for (int64_t i = n - 1; i >= 0; --i) {  // tail first
    const int32_t id = blocks[i];
    if (--bm->blk[id].ref == 0) bm->queue_push_tail(id);
  }
  return PKV_OK;
}

pkv_status pkv_bm_share(pkv_block_manager* bm, const int32_t* blocks, int64_t n) {
  if (!bm || n < 0 || (n > 0 && !blocks)) return bm_fail(PKV_ERR_INVALID_ARG, "share: bad arguments");
  for (int64_t i = 0; i < n; ++i)
    if (!bm->valid(blocks[i]) || bm->blk[blocks[i]].ref <= 0)
      return bm_fail(PKV_ERR_INVALID_ARG, "share: block %d is not held", blocks[i]);
  for (int64_t i = 0; i < n; ++i) ++bm->blk[blocks[i]].ref;
  return PKV_OK;
}

pkv_status pkv_bm_copy_on_write(pkv_block_manager* bm, int32_t block, int32_t* out_block, int32_t* needs_copy) {
  if (!bm || !out_block || !needs_copy) return bm_fail(PKV_ERR_INVALID_ARG, "copy_on_write: bad arguments");
  if (!bm->valid(block) || bm->blk[block].ref <= 0)
    return bm_fail(PKV_ERR_INVALID_ARG, "copy_on_write: block %d is not held", block);
  auto& b = bm->blk[block];
  if (b.ref == 1 && !b.cached) {
    *out_block = block;
    *needs_copy = 0;
    return PKV_OK;
  }
  int32_t fresh = -1;
  pkv_status st = pkv_bm_allocate(bm, 1, &fresh);
  if (st != PKV_OK) return st;
  if (--b.ref == 0) bm->queue_push_tail(block);  // a cached block this writer held alone
  *out_block = fresh;
  *needs_copy = 1;
  return PKV_OK;
}

int64_t pkv_bm_num_free(const pkv_block_manager* bm) { return bm ? bm->num_free : -1; }

int64_t pkv_bm_num_cached(const pkv_block_manager* bm) { return bm ? static_cast<int64_t>(bm->table.size()) : -1; }

int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block) {
  if (!bm || !bm->valid(block)) return -1;
  return bm->blk[block].ref;
}

int32_t pkv_bm_block_hash(const pkv_block_manager* bm, int32_t block, uint8_t* out) {
  if (!bm || !bm->valid(block)) return -1;
  if (!bm->blk[block].cached) return 0;
  if (out) std::memcpy(out, bm->blk[block].hash.b, 32);
  return 1;
}

int32_t pkv_bm_lookup(const pkv_block_manager* bm, const uint8_t hash[32]) {
  if (!bm || !hash) return -1;
  Hash h;
  std::memcpy(h.b, hash, 32);
  auto it = bm->table.find(h);
  return it == bm->table.end() ? -1 : it->second;
}

int64_t pkv_bm_free_queue(const pkv_block_manager* bm, int32_t* out, int64_t max_out) {
  if (!bm || max_out < 0 || (max_out > 0 && !out)) return -1;
  int64_t n = 0;
  for (int32_t id = bm->blk[bm->sentinel()].next; id != bm->sentinel() && n < max_out; id = bm->blk[id].next)
    out[n++] = id;
  return n;
}

}  // extern "C"
