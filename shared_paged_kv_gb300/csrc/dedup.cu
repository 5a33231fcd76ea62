// Block fingerprints and exact deduplication into a shared physical pool.
//
// What is computed: shared-memory KV pool post §3.2 (CalcHash: FNV-1a-style
// over whole 32-bit token ids with offset basis 1469598103934665603 and prime
// 1099511628211, then the tag); INMS walkthrough §2.2 / §3.2 / §5.1 (blocks
// are reused only with equal content, tier and position range, up to the
// first divergence; the tier is part of the fingerprint); TokenDance summary
// section 1 (with explicit segment boundaries the hashing is per segment).
// Two full blocks share a physical block iff they have the same non-PRIVATE
// tier, the same index inside their hashed segment and identical token runs
// from the segment start through the block.  Ids follow first occurrence in
// sequence-major order; refcount = references.
//
// How (GB300, all on device, no host round trip):
//  1. hash: one thread per block slot computes CalcHash of each full block;
//     prep: one warp per sequence finds the segment start of each block
//     (accepted starts by a warp max-scan, then a running maximum over the
//     blocks) and the segment-local chain key with a warp-wide segmented
//     scan of the affine map h -> h*M + fp (restarted at segment starts),
//     finalised with SplitMix64's mixer and folded with the local index.
//  2. insert: every shareable block inserts its key into an open-addressing
//     table; atomicMin keeps the lowest (sequence, block) slot per key.
//  3. resolve: each block takes the table's owner as its representative and
//     verifies it: same tier, same local index, equal block tokens, and the
//     predecessor blocks resolve to the same representative (induction over
//     the segment).  A failure (a key collision) raises a flag.
//  4. fallback (only when flagged): exact brute-force representative search.
//  5. count, tiles, number: first occurrences counted per 1024-slot tile,
//     the counts turned into prefix sums by one CTA, then numbered in slot
//     order (deterministic).
//  6. table: block_table and refcounts.
//  7. (optional) owner of each id, and the references of each id as a CSR.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr uint64_t kFnvOffset = 1469598103934665603ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;
constexpr uint32_t kPrivateTier = 0xFFFFFFFFu;
constexpr uint64_t kChainMul = 0x9E3779B97F4A7C15ull;

struct DedupParams {
  const uint32_t* tokens;
  const int64_t* seq_off;
  const uint32_t* tier;
  const int64_t* seg_off;
  const int32_t* seg_blocks;
  uint64_t* fp_out;
  int32_t* block_table;
  int32_t* refcount;
  int32_t* n_phys;
  int32_t* owner;     // optional [capacity]: sequence of each id's first occurrence
  int64_t* ref_off;   // optional [capacity + 1]: CSR offsets of the references per id
  int32_t* ref_seq;   // optional [n_seq * max_blocks]: referencing sequence per reference
  uint32_t* status;
  // workspace
  unsigned long long* tkeys;
  int32_t* tmin;
  uint64_t* key;      // per slot, 0 = not shareable
  int32_t* rep;       // per slot representative slot (or -1 unused)
  int32_t* segstart;  // per slot
  int32_t* pid;       // per slot physical id of first occurrences
  uint32_t* flags;    // [0] collision
  int32_t* tile_cnt;  // first occurrences per numbering tile
  int32_t* ref_cnt;   // [kRefChunks][min(capacity, slots)] per-chunk reference counts, then starts
  int n_seq, max_blocks, B, capacity, weak;
  uint32_t tmask;
};

__device__ __forceinline__ uint64_t splitmix_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ void seq_geom(const DedupParams& p, int s, int64_t& off, int& nblk, int& full) {
  off = p.seq_off[s];
  const int64_t len = p.seq_off[s + 1] - off;
  int64_t nb = (len + p.B - 1) / p.B;
  int64_t fu = len / p.B;
  if (len < 0) nb = fu = 0;
  if (nb > p.max_blocks) {
    nb = p.max_blocks;
    if (fu > nb) fu = nb;
  }
  nblk = static_cast<int>(nb);
  full = static_cast<int>(fu);
}

// 1a. CalcHash of every full block, one thread per slot
__global__ void dedup_hash(DedupParams p) {
  pdl_enter();
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= p.n_seq * p.max_blocks) return;
  const int s = slot / p.max_blocks, b = slot - s * p.max_blocks;
  int64_t off;
  int nblk, full;
  seq_geom(p, s, off, nblk, full);
  uint64_t fp = 0;
  if (b < full) {
    const uint32_t* t = p.tokens + off + (int64_t)b * p.B;
    uint64_t h = kFnvOffset;
    for (int i = 0; i < p.B; ++i) {
      h ^= (uint64_t)__ldg(t + i);
      h *= kFnvPrime;
    }
    h ^= (uint64_t)(p.tier ? p.tier[s] : 0u);
    h *= kFnvPrime;
    fp = h;
  }
  p.fp_out[slot] = fp;
}

// 1b. one warp per sequence: segment starts and chain keys
// One CTA per sequence; its warps take contiguous 32-block-aligned ranges of
// the block row.  Both scans over the row (the running maximum of the
// segment marks, and the chain x -> A x + C) are associative: pass 1 finds
// each range's aggregate (its largest mark and its composed map; whether a
// block starts a segment is its own mark's business), pass 2 runs every
// range again from the composition of the ranges before it.
constexpr int kPrepMaxWarps = 8;
constexpr int kPrepRange = 128;   // blocks per warp aimed at

__global__ void __launch_bounds__(kPrepMaxWarps * 32) dedup_prep(DedupParams p) {
  pdl_enter();
  __shared__ uint64_t s_aggA[kPrepMaxWarps], s_aggC[kPrepMaxWarps];
  __shared__ int s_aggM[kPrepMaxWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int s = blockIdx.x;
  int64_t off;
  int nblk, full;
  seq_geom(p, s, off, nblk, full);
  if (threadIdx.x == 0) {
    const int64_t len = p.seq_off[s + 1] - off;
    if (len < 0 || (len + p.B - 1) / p.B > p.max_blocks) set_err(p.status, KVS_DEVERR_SEQ_LEN);
  }
  const uint32_t tier = p.tier ? p.tier[s] : 0u;
  const size_t row = (size_t)s * p.max_blocks;
  // without a segment list every block's segment starts at block 0: the marks
  // are all zero and need neither clearing nor reading back below
  const bool segs = p.seg_off != nullptr;
  if (segs) {
    for (int b = threadIdx.x; b < p.max_blocks; b += blockDim.x) p.segstart[row + b] = 0;
    __syncthreads();
    // An entry starts a segment iff it lies inside the sequence and beyond
    // every earlier in-range entry (unsorted and out-of-range starts are
    // ignored); each accepted start marks its own block.
    if (warp == 0) {
      const int64_t e0 = p.seg_off[s], e1 = p.seg_off[s + 1];
      int carry = 0;
      for (int64_t base = e0; base < e1; base += 32) {
        const int64_t e = base + lane;
        const int st = e < e1 ? p.seg_blocks[e] : 0;
        const int v = (e < e1 && st < nblk) ? st : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl = max(incl, y);
        }
        int excl = __shfl_up_sync(0xffffffffu, incl, 1);
        excl = max(carry, lane ? excl : 0);
        if (e < e1 && st < nblk && st > excl) p.segstart[row + st] = st;
        carry = max(carry, __shfl_sync(0xffffffffu, incl, 31));
      }
    }
    __syncthreads();
  }
  // this warp's range [b0, b1)
  const int per = ((p.max_blocks + nw - 1) / nw + 31) / 32 * 32;
  const int b0 = warp * per, b1 = min(p.max_blocks, b0 + per);

  // ---- pass 1 (several warps only): each range's largest mark and composed map
  int scarry = 0;
  uint64_t carryA = 1, carryC = 0;
  if (nw > 1) {
    uint64_t aggA = 1, aggC = 0;
    int aggM = 0;
    for (int base = b0; base < b1; base += 32) {
      const int b = base + lane;
      const bool in = b < b1;
      const uint64_t fp = in ? p.fp_out[row + b] : 0;
      const int mk = (segs && in && b < nblk) ? p.segstart[row + b] : 0;
      // a block starts a segment iff it is block 0 or carries its own mark
      const bool start = b == 0 || mk == b;
      uint64_t A = !in ? 1ull : (b < nblk && !start) ? kChainMul : (b < nblk ? 0ull : 1ull);
      uint64_t Cc = !in ? 0ull : (b < nblk) ? (start ? fp + kChainMul : fp) : 0ull;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t A2 = __shfl_up_sync(0xffffffffu, A, o);
        const uint64_t C2 = __shfl_up_sync(0xffffffffu, Cc, o);
        if (lane >= o) {
          Cc = A * C2 + Cc;
          A = A * A2;
        }
      }
      const uint64_t cA = __shfl_sync(0xffffffffu, A, 31), cC = __shfl_sync(0xffffffffu, Cc, 31);
      aggC = cA * aggC + cC;
      aggA = cA * aggA;
      int m = mk;
#pragma unroll
      for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      aggM = max(aggM, m);
    }
    if (lane == 0) {
      s_aggA[warp] = aggA;
      s_aggC[warp] = aggC;
      s_aggM[warp] = aggM;
    }
    __syncthreads();
    // the composition of the ranges before this one, in order
    for (int w = 0; w < warp; ++w) {
      carryC = s_aggA[w] * carryC + s_aggC[w];
      carryA = s_aggA[w] * carryA;
      scarry = max(scarry, s_aggM[w]);
    }
  }

  // ---- pass 2: the segment start of every block is the running maximum of
  // the marks; the fingerprints and marks of the next two chunks of this
  // range are loaded ahead of use (the chunk written back is always behind
  // the ones read ahead, and no range reads another's marks)
  const int nb1 = min(nblk, b1);
  uint64_t fp_n1 = b0 + lane < b1 ? p.fp_out[row + b0 + lane] : 0;
  uint64_t fp_n2 = b0 + lane + 32 < b1 ? p.fp_out[row + b0 + lane + 32] : 0;
  int st_n1 = (segs && b0 + lane < nb1) ? p.segstart[row + b0 + lane] : 0;
  int st_n2 = (segs && b0 + lane + 32 < nb1) ? p.segstart[row + b0 + lane + 32] : 0;
  for (int base = b0; base < b1; base += 32) {
    const int b = base + lane;
    const uint64_t fp = fp_n1;
    fp_n1 = fp_n2;
    fp_n2 = b + 64 < b1 ? p.fp_out[row + b + 64] : 0;
    int st = (b < nblk) ? st_n1 : 0;
    st_n1 = st_n2;
    st_n2 = (segs && b + 64 < nb1) ? p.segstart[row + b + 64] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, st, o);
      if (lane >= o) st = max(st, y);
    }
    st = max(st, scarry);
    scarry = __shfl_sync(0xffffffffu, st, 31);
    if (b >= nblk) st = 0;
    if (b < b1) p.segstart[row + b] = st;
    const bool shareable = b < full && tier != kPrivateTier;
    // segmented scan of x -> A x + C
    uint64_t A = (b < nblk && b != st) ? kChainMul : (b < nblk ? 0ull : 1ull);
    uint64_t Cc = (b < nblk) ? (b == st ? fp + kChainMul : fp) : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t A2 = __shfl_up_sync(0xffffffffu, A, o);
      const uint64_t C2 = __shfl_up_sync(0xffffffffu, Cc, o);
      if (lane >= o) {
        Cc = A * C2 + Cc;
        A = A * A2;
      }
    }
    const uint64_t gC = A * carryC + Cc;
    const uint64_t gA = A * carryA;
    carryA = __shfl_sync(0xffffffffu, gA, 31);
    carryC = __shfl_sync(0xffffffffu, gC, 31);
    if (b < b1) {
      uint64_t k = 0;
      if (shareable) {
        k = splitmix_mix(gC ^ ((uint64_t)(b - st) * 0xD6E8FEB86659FD93ull) ^ ((uint64_t)tier << 32));
        if (p.weak) k = (k & 63ull) + 1ull;
        if (k == 0) k = 1;
      }
      p.key[row + b] = k;
      p.rep[row + b] = b < nblk ? (int32_t)(row + b) : -1;
    }
  }
}

__device__ __forceinline__ uint32_t table_slot(uint64_t k, uint32_t mask) {
  return static_cast<uint32_t>(splitmix_mix(k ^ 0x5851F42D4C957F2Dull)) & mask;
}

// 2. insert every shareable slot
__global__ void dedup_insert(DedupParams p) {
  pdl_enter();
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= p.n_seq * p.max_blocks) return;
  const uint64_t k = p.key[slot];
  if (!k) return;
  uint32_t i = table_slot(k, p.tmask);
  for (uint32_t probe = 0; probe <= p.tmask; ++probe) {
    const unsigned long long old = atomicCAS(p.tkeys + i, 0ull, (unsigned long long)k);
    if (old == 0ull || old == k) {
      atomicMin(p.tmin + i, slot);
      return;
    }
    i = (i + 1) & p.tmask;
  }
}

__device__ __forceinline__ int table_owner(const DedupParams& p, uint64_t k) {
  uint32_t i = table_slot(k, p.tmask);
  for (uint32_t probe = 0; probe <= p.tmask; ++probe) {
    const unsigned long long v = p.tkeys[i];
    if (v == k) return p.tmin[i];
    if (v == 0ull) return -1;
    i = (i + 1) & p.tmask;
  }
  return -1;
}

__device__ __forceinline__ bool same_block_tokens(const DedupParams& p, int s1, int b1, int s2, int b2) {
  const uint32_t* t1 = p.tokens + p.seq_off[s1] + (int64_t)b1 * p.B;
  const uint32_t* t2 = p.tokens + p.seq_off[s2] + (int64_t)b2 * p.B;
  for (int i = 0; i < p.B; ++i)
    if (t1[i] != t2[i]) return false;
  return true;
}

// 3. resolve and verify representatives
__global__ void dedup_resolve(DedupParams p) {
  pdl_enter();
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= p.n_seq * p.max_blocks) return;
  const uint64_t k = p.key[slot];
  if (!k) return;
  const int r = table_owner(p, k);
  bool ok = r >= 0;
  if (ok && r != slot) {
    const int s = slot / p.max_blocks, b = slot - s * p.max_blocks;
    const int s2 = r / p.max_blocks, b2 = r - s2 * p.max_blocks;
    const uint32_t t1 = p.tier ? p.tier[s] : 0u, t2 = p.tier ? p.tier[s2] : 0u;
    const int st1 = p.segstart[slot], st2 = p.segstart[r];
    ok = p.key[r] != 0 && t1 == t2 && (b - st1) == (b2 - st2) && same_block_tokens(p, s, b, s2, b2);
    if (ok && b > st1) {
      const int r1 = table_owner(p, p.key[slot - 1]);
      const int r2 = table_owner(p, p.key[r - 1]);
      ok = r1 >= 0 && r1 == r2;
    }
  }
  if (ok) {
    p.rep[slot] = r;
  } else {
    atomicOr(p.flags, 1u);
  }
}

// 4. exact brute force, only after a collision was detected
__global__ void dedup_fallback(DedupParams p) {
  pdl_enter();
  if (*(volatile uint32_t*)p.flags == 0u) return;
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= p.n_seq * p.max_blocks) return;
  if (!p.key[slot]) return;
  const int s = slot / p.max_blocks, b = slot - s * p.max_blocks;
  const uint32_t t1 = p.tier ? p.tier[s] : 0u;
  const int st1 = p.segstart[slot];
  const int local = b - st1;
  for (int s2 = 0; s2 <= s; ++s2) {
    if ((p.tier ? p.tier[s2] : 0u) != t1) continue;
    int64_t off2;
    int nblk2, full2;
    seq_geom(p, s2, off2, nblk2, full2);
    const int bend = (s2 == s) ? b : full2;
    for (int b2 = 0; b2 < bend && b2 < full2; ++b2) {
      const int o = s2 * p.max_blocks + b2;
      if (!p.key[o]) continue;
      const int st2 = p.segstart[o];
      if (b2 - st2 != local) continue;
      bool eq = true;
      for (int j = 0; j <= local && eq; ++j) eq = same_block_tokens(p, s, st1 + j, s2, st2 + j);
      if (eq) {
        p.rep[slot] = o;
        return;
      }
    }
  }
  p.rep[slot] = slot;
}

// 5a. first occurrences (slots that are their own representative) per tile
// of 1024 slots
constexpr int kNumTile = 1024;

__device__ __forceinline__ int block_sum_1024(int f, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = __reduce_add_sync(0xffffffffu, f);
  if (lane == 0) warp_sums[warp] = x;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += warp_sums[w];
  return t;
}

__global__ void __launch_bounds__(kNumTile) dedup_count(DedupParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  const int n = p.n_seq * p.max_blocks;
  const int slot = blockIdx.x * kNumTile + threadIdx.x;
  const int f = (slot < n && p.rep[slot] == slot) ? 1 : 0;
  const int t = block_sum_1024(f, warp_sums);
  if (threadIdx.x == 0) p.tile_cnt[blockIdx.x] = t;
}

// 5b. one CTA: the tiles' counts become their exclusive prefix sums (slot
// order), and the total is the number of physical blocks
__global__ void __launch_bounds__(kNumTile) dedup_tiles(DedupParams p, int n_tiles) {
  pdl_enter();
  __shared__ int warp_sums[32];
  int carry = 0;
  for (int base = 0; base < n_tiles; base += kNumTile) {
    const int t = base + threadIdx.x;
    const int c = t < n_tiles ? p.tile_cnt[t] : 0;
    int total;
    const int pos = block_exclusive_scan(c, warp_sums, total);
    if (t < n_tiles) p.tile_cnt[t] = carry + pos;
    carry += total;
  }
  if (threadIdx.x == 0) {
    *p.n_phys = carry;
    if (carry > p.capacity) set_err(p.status, KVS_DEVERR_CAPACITY);
  }
}

// 5c. number the first occurrences in slot order from the tile's offset
__global__ void __launch_bounds__(kNumTile) dedup_number(DedupParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  const int n = p.n_seq * p.max_blocks;
  const int slot = blockIdx.x * kNumTile + threadIdx.x;
  const int f = (slot < n && p.rep[slot] == slot) ? 1 : 0;
  int total;
  const int pos = block_exclusive_scan(f, warp_sums, total);
  if (f) {
    const int id = p.tile_cnt[blockIdx.x] + pos;
    p.pid[slot] = id;
    if (p.owner && id < p.capacity) p.owner[id] = slot / p.max_blocks;
  }
}

// 6. block table + refcounts
__global__ void dedup_table(DedupParams p) {
  pdl_enter();
  const int slot = blockIdx.x * blockDim.x + threadIdx.x;
  if (slot >= p.n_seq * p.max_blocks) return;
  const int r = p.rep[slot];
  if (r < 0) {
    p.block_table[slot] = -1;
    return;
  }
  const int id = p.pid[r];
  p.block_table[slot] = id;
  if (id < p.capacity) atomicAdd(p.refcount + id, 1);
}

// 7. (optional) the references of every physical block: ref_off = exclusive
// prefix sum of the refcounts, and ref_seq[ref_off[id] ..] the sequences of
// the slots that map to id, in ascending slot (sequence, block) order.  One
// CTA of kRefChunks warps: warp k owns a contiguous range of slots and counts
// its references per id; the counts become each warp's first position per id
// (ids in parallel, chunks in order); then every warp walks its range in
// order, ranking equal ids among the 32 lanes of a step by __match_any_sync,
// so the order is deterministic and needs no sort.
constexpr int kRefChunks = 32;

__global__ void __launch_bounds__(kRefChunks * 32) dedup_refs(DedupParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n_seq * p.max_blocks;
  const int cap = p.capacity;
  // every id in use is below min(capacity, slots): a physical block has at
  // least one slot, so the per-chunk counts need only that many columns
  const int ids = min(cap, n);
  const int per = (n + kRefChunks - 1) / kRefChunks;
  const int lo = min(n, warp * per), hi = min(n, lo + per);
  int32_t* cnt = p.ref_cnt + (size_t)warp * ids;
  for (long long i = threadIdx.x; i < (long long)kRefChunks * ids; i += blockDim.x) p.ref_cnt[i] = 0;
  __syncthreads();
  for (int sl = lo + lane; sl < hi; sl += 32) {
    const int id = p.block_table[sl];
    if (id >= 0 && id < ids) atomicAdd(cnt + id, 1);
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < ids; base += blockDim.x) {
    const int id = base + threadIdx.x;
    const int c = id < ids ? p.refcount[id] : 0;
    int total;
    const int pos = block_exclusive_scan(c, warp_sums, total);
    if (id < ids) {
      int run = carry + pos;
      p.ref_off[id] = run;
      for (int k = 0; k < kRefChunks; ++k) {
        int32_t* e = p.ref_cnt + (size_t)k * ids + id;
        const int ck = *e;
        *e = run;
        run += ck;
      }
    }
    carry += total;
  }
  for (int id = ids + threadIdx.x; id <= cap; id += blockDim.x) p.ref_off[id] = carry;   // unused ids, and the end
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int base = lo; base < hi; base += 32) {
    const int sl = base + lane;
    const int id = sl < hi ? p.block_table[sl] : -1;
    const bool ok = id >= 0 && id < ids;
    const unsigned m = __match_any_sync(0xffffffffu, ok ? id : -1);
    const int leader = __ffs(m) - 1;
    const int first = (ok && lane == leader) ? cnt[id] : 0;
    const int at = __shfl_sync(0xffffffffu, first, leader) + __popc(m & lt);
    if (ok) {
      p.ref_seq[at] = sl / p.max_blocks;
      if (lane == leader) cnt[id] = first + __popc(m);
    }
  }
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_fingerprint_dedup(kvs_pool* pool, const uint32_t* tokens_dev, const int64_t* seq_off_dev,
                                            int32_t n_seq, const uint32_t* tier_dev, const int64_t* seg_off_dev,
                                            const int32_t* seg_blocks_dev, uint64_t* fp_out_dev,
                                            int32_t* block_table_dev, int32_t max_blocks, int32_t* refcount_dev,
                                            int32_t* n_phys_dev, int32_t* owner_seq_dev, int64_t* ref_off_dev,
                                            int32_t* ref_seq_dev, uint32_t flags, void* ws, size_t ws_bytes,
                                            cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: null pool");
  if (n_seq < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: bad sizes");
  if (!seq_off_dev || !fp_out_dev || !block_table_dev || !refcount_dev || !n_phys_dev || !ws)
    return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: null pointer");
  if (n_seq > 0 && !tokens_dev) return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: null tokens");
  if ((seg_off_dev == nullptr) != (seg_blocks_dev == nullptr))
    return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: seg_off and seg_blocks go together");
  if ((ref_off_dev == nullptr) != (ref_seq_dev == nullptr))
    return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: ref_off and ref_seq go together");
  if (!aligned16(ws)) return fail(KVS_ERR_INVALID_ARG, "fingerprint_dedup: ws must be 16-byte aligned");
  if ((long long)n_seq * max_blocks > 0x3fffffffll) return fail(KVS_ERR_CAPACITY, "fingerprint_dedup: too many slots");
  size_t need = 0;
  kvs_workspace_size(pool, KVS_OP_DEDUP, n_seq, max_blocks, 0, &need);
  if (ws_bytes < need) return fail(KVS_ERR_CAPACITY, "fingerprint_dedup: workspace too small");
  const size_t slots = (size_t)n_seq * max_blocks;
  size_t T = 1024;
  while (T < 2 * slots) T <<= 1;

  DedupParams p{};
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto take = [&](size_t bytes) {
    uint8_t* r = w;
    w += (bytes + 255) & ~size_t(255);
    return r;
  };
  p.tkeys = reinterpret_cast<unsigned long long*>(take(T * 8));
  p.tmin = reinterpret_cast<int32_t*>(take(T * 4));
  p.key = reinterpret_cast<uint64_t*>(take(slots * 8));
  p.rep = reinterpret_cast<int32_t*>(take(slots * 4));
  p.segstart = reinterpret_cast<int32_t*>(take(slots * 4));
  p.pid = reinterpret_cast<int32_t*>(take(slots * 4));
  p.flags = reinterpret_cast<uint32_t*>(take(16));
  const int n_tiles = static_cast<int>((slots + kNumTile - 1) / kNumTile);
  p.tile_cnt = reinterpret_cast<int32_t*>(take((size_t)n_tiles * 4));
  p.ref_cnt = reinterpret_cast<int32_t*>(take((size_t)kRefChunks * std::min<size_t>(pool->desc.capacity_blocks, slots) * 4));
  p.tokens = tokens_dev;
  p.seq_off = seq_off_dev;
  p.tier = tier_dev;
  p.seg_off = seg_off_dev;
  p.seg_blocks = seg_blocks_dev;
  p.fp_out = fp_out_dev;
  p.block_table = block_table_dev;
  p.refcount = refcount_dev;
  p.n_phys = n_phys_dev;
  p.owner = owner_seq_dev;
  p.ref_off = ref_off_dev;
  p.ref_seq = ref_seq_dev;
  p.status = pool->status;
  p.n_seq = n_seq;
  p.max_blocks = max_blocks;
  p.B = pool->desc.block_tokens;
  p.capacity = pool->desc.capacity_blocks;
  p.weak = (flags & KVS_DEDUP_TEST_WEAK_KEYS) ? 1 : 0;
  p.tmask = static_cast<uint32_t>(T - 1);

  if (cudaMemsetAsync(p.tkeys, 0, T * 8, stream) != cudaSuccess ||
      cudaMemsetAsync(p.tmin, 0x7f, T * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(p.flags, 0, 16, stream) != cudaSuccess ||
      cudaMemsetAsync(refcount_dev, 0, (size_t)pool->desc.capacity_blocks * 4, stream) != cudaSuccess ||
      (owner_seq_dev &&
       cudaMemsetAsync(owner_seq_dev, 0xff, (size_t)pool->desc.capacity_blocks * 4, stream) != cudaSuccess))
    return fail(KVS_ERR_CUDA, "fingerprint_dedup: memset failed");
  if (n_seq == 0) {
    if (cudaMemsetAsync(n_phys_dev, 0, 4, stream) != cudaSuccess ||
        (ref_off_dev &&
         cudaMemsetAsync(ref_off_dev, 0, ((size_t)pool->desc.capacity_blocks + 1) * 8, stream) != cudaSuccess))
      return fail(KVS_ERR_CUDA, "fingerprint_dedup: memset failed");
    return KVS_OK;
  }
  const int n = static_cast<int>(slots);
  const int tb = 256;
  const dim3 gs((n + tb - 1) / tb);
  cudaError_t e = launch_pdl(dedup_hash, gs, dim3(tb), stream, p);
  // dedup_prep: one CTA per sequence, about kPrepRange blocks per warp
  const int prep_warps = std::max(1, std::min(kPrepMaxWarps, (max_blocks + kPrepRange - 1) / kPrepRange));
  if (e == cudaSuccess) e = launch_pdl(dedup_prep, dim3(n_seq), dim3(32 * prep_warps), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_insert, gs, dim3(tb), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_resolve, gs, dim3(tb), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_fallback, gs, dim3(tb), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_count, dim3(n_tiles), dim3(kNumTile), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_tiles, dim3(1), dim3(kNumTile), stream, p, n_tiles);
  if (e == cudaSuccess) e = launch_pdl(dedup_number, dim3(n_tiles), dim3(kNumTile), stream, p);
  if (e == cudaSuccess) e = launch_pdl(dedup_table, gs, dim3(tb), stream, p);
  if (e == cudaSuccess && ref_off_dev) e = launch_pdl(dedup_refs, dim3(1), dim3(kRefChunks * 32), stream, p);
  if (e != cudaSuccess) return fail(KVS_ERR_CUDA, "fingerprint_dedup: launch failed");
  count_launch(ref_off_dev ? 10 : 9);
  return check_launch("fingerprint_dedup");
}
