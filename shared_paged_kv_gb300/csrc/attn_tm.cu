// Paged decode attention, token-major persistent variant (GQA group <= 8).
//
// Computes exactly what attn.cu computes (TokenDance summary section 3 /
// Fig. 8: mirror diffs corrected on chip; INMS walkthrough §3.2: reused K
// rotated by the position shift, V untouched; MemDecay post §4.2: softmax of
// q.k / sqrt(d) weighting V):
//   out[a][h] = sum_t softmax_t(scale * <q, R(delta)(K + DK)>) (V + DV)
//
// GB300 layout of the work:
//  * The 16 tokens of a block are the M dimension of mma.sync m16n8k16 and
//    eight query columns are the N dimension: S^T = K q^T and O^T = V^T P^T.
//    K is the A operand straight from shared memory (ldmatrix), V^T too
//    (ldmatrix.trans); P^T reaches the B operand through movmatrix.  P and a
//    rotated query enter as bf16 hi + lo pairs.
//  * Shared blocks computed once (the INMS walkthrough §6.1 idea of sharing
//    attention work on a common prefix, not only its KV): sequences are taken
//    in groups of R = 8 / G (G = query heads per KV head), so one 8-column MMA
//    tile holds the queries of a whole group.  A per-step plan marks, per
//    group and logical block, whether every member that reaches that block
//    holds the same physical block (no mirror diff, full block).  "Shared
//    items" stream such blocks once for all members; "private items" stream
//    each sequence's remaining blocks with only its own columns live.
//  * Persistent warps take the plan's items in a fixed round-robin order, so
//    a warp knows its next items in advance: the item entry two ahead and the
//    block-table entries of the next item are in flight while the current
//    item computes, and the next item's query rows are prefetched into L1.
//    The whole warp runs the producer logic (lane j holds block j of the
//    item); lane 0 issues a ring of TMA stages that runs ahead across item
//    boundaries.  What the consumer needs about an item reaches it through a
//    small shared-memory ring of claim records.
//  * Each item leaves one (m, l, acc) split per sequence it touched;
//    tm_merge_kernel, queued behind the attention kernel as a programmatic
//    dependent launch, merges them.
//  * Rotation is applied to the query (R(-delta) q) whenever the RoPE segment
//    changes; the diff overlay adds DK / DV tiles through the same MMAs.
//    Calls with rotation use groups of one sequence.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr int kTmWarps = 4;
// Lazy-rescale threshold of the online softmax, in log2 units of P.
constexpr float kTmLazyLog2 = 8.f;
constexpr int kTmMaxIb = 32;
constexpr int kTmRec = 8;   // claim records per warp (more than stages + 1)
constexpr int kPlanMagic = 0x6b76730a;

#ifndef KVS_TM_STAGES_D128
#define KVS_TM_STAGES_D128 2
#endif
#ifndef KVS_TM_MIN_CTAS
#define KVS_TM_MIN_CTAS 3
#endif
#ifndef KVS_TM_ITEMS_PER_WARP
#define KVS_TM_ITEMS_PER_WARP 4
#endif
#ifndef KVS_TM_MAX_SPLITS
#define KVS_TM_MAX_SPLITS 64
#endif

// Ring stages per warp.  A stage holds one block's K and V tiles; a block
// that carries a mirror diff takes two consecutive positions (K/V, then
// DK/DV), so diff blocks need no larger stages.
template <int D>
__host__ __device__ constexpr int tm_stages() {
  return D == 128 ? KVS_TM_STAGES_D128 : 4;
}

template <int D>
__host__ __device__ constexpr int tm_smem_bytes() {
  return 1024 + kTmWarps * tm_stages<D>() * 2 * (16 * D * 2);
}

// ------------------------------------------------------------- plan layout
// Sharing groups.  Without a wide tile, sequences are taken in groups of
// R = 8 / G, so one 8-column token-major tile holds a whole group's queries.
// With a wide tile (head_dim 128, G >= 4, no rotation), groups hold
// W = min(32, 128 / G) sequences whose W * G query rows fill the M = 128 rows
// of a tcgen05 tile (attn_wide.cu); the token-major kernel then takes single
// sequences (R = 1) and only their unshared blocks.  SG is the group size
// either way (1: no groups).
struct TmLayout {
  int R, SG, ib, n_chunks, ibs, n_chunks_s, n_groups;   // private and shared chunk sizes / counts
  bool wide, runs;   // runs: rotation call on the wide tile (shared 8-block segment runs)
  bool compact;      // private items over each member's list of unshared blocks
  size_t max_items, max_witems;
  int max_sub;   // 8-block sub-tiles per wide item
  size_t off_hdr, off_items, off_witems, off_wsub, off_wmem, off_wclaims, off_gmask, off_gphys, off_bdelta, off_bwin, off_pne, off_spm,
      off_plist, off_pcnt, off_p1, off_p2, total;
};

constexpr int kMaxRanges = 256;    // wide-tile claims (split slots) per group, at most

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

#ifndef KVS_RUNS_WIDE_PCT
#define KVS_RUNS_WIDE_PCT 50
#endif
// Rotation calls: the wide tile (latency-bound on its row warps, light on
// DRAM) takes this share of the SMs, and the token-major kernel
// (bandwidth-bound) starts at once on the others and takes all SMs once the
// tile is done.
int runs_wide_ctas(const kvs_pool* pool) { return std::max(1, pool->num_sms * KVS_RUNS_WIDE_PCT / 100); }

// Work-item size (blocks): about KVS_TM_ITEMS_PER_WARP items per resident
// warp, at least max_blocks / (KVS_TM_MAX_SPLITS * split_mult) (bounding the
// splits of one sequence per kind), at most 32 (one block-table entry per lane),
// rounded up to 4, 8 or a multiple of 8.  The work
// estimate counts every sequence's blocks; with groups (R > 1) the blocks a
// group shares become one item for all members, so fewer items result and
// the target is doubled.  With a wide tile the token-major kernel sees only
// unshared blocks, so the work estimate is halved (work_div).  On the 7B
// config (8 x 1024 blocks, 32 KV heads, static round-robin claims) items of
// 8 / 12 / 16 / 24 / 32 blocks measured 169.9 / 168.0 / 167.8 / 166.2 / 179.3 us
// per layer: 24 blocks make 5,440 claims, three nearly full rounds of the
// 1,824 warps, where 16 blocks leave a fifth round for a third of them.
int tm_item_blocks(const kvs_pool* pool, int n_seq, int max_blocks, int R, int split_mult, int work_div) {
  const long long work = (long long)n_seq * pool->desc.num_kv_heads * max_blocks / work_div;
  const long long warps = (long long)pool->num_sms * KVS_TM_MIN_CTAS * kTmWarps;
  long long ib = work / (warps * KVS_TM_ITEMS_PER_WARP * (R > 1 ? 2 : 1));
  const long long max_splits = (long long)KVS_TM_MAX_SPLITS * split_mult;
  const long long min_ib = (max_blocks + max_splits - 1) / max_splits;
  if (ib < min_ib) ib = min_ib;
  if (ib <= 4) return 4;
  if (ib <= 8) return 8;
  return (int)std::min<long long>(kTmMaxIb, (ib + 7) / 8 * 8);
}

bool tm_wide_tile(const kvs_pool* pool, int g, bool rope) {
  (void)rope;
  return pool->desc.head_dim == 128 && g >= 4 && g <= kTmMaxGroup && !pool->tk1.empty();
}

static TmLayout tm_layout(const kvs_pool* pool, int n_seq, int max_blocks, int g, bool rope) {
  TmLayout L{};
  L.wide = tm_wide_tile(pool, g, rope);
  L.runs = L.wide && rope;
  L.R = (rope || L.wide) ? 1 : std::max(1, 8 / g);
  L.SG = L.wide ? std::min(32, 128 / g) : L.R;
  // With a wide tile, shared chunks are whole 8-block sub-tiles of the wide
  // tile (the private chunks keep their own size).
  L.ib = tm_item_blocks(pool, n_seq, max_blocks, L.R, 1, L.wide ? 2 : 1);
  L.n_chunks = (max_blocks + L.ib - 1) / L.ib;
  L.ibs = L.ib;
  if (L.wide) L.ibs = L.runs ? 8 : (std::max(tm_item_blocks(pool, n_seq, max_blocks, 1, 1, 1), 8) + 7) / 8 * 8;
  L.n_chunks_s = (max_blocks + L.ibs - 1) / L.ibs;
  L.n_groups = (n_seq + L.SG - 1) / L.SG;
  const size_t grp = L.SG > 1 ? (size_t)L.n_groups : 0;   // group arrays exist only with grouping
  // a rotation call's items are 8-block runs keyed by physical block: a group
  // can hold up to half its members' runs as items
  L.max_witems = L.wide ? grp * L.n_chunks_s * (L.runs ? std::max(1, L.SG / 2) : 1) : 0;
  if (L.runs) {
    // the shared splits of a rotation call are one per claim range, and a
    // group cuts its runs into at most its share of the wide grid's CTAs
    const int share = std::max(1, runs_wide_ctas(pool) / std::max(1, pool->desc.num_kv_heads * L.n_groups));
    L.n_chunks_s = std::min(std::min(L.n_chunks_s, kMaxRanges), share);
  }
  // Rotation calls: a member's unshared blocks are its private history plus
  // the scattered segment blocks that carry a mirror diff.  Its private items
  // are taken over the list of those blocks (positions k, k + n, k + 2n, ...
  // for item k of n), so that the diff blocks spread over all its items.
  L.compact = L.runs;
#ifndef KVS_COMPACT_IB
#define KVS_COMPACT_IB 24
#endif
  // Compact items take a fixed size: their lists hold unshared blocks only,
  // so the split bound above does not apply.  On the all-gather round (about
  // three claims per warp) items of 8 / 12 / 16 / 24 / 32 blocks measured
  // 266 / 254 / 242 / 239 / 240 us per layer: below 24 the per-item costs
  // (query load, split, merge slot) win, above it the last claims' tail.
  if (L.compact) {
    L.ib = KVS_COMPACT_IB;
    L.n_chunks = (max_blocks + L.ib - 1) / L.ib;
  }
  L.max_items = (L.wide ? 0 : grp * L.n_chunks_s) + (size_t)n_seq * L.n_chunks;
  L.max_sub = (L.ibs + 7) / 8;
  const size_t per_split = (size_t)n_seq * pool->desc.num_kv_heads * g * (pool->desc.head_dim + 2) * sizeof(float);
  const size_t split_bytes = per_split * L.n_chunks, split_bytes_s = per_split * L.n_chunks_s;
  size_t o = 0;
  L.off_hdr = o; o = align256(o + 64);
  L.off_items = o; o = align256(o + L.max_items * sizeof(int4));
  L.off_witems = o; o = align256(o + L.max_witems * sizeof(int4));
  L.off_wsub = o; o = align256(o + L.max_witems * L.max_sub * 8 * sizeof(int2));
  L.off_wmem = o; o = align256(o + (L.runs ? L.max_witems * 32 * sizeof(int2) : 0));
  L.off_wclaims = o; o = align256(o + (L.runs ? L.max_witems * sizeof(int4) : 0));
  L.off_gmask = o; o = align256(o + grp * max_blocks * sizeof(uint32_t));
  L.off_gphys = o; o = align256(o + grp * max_blocks * sizeof(int32_t));
  L.off_bdelta = o; o = align256(o + (rope ? (size_t)n_seq * max_blocks * sizeof(int32_t) : 0));
  L.off_bwin = o; o = align256(o + (rope ? (size_t)n_seq * max_blocks * sizeof(int32_t) : 0));
  L.off_pne = o; o = align256(o + (size_t)n_seq * L.n_chunks);
  L.off_spm = o; o = align256(o + grp * L.n_chunks_s * sizeof(uint32_t));
  L.off_plist = o; o = align256(o + (L.compact ? (size_t)n_seq * max_blocks * sizeof(int32_t) : 0));
  L.off_pcnt = o; o = align256(o + (L.compact ? (size_t)n_seq * sizeof(int32_t) : 0));
  L.off_p1 = o; o = align256(o + split_bytes);
  L.off_p2 = o; o = align256(o + (L.SG > 1 ? split_bytes_s : 0));
  L.total = o;
  return L;
}

size_t tm_workspace_bytes(const kvs_pool* pool, int n_seq, int max_blocks, int g) {
  return std::max(tm_layout(pool, n_seq, max_blocks, g, false).total,
                  tm_layout(pool, n_seq, max_blocks, g, true).total) + 256;
}

// ------------------------------------------------------------------- plan
// Items are int4 {x: kind (bit 30) | group or sequence, y: chunk, z: end
// block (exclusive), w: member mask of the columns that take part}.  With a
// wide tile the shared items form their own list (witems), taken by the
// tcgen05 kernel; the token-major list then holds private items only.
//
// Header: [0] token-major items, [1] magic, [2] n_seq, [3] max_blocks, [4] R,
// [5] ib, [6] hkv, [7] SG, [8] wide items, [9] ibs, [10] wide claims (rotation
// calls: ranges of run items), [11] compact private items.
struct PlanParams {
  const int32_t* block_table;
  const int32_t* seq_len;
  const int32_t* diff_table;
  int* hdr;
  int4* items;
  int4* witems;      // wide shared items (wide tile only)
  int2* wsub;        // per wide item and 8-block sub-tile: {members, physical block} of each block
  int2* wmem;        // rotation calls: per wide item and member, {split slot, RoPE shift}
  int4* wclaims;     // rotation calls: claims {group, first item, items | slot << 16, members}
  uint32_t* gmask;   // [n_groups][max_blocks] members computed by the group's shared item (SG > 1)
  int32_t* gphys;    // [n_groups][max_blocks] that shared physical block, or -1 (SG > 1)
  uint8_t* pne;      // [n_seq][n_chunks] private chunk has unshared work
  uint32_t* spm;     // [n_groups][n_chunks_s] members taking part in the shared chunk (SG > 1)
  const int32_t* rope_off;   // rotation calls: segment CSR
  const int4* rope_segs;
  int32_t* bdelta;   // [n_seq][max_blocks] RoPE shift of each logical block (rotation calls)
  int32_t* bwin;     // [n_seq][max_blocks] the last entry covering each block (from the sequence's first), or -1
  uint32_t* status;
  float* p1_ml;      // (m, l) of the private splits [n_seq][hkv][g][n_chunks]
  float* p2_ml;      // (m, l) of the shared splits [n_seq][hkv][g][n_chunks_s] (SG > 1)
  int n_seq, max_blocks, R, SG, G, ib, n_chunks, ibs, n_chunks_s, n_groups, capacity, hkv, wide, max_sub, runs;
  int max_witems;
  int wide_ctas;     // CTAs of the wide tile's grid (rotation calls size their claims to it)
  int32_t* plist;    // compact items: [n_seq][max_blocks] each member's unshared logical blocks, in order
  int32_t* pcnt;     // compact items: [n_seq] length of that list
  int compact;
};

__device__ __forceinline__ int plan_seq_blocks(const int32_t* seq_len, int a, int max_blocks) {
  int L = seq_len[a];
  if (L < 0) L = 0;
  if (L > max_blocks * 16) L = max_blocks * 16;
  return (L + 15) / 16;
}

// Plan, part 1 (it depends on the tables only, so one plan serves every
// layer of a decode step).  One CTA per group of SG sequences:
//  * gmask / gphys: at each logical block, the members eligible to share it
//    (a valid full physical block, no mirror diff) are grouped by physical
//    block; the largest such set (the earliest member's on a tie) shares the
//    block when it has at least two members.  The others take the block in
//    their private items;
//  * pne / spm: which private chunks have unshared work, which members take
//    part in each shared chunk;
//  * the (m, l) of every split that will not be written is set to (-inf, 0),
//    so the merge can read all of them without consulting pne / spm first;
//  * rotation calls: bdelta, the shift of the segment covering each logical
//    block (the last entry covering it; 0 outside every entry).
// Rotation calls on the wide tile: the group's shared work is keyed by
// physical block instead of logical position.  A "run" is 8 logical blocks of
// one member, inside one RoPE segment (one shift, the covering entry of every
// block), full, without mirror diffs, holding 8 consecutive physical blocks;
// runs of different members with the same first physical block hold the same
// K and V and differ only in the shift, which the tile applies to each
// member's query.  A block of a run that carries a mirror diff for a member
// is left to that member's private items (the rest of the run is shared).
// Runs found by at least two members become wide items; a member's other
// blocks stay private.  All threads of the CTA call this.
constexpr int kRunCap = 2048;

__device__ void plan_runs(const PlanParams& pp, int gi, int a0, int nm, unsigned long long* s_key, int* s_dl,
                          uint8_t* s_ex, int* s_n) {
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) *s_n = 0;
  for (int b = tid; b < pp.max_blocks; b += nt) pp.gmask[(size_t)gi * pp.max_blocks + b] = 0u;
  for (int c = tid; c < pp.n_chunks_s; c += nt) pp.spm[(size_t)gi * pp.n_chunks_s + c] = 0u;
  __syncthreads();
  // candidates {first physical block, member, first logical block; shift;
  // blocks with a mirror diff}.  The group's entries are contiguous in the
  // CSR: threads take them in turn and find their member.
  const int eg0 = pp.rope_off[a0], eg1 = pp.rope_off[a0 + nm];
  for (int e = eg0 + tid; e < eg1; e += nt) {
    int r = 0;
    while (r + 1 < nm && pp.rope_off[a0 + r + 1] <= e) ++r;
    const int a = a0 + r, e0 = pp.rope_off[a];
    const int L = min(max(pp.seq_len[a], 0), pp.max_blocks * 16);
    const int4 sg = __ldg(pp.rope_segs + e);
    if (sg.z <= -(1 << 18) || sg.z >= (1 << 18) || sg.x < 0) continue;
    const int* row = pp.block_table + (size_t)a * pp.max_blocks;
    const size_t rb = (size_t)a * pp.max_blocks;
    for (int b = sg.x; b + 8 <= sg.x + sg.y && b + 8 <= pp.max_blocks && (b + 8) * 16 <= L; b += 8) {
      // the 8 blocks hold consecutive physical blocks, this entry is the
      // last one covering each of them (so that a logical block belongs to
      // one run at most), and their shift is the entry's; all loads at once
      int ph[8], wn[8], dl[8], df[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ph[k] = row[b + k];
        wn[k] = pp.bwin[rb + b + k];
        dl[k] = pp.bdelta[rb + b + k];
        df[k] = pp.diff_table ? pp.diff_table[rb + b + k] : -1;
      }
      bool ok = ph[0] >= 0 && ph[0] <= pp.capacity - 8;
      uint32_t ex = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ok = ok && ph[k] == ph[0] + k && wn[k] == e - e0 && dl[k] == sg.z;
        ex |= (df[k] >= 0 ? 1u : 0u) << k;
      }
      if (!ok || ex == 0xffu) continue;
      const int idx = atomicAdd(s_n, 1);
      if (idx < kRunCap) s_key[idx] = ((unsigned long long)(unsigned)ph[0] << 32) | ((unsigned long long)r << 20) | (unsigned)b;
    }
  }
  __syncthreads();
  const int n = min(*s_n, kRunCap);
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + tid; i < P; i += nt) s_key[i] = ~0ull;
  __syncthreads();
  // bitonic sort by (physical block, member, logical block): deterministic
  for (int k = 2; k <= P; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += nt) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const unsigned long long x = s_key[i], y = s_key[ixj];
          if ((x > y) == up) {
            s_key[i] = y;
            s_key[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  // the shift and the diff blocks of each sorted candidate (the run check
  // found the shift of all 8 blocks equal to the entry's)
  for (int i = tid; i < n; i += nt) {
    const int r = (int)((s_key[i] >> 20) & 31u), b = (int)(s_key[i] & 0xFFFFFu);
    const size_t rb = (size_t)(a0 + r) * pp.max_blocks + b;
    uint32_t ex = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) ex |= ((pp.diff_table && pp.diff_table[rb + k] >= 0) ? 1u : 0u) << k;
    s_dl[i] = pp.bdelta[rb];
    s_ex[i] = (uint8_t)ex;
  }
  __syncthreads();
  // one item per physical run held by two or more members (a member's first
  // run with that block, by logical position).  Each thread takes a
  // contiguous range of the sorted candidates, so the group's items get
  // consecutive indices in key order.
  const int per = (n + nt - 1) / nt, i0 = min(n, tid * per), i1 = min(n, i0 + per);
  auto is_item = [&](int i, uint32_t& mask, int& j) {
    const unsigned key = (unsigned)(s_key[i] >> 32);
    if (i > 0 && (unsigned)(s_key[i - 1] >> 32) == key) return false;
    mask = 0;
    int cnt = 0;
    for (j = i; j < n && (unsigned)(s_key[j] >> 32) == key; ++j) {
      const int r = (int)((s_key[j] >> 20) & 31u);
      if (!((mask >> r) & 1u)) {
        mask |= 1u << r;
        ++cnt;
      }
    }
    return cnt >= 2;
  };
  int mine = 0;
  for (int i = i0; i < i1; ++i) {
    uint32_t mask;
    int j;
    mine += is_item(i, mask, j) ? 1 : 0;
  }
  __shared__ int warp_sums[32];
  __shared__ int s_base, s_rbase, s_created, s_rg;
  __shared__ uint32_t s_rmask[kMaxRanges];
  int total;
  const int off = block_exclusive_scan(mine, warp_sums, total);
  if (tid == 0) {
    const int base = total ? atomicAdd(pp.hdr + 8, total) : 0;
    const int created = max(0, min(total, pp.max_witems - base));   // beyond the capacity: stays private
    // claims of the wide tile: ranges of consecutive items (one split per
    // member and range).  Every group's runs cost the same per item, so each
    // group takes an equal share of the wide grid's CTAs per KV head and
    // cuts its items into that many ranges: one claim per CTA, the fewest
    // items per CTA, one split per member and range.  At most
    // min(n_chunks_s, kMaxRanges) ranges (the split slots).
    const int share = max(1, pp.wide_ctas / max(1, pp.hkv * pp.n_groups));
    const int max_r = min(min(pp.n_chunks_s, kMaxRanges), share);
    const int rg = max(1, (created + max_r - 1) / max_r);
    const int n_r = (created + rg - 1) / rg;
    s_base = base;
    s_created = created;
    s_rg = rg;
    s_rbase = n_r ? atomicAdd(pp.hdr + 10, n_r) : 0;
  }
  for (int q = tid; q < kMaxRanges; q += nt) s_rmask[q] = 0u;
  __syncthreads();
  int k = off;
  for (int i = i0; i < i1; ++i) {
    uint32_t mask;
    int j;
    if (!is_item(i, mask, j)) continue;
    const int kk = k++;
    if (kk >= s_created) continue;
    const int wi = s_base + kk, q_r = kk / s_rg;
    const unsigned key = (unsigned)(s_key[i] >> 32);
    pp.witems[wi] = make_int4((1 << 30) | gi, 0, 8, (int)mask);
    for (int r = 0; r < 32; ++r) pp.wmem[(size_t)wi * 32 + r] = make_int2(q_r, 0);
    uint32_t seen = 0, bm[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // members taking each block
    for (int q = i; q < j; ++q) {
      const int r = (int)((s_key[q] >> 20) & 31u), b = (int)(s_key[q] & 0xFFFFFu);
      if ((seen >> r) & 1u) continue;
      seen |= 1u << r;
      pp.wmem[(size_t)wi * 32 + r] = make_int2(q_r, s_dl[q]);
      for (int kb = 0; kb < 8; ++kb) {
        if ((s_ex[q] >> kb) & 1u) continue;   // diff block: private for this member
        bm[kb] |= 1u << r;
        atomicOr(pp.gmask + (size_t)gi * pp.max_blocks + b + kb, 1u << r);
      }
    }
    for (int kb = 0; kb < 8; ++kb) pp.wsub[(size_t)wi * 8 + kb] = make_int2((int)bm[kb], (int)key + kb);
    atomicOr(&s_rmask[q_r], mask);
  }
  __syncthreads();
  const int n_r = (s_created + s_rg - 1) / s_rg;
  for (int q = tid; q < n_r; q += nt) {
    const int first = q * s_rg, cnt = min(s_rg, s_created - first);
    if (s_rbase + q < pp.max_witems)
      pp.wclaims[s_rbase + q] = make_int4(gi, s_base + first, cnt | (q << 16), (int)s_rmask[q]);
    pp.spm[(size_t)gi * pp.n_chunks_s + q] = s_rmask[q];
  }
}

// Plan, part 0 (rotation calls): the shift of every logical block, one CTA
// per sequence.  The last entry covering a block wins (entries in order), so
// every entry marks its blocks with an atomic maximum of its index; a block
// no entry covers keeps shift 0.  bwin keeps the winning index for the run
// search (a run must lie in the last entry covering each of its blocks).
__global__ void __launch_bounds__(256) tm_plan_shifts(PlanParams pp) {
  pdl_enter();
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int a = blockIdx.x; a < pp.n_seq; a += gridDim.x) {
    int32_t* win = pp.bwin + (size_t)a * pp.max_blocks;
    for (int b = tid; b < pp.max_blocks; b += nt) win[b] = -1;
    __syncthreads();
    const int e0 = pp.rope_off[a], e1 = pp.rope_off[a + 1];
    for (int e = e0 + tid; e < e1; e += nt) {
      const int4 sg = __ldg(pp.rope_segs + e);
      const int lo = max(sg.x, 0), hi = (int)min((long long)sg.x + sg.y, (long long)pp.max_blocks);
      for (int b = lo; b < hi; ++b) atomicMax(win + b, e - e0);
    }
    __syncthreads();
    for (int b = tid; b < pp.max_blocks; b += nt) {
      const int w = win[b];
      int dl = w >= 0 ? __ldg(pp.rope_segs + e0 + w).z : 0;
      if (dl <= -(1 << 18) || dl >= (1 << 18)) {
        set_err(pp.status, KVS_DEVERR_ROPE_RANGE);
        dl = 0;
      }
      pp.bdelta[(size_t)a * pp.max_blocks + b] = dl;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(512) tm_plan_groups(PlanParams pp) {
  pdl_enter();
  __shared__ unsigned long long s_key[kRunCap];
  __shared__ int s_dl[kRunCap];
  __shared__ uint8_t s_ex[kRunCap];
  __shared__ int s_n;
  const int tid = threadIdx.x, nt = blockDim.x;
  if (blockIdx.x == 0 && tid == 0) {
    pp.hdr[0] = 0;   // item counts, accumulated by tm_plan_items (and, for runs, here)
    pp.hdr[1] = kPlanMagic;
    pp.hdr[2] = pp.n_seq;
    pp.hdr[3] = pp.max_blocks;
    pp.hdr[4] = pp.R;
    pp.hdr[5] = pp.ib;
    pp.hdr[6] = pp.hkv;
    pp.hdr[7] = pp.SG;
    pp.hdr[9] = pp.ibs;
    pp.hdr[11] = pp.compact;
  }
  const float2 none = make_float2(-INFINITY, 0.f);
  const int SG = pp.SG;
  for (int gi = blockIdx.x; gi < pp.n_groups; gi += gridDim.x) {
    const int a0 = gi * SG, nm = min(SG, pp.n_seq - a0);
    // (rotation calls: bdelta and bwin come from tm_plan_shifts)
    // 1. sharing
    if (SG > 1 && pp.runs) {
      plan_runs(pp, gi, a0, nm, s_key, s_dl, s_ex, &s_n);
      __syncthreads();
    } else if (SG > 1) {
      for (int b = tid; b < pp.max_blocks; b += nt) {
        int ph[32];
        for (int r = 0; r < nm; ++r) {
          const int a = a0 + r;
          const int L = min(max(pp.seq_len[a], 0), pp.max_blocks * 16);
          const int e = pp.block_table[(size_t)a * pp.max_blocks + b];
          const bool full = (b + 1) * 16 <= L;
          const int d = pp.diff_table ? pp.diff_table[(size_t)a * pp.max_blocks + b] : -1;
          ph[r] = (full && d < 0 && e >= 0 && e < pp.capacity) ? e : -1;
        }
        // the first member of the largest set of equal physical blocks
        int best = -1, bestc = 1;
        for (int r = 0; r < nm; ++r) {
          if (ph[r] < 0) continue;
          int cnt = 0;
          for (int r2 = r; r2 < nm; ++r2) cnt += ph[r2] == ph[r];
          if (cnt > bestc) {
            bestc = cnt;
            best = ph[r];
          }
        }
        uint32_t mask = 0;
        if (best >= 0)
          for (int r = 0; r < nm; ++r) mask |= (ph[r] == best ? 1u : 0u) << r;
        pp.gmask[(size_t)gi * pp.max_blocks + b] = mask;
        pp.gphys[(size_t)gi * pp.max_blocks + b] = best;
      }
      __syncthreads();
    }
    // 2. chunk occupancy (compact items: the list of unshared blocks first)
    if (pp.compact) {
      // one warp per member: its unshared blocks in order, by ballots
      const int wid = tid >> 5, ln = tid & 31, nw = nt >> 5;
      for (int r = wid; r < nm; r += nw) {
        const int a = a0 + r;
        const int nb = plan_seq_blocks(pp.seq_len, a, pp.max_blocks);
        int cnt = 0;
        for (int b0 = 0; b0 < nb; b0 += 32) {
          const int b = b0 + ln;
          const bool keep = b < nb && !((pp.gmask[(size_t)gi * pp.max_blocks + b] >> r) & 1u);
          const unsigned bal = __ballot_sync(0xffffffffu, keep);
          if (keep) pp.plist[(size_t)a * pp.max_blocks + cnt + __popc(bal & ((1u << ln) - 1u))] = b;
          cnt += __popc(bal);
        }
        const int ni = (cnt + pp.ib - 1) / pp.ib;
        if (ln == 0) pp.pcnt[a] = cnt;
        for (int c = ln; c < pp.n_chunks; c += 32) pp.pne[(size_t)a * pp.n_chunks + c] = (uint8_t)(c < ni);
      }
    } else
    for (int i = tid; i < nm * pp.n_chunks; i += nt) {
      const int r = i / pp.n_chunks, c = i - r * pp.n_chunks, a = a0 + r;
      const int nb = plan_seq_blocks(pp.seq_len, a, pp.max_blocks);
      int any_priv = 0;
      for (int b = c * pp.ib; b < min((c + 1) * pp.ib, nb); ++b)
        any_priv |= SG > 1 ? !((pp.gmask[(size_t)gi * pp.max_blocks + b] >> r) & 1u) : 1;
      pp.pne[(size_t)a * pp.n_chunks + c] = (uint8_t)any_priv;
    }
    if (SG > 1 && !pp.runs) {
      for (int c = tid; c < pp.n_chunks_s; c += nt) {
        uint32_t m = 0;
        for (int b = c * pp.ibs; b < min((c + 1) * pp.ibs, pp.max_blocks); ++b)
          m |= pp.gmask[(size_t)gi * pp.max_blocks + b];
        pp.spm[(size_t)gi * pp.n_chunks_s + c] = m;
      }
    }
    __syncthreads();
    // 3. splits that no item writes (their (m, l) at [a][h][hh][c]): one
    // (member, chunk) per thread, its flag read once
    for (int i = tid; i < nm * pp.n_chunks; i += nt) {
      const int r = i / pp.n_chunks, c = i - r * pp.n_chunks, a = a0 + r;
      if (pp.pne[(size_t)a * pp.n_chunks + c]) continue;
      float2* ml = reinterpret_cast<float2*>(pp.p1_ml) + (size_t)a * pp.hkv * pp.n_chunks * pp.G;
      for (int h = 0; h < pp.hkv; ++h)
        for (int hh = 0; hh < pp.G; ++hh) ml[((size_t)h * pp.G + hh) * pp.n_chunks + c] = none;
    }
    if (SG > 1) {
      for (int i = tid; i < nm * pp.n_chunks_s; i += nt) {
        const int r = i / pp.n_chunks_s, c = i - r * pp.n_chunks_s, a = a0 + r;
        if ((pp.spm[(size_t)gi * pp.n_chunks_s + c] >> r) & 1u) continue;
        float2* ml = reinterpret_cast<float2*>(pp.p2_ml) + (size_t)a * pp.hkv * pp.n_chunks_s * pp.G;
        for (int h = 0; h < pp.hkv; ++h)
          for (int hh = 0; hh < pp.G; ++hh) ml[((size_t)h * pp.G + hh) * pp.n_chunks_s + c] = none;
      }
    }
    __syncthreads();
  }
}

// Plan, part 2: the compact item lists, shared items (group, chunk) then
// private items (sequence, chunk), chunk-major.  Each CTA compacts a run of
// slots and reserves its place with one atomic add per list, so a list is
// chunk-major up to the interleaving of CTAs; results do not depend on the
// order (every split has a fixed slot and a fixed merge order).
__global__ void __launch_bounds__(256) tm_plan_items(PlanParams pp) {
  pdl_enter();
  __shared__ int warp_sums[32];
  __shared__ int s_base, s_wbase;
  const int n_sh = (pp.SG > 1 && !pp.runs) ? pp.n_groups * pp.n_chunks_s : 0, n_pr = pp.n_seq * pp.n_chunks;
  const int total = n_sh + n_pr;
  for (int base = blockIdx.x * blockDim.x; base < total; base += gridDim.x * blockDim.x) {
    const int i = base + threadIdx.x;
    int keep = 0, keep_w = 0;
    int4 item = make_int4(0, 0, 0, 0);
    if (i < n_sh) {
      const int c = i / pp.n_groups, gi = i - c * pp.n_groups;
      const uint32_t m = pp.spm[(size_t)gi * pp.n_chunks_s + c];
      if (m != 0) {
        int nb = 0;
        for (int r = 0; r < pp.SG && gi * pp.SG + r < pp.n_seq; ++r)
          nb = max(nb, plan_seq_blocks(pp.seq_len, gi * pp.SG + r, pp.max_blocks));
        item = make_int4((1 << 30) | gi, c, min((c + 1) * pp.ibs, nb), (int)m);
        if (pp.wide) keep_w = 1; else keep = 1;
      }
    } else if (i < total) {
      const int j = i - n_sh;
      const int c = j / pp.n_seq, a = j - c * pp.n_seq;
      keep = pp.pne[(size_t)a * pp.n_chunks + c];
      // z: the end block, or (compact items) the length of the member's list
      if (keep)
        item = make_int4(a, c, pp.compact ? pp.pcnt[a] : min((c + 1) * pp.ib, plan_seq_blocks(pp.seq_len, a, pp.max_blocks)),
                         1 << (a % pp.R));
    }
    int cnt, cnt_w = 0, pos_w = 0;
    const int pos = block_exclusive_scan(keep, warp_sums, cnt);
    if (pp.wide) pos_w = block_exclusive_scan(keep_w, warp_sums, cnt_w);
    if (threadIdx.x == 0) {
      s_base = cnt ? atomicAdd(pp.hdr, cnt) : 0;
      s_wbase = cnt_w ? atomicAdd(pp.hdr + 8, cnt_w) : 0;
    }
    __syncthreads();
    if (keep) pp.items[s_base + pos] = item;
    if (keep_w) {
      // the item's blocks as one record per 8-block sub-tile, so the tile
      // kernel reads a sub-tile's members and physical blocks in one load
      const int wi = s_wbase + pos_w, gi = item.x & ((1 << 30) - 1), b0 = item.y * pp.ibs;
      pp.witems[wi] = item;
      for (int e = 0; e < pp.max_sub * 8; ++e) {
        const int b = b0 + e;
        int2 v = make_int2(0, -1);
        if (b < item.z && e < pp.ibs)
          v = make_int2((int)pp.gmask[(size_t)gi * pp.max_blocks + b], pp.gphys[(size_t)gi * pp.max_blocks + b]);
        pp.wsub[(size_t)wi * pp.max_sub * 8 + e] = v;
      }
    }
    __syncthreads();
  }
}

// -------------------------------------------------------------- attention
struct TmParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_len;
  const int32_t* diff_table;
  const int32_t* bdelta;   // RoPE shift per logical block (rotation calls)
  float* out;
  float* p1;          // private splits [n_seq][hkv][n_chunks][g][D]
  float* p1_ml;       // [n_seq][hkv][g][n_chunks][2]: a row's (m, l) are contiguous
  float* p2;          // shared splits, same shape
  float* p2_ml;
  const int* hdr;
  const int4* items;
  const uint32_t* gmask;
  const int32_t* gphys;
  const int32_t* plist;   // compact items: each member's unshared logical blocks
  uint32_t* status;
  int compact;            // private items over plist (rotation calls on the wide tile)
  int max_blocks, n_seq, hkv, g, hq, ib, n_chunks, ibs, n_chunks_s, R, SG, capacity, diff_capacity;
  int mwpr;           // merge warps per output row
  // the merge prefetches every split slot's data into L2 before its wait:
  // worth it when its CTAs become resident long before the attention grid
  // completes (no wide tile beside it: on the 7B layer 161.8-162.1 us against
  // 164.9-165.1 us per layer), not behind the wide tile, where they start
  // about 1 us before the end and the lines of slots without a split would
  // only compete with the reads (GQA fan-out 21.2 against 20.7 us)
  int merge_prefetch;
  // the merge lets the next kernel on the stream be scheduled right after its
  // own wait: worth it behind the wide tile of a call without rotation (GQA
  // fan-out 19.59 against 19.91 us per layer), not on the 7B layer, where the
  // next token-major CTAs would only wait beside it (0.2 % slower)
  int merge_trigger;
  // Rotation calls: the token-major grid starts beside the wide tile on the
  // SMs it leaves free and its other CTAs start as the tile finishes, so
  // claims are taken in turn from a per-pool counter (dyn), one claim ahead;
  // the merge kernel queued behind resets it once this grid has completed.
  int dyn;
  unsigned int* claim_ctr;
  // Every launch is a programmatic dependent of the kernel before it on the
  // stream.  The first kernel of a call (first_wait) waits for that kernel
  // to complete before it reads anything; behind the wide tile the kernel
  // runs beside it and waits only before it completes.
  int first_wait;
  int stall_first;    // test-only (KVS_TEST_STALL_ONE_STAGE): leave one stage unarmed
  float scale_log2;
  RopeSplit rs;
};

// What the consumer needs about a claimed item, written by the producer.
struct TmRec {
  int id;                  // item * hkv + kv head
  int x;                   // kind (bit 30) | group or sequence
  int chunk;
  int cact;                // members whose columns take part
  int len[kTmMaxGroup];    // context lengths: of each member (shared), of the sequence in len[0] (private)
  int pad[4];
};

// the plan was built for this call's shapes (every compare evaluated, no
// short circuit)
__device__ __forceinline__ bool tm_plan_ok(const PlanHdr& h, const TmParams& p) {
  return (h.v[1] == kPlanMagic) & (h.v[2] == p.n_seq) & (h.v[3] == p.max_blocks) & (h.v[4] == p.R) &
         (h.v[5] == p.ib) & (h.v[6] == p.hkv) & (h.v[7] == p.SG) & (h.v[9] == p.ibs) & (h.v[11] == p.compact);
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void prefetch_l1(const void* ptr) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(ptr));
}

template <int D, bool DIFF, bool ROPE>
__global__ void __launch_bounds__(128, KVS_TM_MIN_CTAS)
attn_tm_kernel(const __grid_constant__ TmParams p, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdk,
               const __grid_constant__ CUtensorMap tdv) {
  constexpr int B = 16, TILE = B * D * 2, KS = D / 16;
  constexpr int S = tm_stages<D>();
  constexpr int STAGE = 2 * TILE;
  static_assert(kTmRec > S + 1, "claim records must outnumber the items a ring can hold");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kTmWarps][S];
  __shared__ TmRec recs[kTmWarps][kTmRec];
  __shared__ float rsc[ROPE ? 4 * 64 : 1];   // RoPE frequency pieces (rotation calls)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // a merge kernel queued behind this one (programmatic dependent launch) may
  // be scheduled now; it waits for this grid to complete before reading
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    if (DIFF) {
      prefetch_tmap(&tdk);
      prefetch_tmap(&tdv);
    }
  }
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* wbase = base + warp * S * STAGE;
  const uint32_t wbase_u32 = smem_u32(wbase);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
  }
  if (p.first_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (ROPE) {
    for (int i = threadIdx.x; i < 4 * 64; i += blockDim.x) rsc[i] = p.rs.c[i >> 6][i & 63];
    __syncthreads();
  }
  __syncwarp();

  // the plan must have been built for this call's shapes
  const PlanHdr ph = load_plan_hdr(p.hdr);
  const bool plan_ok = tm_plan_ok(ph, p);
  if (!plan_ok && threadIdx.x == 0 && blockIdx.x == 0) set_err(p.status, KVS_DEVERR_PLAN);
  const int n_claims = plan_ok ? ph.v[0] * p.hkv : 0;
  const int R = p.R;

  // ------------------------------------------ producer state (warp-uniform)
  // This warp's claims are gw, gw + T, gw + 2T, ... (claim id = item * hkv +
  // kv head).  The item entry of the claim after next and the per-lane block
  // entries of the next claim are loaded one claim early, so they have
  // arrived by the time they are used.
  const int T = gridDim.x * kTmWarps;
  auto take = [&]() {   // dynamic claims: the next claim id
    int id = 0;
    if (lane == 0) id = (int)atomicAdd(p.claim_ctr, 1u);
    return __shfl_sync(0xffffffffu, id, 0);
  };
  int n_id = p.dyn ? take() : blockIdx.x * kTmWarps + warp;   // next claim
  int4 n_it = make_int4(0, 0, 0, 0), nn_it = n_it;
  int n_tab = -1, n_aux = 0, n_dif = -1, n_len = 0, n_dlt = 0, n_lb = 0;
  auto load_item = [&](int id) {
    return id < n_claims ? __ldg(p.items + id / p.hkv) : make_int4(0, 0, 0, 0);
  };
  // issue the loads for claim id (item entry it); nothing here consumes them
  auto prepare = [&](int id, const int4& it) {
    n_tab = -1; n_aux = 0; n_dif = -1; n_len = 0; n_dlt = 0; n_lb = 0;
    if (id >= n_claims) return;
    const int kind = it.x >> 30, idx = it.x & ((1 << 30) - 1);
    // lane j holds the item's block j: logical block chunk * ib + j, or
    // (compact items, private) position chunk + j * n of the member's list
    // of unshared blocks, n = its item count
    int b = it.y * p.ib + lane;
    bool in = b < it.z;
    if (p.compact && !kind) {
      const int ni = (it.z + p.ib - 1) / p.ib, li = it.y + lane * ni;
      in = lane < p.ib && li < it.z;
      b = in ? __ldg(p.plist + (size_t)idx * p.max_blocks + li) : 0;
    }
    n_lb = b;
    if (kind) {
      if (in) {
        n_tab = __ldg(p.gphys + (size_t)idx * p.max_blocks + b);
        n_aux = (int)__ldg(p.gmask + (size_t)idx * p.max_blocks + b);
      }
      if (lane < R && idx * R + lane < p.n_seq) n_len = __ldg(p.seq_len + idx * R + lane);
    } else {
      if (in) {
        n_tab = __ldg(p.block_table + (size_t)idx * p.max_blocks + b);
        // raw member bits (a compact list holds unshared blocks only)
        if (p.SG > 1 && !p.compact) n_aux = (int)__ldg(p.gmask + (size_t)(idx / p.SG) * p.max_blocks + b);
        if (DIFF) n_dif = __ldg(p.diff_table + (size_t)idx * p.max_blocks + b);
        if (ROPE) n_dlt = __ldg(p.bdelta + (size_t)idx * p.max_blocks + b);
      }
      if (lane == 0) n_len = __ldg(p.seq_len + idx);
    }
    // the query rows of the item's live columns, into L1 for the consumer
    constexpr int LPR = D * 2 / 128;   // 128-byte lines per query row
    const int col = lane / LPR, part = lane - col * LPR;
    const int h = id - (id / p.hkv) * p.hkv;
    if (col < 8 && col < R * p.g) {
      const int slot = col / p.g, hh = col - slot * p.g;
      if ((it.w >> slot) & 1) {
        const int a = kind ? idx * R + slot : idx;
        if (a < p.n_seq) prefetch_l1(p.q + ((size_t)a * p.hq + h * p.g + hh) * D + part * 64);
      }
    }
  };
  n_it = load_item(n_id);
  if (!p.dyn) nn_it = load_item(n_id + T);
  prepare(n_id, n_it);

  int ord = -1;   // ordinal of the current claim
  int p_kind = 0, p_h = 0, p_b = 0, p_b0 = 0, p_bend = 0, p_mask = 0, p_slot = 0;
  int tab_ent = -1, dif_ent = -1, aux_ent = 0, dlt_ent = 0, lb_ent = 0;
  bool p_compact = false;   // the current item's blocks come from lb_ent
  bool p_done = false;
  auto claim = [&]() {
    if (n_id >= n_claims) {
      p_done = true;
      return;
    }
    const int4 it = n_it;
    ++ord;
    p_kind = it.x >> 30;
    p_h = n_id - (n_id / p.hkv) * p.hkv;
    p_b0 = p_b = it.y * p.ib;
    p_bend = it.z;
    p_compact = p.compact && !p_kind;
    if (p_compact) {   // the item's block count: list positions it.y + j * n below it.z
      const int ni = (it.z + p.ib - 1) / p.ib;
      p_b0 = p_b = 0;
      p_bend = (it.z - it.y + ni - 1) / ni;
    }
    p_mask = it.w;
    p_slot = p_kind ? 0 : (it.x & ((1 << 30) - 1)) % p.SG;
    tab_ent = n_tab;
    aux_ent = n_aux;
    dif_ent = n_dif;
    dlt_ent = n_dlt;
    lb_ent = n_lb;
    TmRec& rec = recs[warp][ord & (kTmRec - 1)];
    if (lane == 0) {
      rec.id = n_id;
      rec.x = it.x;
      rec.chunk = it.y;
      rec.cact = it.w;
    }
    if (lane < kTmMaxGroup) rec.len[lane] = n_len;
    // advance: the next claim's entries, then the entry of the one after
    if (p.dyn) {
      n_id = take();
      n_it = load_item(n_id);
      prepare(n_id, n_it);
    } else {
      n_id += T;
      n_it = nn_it;
      prepare(n_id, n_it);
      nn_it = load_item(n_id + T);
    }
  };
  // Per stage, the record of what it holds: {claim ordinal (-1: no more
  // work), block index (bit 30: the next position holds the block's diff
  // tiles; bit 29: the block id was out of range and nothing was loaded),
  // group members whose columns take this block, RoPE shift of the block
  // (rotation calls)}.  Every field is warp-uniform, so each lane keeps its
  // own copy in registers (selected by stage, never indexed dynamically).
  int4 st_rec[S];
#pragma unroll
  for (int j = 0; j < S; ++j) st_rec[j] = make_int4(-1, 0, 0, 0);
  auto set_rec = [&](int s, const int4& v) {
#pragma unroll
    for (int j = 0; j < S; ++j)
      if (j == s) st_rec[j] = v;
  };
  // A block that carries a mirror diff takes two positions: {K, DK}, then
  // {V, DV}, so that the first is free as soon as S has been computed.
  int pend_drow = -1, pend_row = 0;   // the {V, DV} position still to issue for the last block
  bool stall_pending = blockIdx.x == 0 && warp == 0;
  auto issue = [&](int s) {   // whole warp; lane 0 issues
    uint64_t* bar = &bars[warp][s];
    uint8_t* st = wbase + s * STAGE;
    if (DIFF && pend_drow >= 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, 2 * TILE);
        tma_load_kv_tile<D>(st, &tv, pend_row, bar);
        tma_load_kv_tile_hint<D>(st + TILE, &tdv, pend_drow, bar, l2_policy_evict_first());
      }
      pend_drow = -1;
      return;
    }
    int phys = -1, did = -1, mask = 0, b = 0, dlt = 0;
    while (true) {
      if (!p_done && p_b >= p_bend) claim();
      if (p_done) break;
      const int j = p_b - p_b0;
      b = p_b++;
      if (p_compact) b = __shfl_sync(0xffffffffu, lb_ent, j);
      const int ent = __shfl_sync(0xffffffffu, tab_ent, j);
      const int aux = __shfl_sync(0xffffffffu, aux_ent, j);
      if (p_kind == 0) {
        if ((aux >> p_slot) & 1) continue;   // computed by the group's shared item
        mask = p_mask;
        if (DIFF) did = __shfl_sync(0xffffffffu, dif_ent, j);
        if (ROPE) dlt = __shfl_sync(0xffffffffu, dlt_ent, j);
      } else {
        if (aux == 0) continue;              // not shared at this block
        mask = aux;
      }
      phys = ent;
      break;
    }
    if (p_done) {
      set_rec(s, make_int4(-1, 0, 0, 0));
      if (lane == 0) mbar_arrive(bar);
      return;
    }
    const bool valid = phys >= 0 && phys < p.capacity;
    const bool dval = DIFF && valid && did >= 0 && did < p.diff_capacity;
    if (dval) {
      pend_drow = (did * p.hkv + p_h) * B;
      pend_row = (phys * p.hkv + p_h) * B;
    }
    // test-only: the first stage of warp 0 of CTA 0 is never armed, so its
    // wait runs out
    const bool stall = p.stall_first && stall_pending;
    stall_pending = false;
    // nothing loaded (stall, or a block id out of range): the consumer skips it
    set_rec(s, make_int4(ord, (stall || !valid) ? (b | (1 << 29)) : dval ? (b | (1 << 30)) : b, mask, dlt));
    if (lane != 0 || stall) return;
    if (!valid) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      mbar_arrive(bar);
      return;
    }
    if (DIFF && did >= p.diff_capacity) set_err(p.status, KVS_DEVERR_DIFF_ID);
    mbar_arrive_expect_tx(bar, 2 * TILE);
    const int row = (phys * p.hkv + p_h) * B;
    // K and V of a block are read once per call here, and so are the diff
    // tiles: evict-first, so that the master blocks under mirror diffs (read
    // by several agents, with the default policy) stay in L2
    const uint64_t pol = l2_policy_evict_first();
    if (dval) {
      tma_load_kv_tile<D>(st, &tk, row, bar);
      tma_load_kv_tile_hint<D>(st + TILE, &tdk, pend_drow, bar, pol);
    } else {
      tma_load_kv_tile_hint<D>(st, &tk, row, bar, pol);
      tma_load_kv_tile_hint<D>(st + TILE, &tv, row, bar, pol);
    }
  };
  for (int s = 0; s < S; ++s) issue(s);

  // --------------------------------------------------- per-lane constants
  uint32_t koff[KS], voff[KS];
  {
    const int mi = lane >> 3, r = lane & 7;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      koff[kk] = kv_tile_off<D>(((mi & 1) << 3) + r, kk * 16 + ((mi >> 1) << 3));   // A = K [token][d]
      voff[kk] = kv_tile_off<D>(((mi >> 1) << 3) + r, kk * 16 + ((mi & 1) << 3));   // A = V^T via .trans
    }
  }

  // ------------------------------------------------------ consumer state
  // Column j of the 8-wide tile belongs to group member j / G (query head
  // j % G).  colslot / colL: member and context length of this lane's two
  // score columns (2c, 2c+1); slot 31 marks a column that is never live.
  int cur = -1, ckind = 0, cidx = 0, ch_ = 0, cchunk = 0, cact = 0;
  int colL[2] = {0, 0};
  int colslot[2] = {31, 31};
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, acc[D / 16][4];
  uint32_t qb[KS][2];
  uint32_t qlo[ROPE ? KS : 1][2];
  bool q_has_lo = false;
  int cur_delta = 0;
  const uint16_t* qrow = nullptr;
  bool qok = false;

  auto load_q = [&]() {
    q_has_lo = false;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int col = kk * 16 + 2 * c;
      qb[kk][0] = qok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + col)) : 0u;
      qb[kk][1] = qok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + col + 8)) : 0u;
    }
  };
  // q' = R(-delta) q, as bf16 hi + lo.  Lane (g, c) holds head dims
  // kk*16 + 2c + half*8 + {0, 1} (and the same + D/2), so the angles it needs
  // depend on c only: the 8 lanes sharing c each compute 2*KS/8 of them and
  // exchange the rest by shuffles.
  auto rotate_q = [&](int delta) {
    q_has_lo = true;
    constexpr int PER = (2 * KS) / 8;   // angles computed per lane
    float cs_own[PER], sn_own[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = g * PER + u;      // idx = (kk * 2 + half) * 2 + e
      const int e = idx & 1, half = (idx >> 1) & 1, kk = idx >> 2;
      rope_cos_sin(rsc, kk * 16 + 2 * c + half * 8 + e, delta, cs_own[u], sn_own[u]);
    }
#pragma unroll
    for (int kk = 0; kk < KS / 2; ++kk) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int col = kk * 16 + 2 * c + half * 8;
        const int i0 = (kk * 2 + half) * 2, i1 = i0 + 1;
        const int src0 = ((i0 / PER) << 2) | c, src1 = ((i1 / PER) << 2) | c;
        const float cs0 = __shfl_sync(0xffffffffu, cs_own[i0 % PER], src0);
        const float sn0 = __shfl_sync(0xffffffffu, sn_own[i0 % PER], src0);
        const float cs1 = __shfl_sync(0xffffffffu, cs_own[i1 % PER], src1);
        const float sn1 = __shfl_sync(0xffffffffu, sn_own[i1 % PER], src1);
        const uint32_t lo = qok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + col)) : 0u;
        const uint32_t hi = qok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + col + D / 2)) : 0u;
        const float l0 = bf16_lo(lo), l1 = bf16_hi(lo), h0 = bf16_lo(hi), h1 = bf16_hi(hi);
        split_bf16(l0 * cs0 + h0 * sn0, l1 * cs1 + h1 * sn1, qb[kk][half], qlo[ROPE ? kk : 0][half]);
        split_bf16(h0 * cs0 - l0 * sn0, h1 * cs1 - l1 * sn1, qb[kk + KS / 2][half],
                   qlo[ROPE ? kk + KS / 2 : 0][half]);
      }
    }
  };

  // write the current item's split(s); tm_merge_kernel combines them
  auto flush = [&]() {
    float lt[2] = {l[0], l[1]};
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lt[0] += __shfl_xor_sync(0xffffffffu, lt[0], o);
      lt[1] += __shfl_xor_sync(0xffffffffu, lt[1], o);
    }
    float* dst = ckind ? p.p2 : p.p1;
    float* dml = ckind ? p.p2_ml : p.p1_ml;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int j = 2 * c + cc;
      const int slot = colslot[cc];
      if (slot != 31) {
        const int a = ckind ? cidx * R + slot : cidx;
        const int hh = j - slot * p.g;
        const int nch = ckind ? p.n_chunks_s : p.n_chunks;
        const size_t it = (((size_t)a * p.hkv + ch_) * nch + cchunk) * p.g + hh;
        float* pr = dst + it * D;
        const size_t im = (((size_t)a * p.hkv + ch_) * p.g + hh) * nch + cchunk;
        // evict-last: the merge reads the split back once the grid is done,
        // and the evict-first K/V stream should not push it out first
        // (all-gather round 227.8 -> 226.3 us per layer, 7B 161.5 -> 161.2 us)
        const uint64_t pol = l2_policy_evict_last();
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          st_hint_f32(pr + mt * 16 + g, acc[mt][cc], pol);
          st_hint_f32(pr + mt * 16 + g + 8, acc[mt][2 + cc], pol);
        }
        if (g == 0) st_hint_v2f32(dml + im * 2, make_float2(m[cc], lt[cc]), pol);
      }
    }
  };

  int i = 0;
  bool timed_out = false;
  for (;;) {
    const int s = i % S;
    // The stage's record was set when the stage was armed: the item switch
    // (the previous item's split stores, the next query loads) and the query
    // rotation below run while the stage's copies are in flight.
    __syncwarp();
    int4 srec = st_rec[0];
#pragma unroll
    for (int j = 1; j < S; ++j)
      if (j == s) srec = st_rec[j];
    const int item = srec.x, bword = srec.y, emask = srec.z;
    if (item < 0) break;   // armed without copies: the claims are exhausted
    const bool has_diff = DIFF && (bword >> 30) != 0;
    const int b = bword & ((1 << 29) - 1);
    const bool loaded = ((bword >> 29) & 1) == 0;
    const int s2 = (i + 1) % S;   // a diff block's {V, DV} stage, waited for before P V
    if (item != cur) {
      if (cur >= 0) flush();
      cur = item;
      __syncwarp();   // the record was written by several lanes
      const TmRec& rec = recs[warp][item & (kTmRec - 1)];
      ch_ = rec.id - (rec.id / p.hkv) * p.hkv;
      cchunk = rec.chunk;
      ckind = rec.x >> 30;
      cidx = rec.x & ((1 << 30) - 1);
      cact = rec.cact;
      int agent_of_col = -1;   // sequence of this lane's query column (n = g)
      {
        const int slot = g / p.g;
        if (g < R * p.g && ((cact >> slot) & 1)) agent_of_col = ckind ? cidx * R + slot : cidx;
      }
      qok = agent_of_col >= 0;
      qrow = p.q + ((size_t)(qok ? agent_of_col : 0) * p.hq + ch_ * p.g + (g % p.g)) * D;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int j = 2 * c + cc;
        const int slot = j / p.g;
        const bool on = j < R * p.g && ((cact >> slot) & 1);
        colslot[cc] = on ? slot : 31;
        colL[cc] = on ? min(max(rec.len[ckind ? slot : 0], 0), p.max_blocks * B) : 0;
      }
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      load_q();
      cur_delta = 0;
    }
    if (ROPE && loaded) {
      const int nd = srec.w;   // the plan checked |nd| < 2^18
      if (nd != cur_delta) {
        if (nd == 0) load_q(); else rotate_q(nd);
        cur_delta = nd;
      }
    }
    if (!mbar_wait_bounded(&bars[warp][s], (i / S) & 1, p.status)) {
      timed_out = true;
      break;
    }
    if (loaded) {
      // {K, V}, or with a diff {K, DK} in stage s and {V, DV} in stage s2
      const uint32_t tkb = wbase_u32 + s * STAGE, dkb = tkb + TILE;
      const uint32_t tvb = has_diff ? wbase_u32 + s2 * STAGE : tkb + TILE, dvb = tvb + TILE;
      // S^T = K q^T : 16 tokens x 8 query columns, two accumulation chains
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        float* acc_s = (kk & 1) ? sd : sc;
        uint32_t a[4];
        ldsm_x4(tkb + koff[kk], a[0], a[1], a[2], a[3]);
        mma_bf16(acc_s, a, qb[kk][0], qb[kk][1]);
        if (ROPE && q_has_lo) mma_bf16(acc_s, a, qlo[ROPE ? kk : 0][0], qlo[ROPE ? kk : 0][1]);
        if (has_diff) {   // the diff tile against the query's hi part only (its lo part
                          // adds about 2^-9 of a correction term that is itself small)
          ldsm_x4(dkb + koff[kk], a[0], a[1], a[2], a[3]);
          mma_bf16(acc_s, a, qb[kk][0], qb[kk][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] += sd[e];
      if (has_diff) {   // K and DK have been read: stage s takes the next position now
        __syncwarp();
        issue(s);
      }
      // sc: (t=g, col 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1); a column is live
      // if its member takes this block (slot 31 never does: emask < 2^8) and
      // the token is inside its context
      {
        const int lim0 = ((emask >> colslot[0]) & 1) ? colL[0] - b * B : 0;
        const int lim1 = ((emask >> colslot[1]) & 1) ? colL[1] - b * B : 0;
        sc[0] = g < lim0 ? sc[0] * p.scale_log2 : -INFINITY;
        sc[1] = g < lim1 ? sc[1] * p.scale_log2 : -INFINITY;
        sc[2] = g + 8 < lim0 ? sc[2] * p.scale_log2 : -INFINITY;
        sc[3] = g + 8 < lim1 ? sc[3] * p.scale_log2 : -INFINITY;
      }
      // Lazy rescale: a column keeps its reference point m while none of its
      // scores exceeds m by more than kTmLazyLog2, so most blocks need no
      // reduction of the column maxima over the tile.  P then stays below
      // 2^kTmLazyLog2, which the bf16 hi + lo split and the fp32 sums carry at
      // full relative precision, and (m, l, acc) keep one reference point
      // for the merge.
      const float t0 = fmaxf(sc[0], sc[2]), t1 = fmaxf(sc[1], sc[3]);
      if (__any_sync(0xffffffffu, t0 > m[0] + kTmLazyLog2 || t1 > m[1] + kTmLazyLog2)) {
        float mx0 = t0, mx1 = t1;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        // (a column whose state is still empty has l = 0 and acc = 0)
        const float al0 = m[0] == -INFINITY ? 0.f : fast_exp2(m[0] - mn0);
        const float al1 = m[1] == -INFINITY ? 0.f : fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        l[0] *= al0;
        l[1] *= al1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          acc[mt][0] *= al0; acc[mt][1] *= al1;
          acc[mt][2] *= al0; acc[mt][3] *= al1;
        }
      }
      // a column with nothing live yet keeps (m, l, acc) = (-inf, 0, 0): its
      // reference point is taken as 0 so that exp2(-inf - 0) = 0
      const float r0 = m[0] == -INFINITY ? 0.f : m[0], r1 = m[1] == -INFINITY ? 0.f : m[1];
      sc[0] = fast_exp2(sc[0] - r0);
      sc[1] = fast_exp2(sc[1] - r1);
      sc[2] = fast_exp2(sc[2] - r0);
      sc[3] = fast_exp2(sc[3] - r1);
      l[0] += sc[0] + sc[2];
      l[1] += sc[1] + sc[3];
      // a diff block's {V, DV} tiles (the stage after S's) are needed from here
      // on: S and the softmax above overlapped their copy
      if (has_diff && !mbar_wait_bounded(&bars[warp][s2], ((i + 1) / S) & 1, p.status)) {
        timed_out = true;
        ++i;   // stage s was re-armed for position i + 2 above: drain from there
        break;
      }
      // P^T as the B operand (k = token, n = query column), bf16 hi + lo
      uint32_t h0, l0_, h1, l1_;
      split_bf16(sc[0], sc[1], h0, l0_);
      split_bf16(sc[2], sc[3], h1, l1_);
      const uint32_t bh0 = movm_t(h0), bh1 = movm_t(h1), bl0 = movm_t(l0_), bl1 = movm_t(l1_);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(tvb + voff[mt], a[0], a[1], a[2], a[3]);
        mma_bf16(acc[mt], a, bh0, bh1);
        mma_bf16(acc[mt], a, bl0, bl1);
        if (has_diff) {   // likewise P's hi part only against the diff tile
          ldsm_x4_t(dvb + voff[mt], a[0], a[1], a[2], a[3]);
          mma_bf16(acc[mt], a, bh0, bh1);
        }
      }
    }
    // The copies issued next overwrite tiles that this warp has only read, and
    // every such read (an ldmatrix whose registers the MMAs above consumed) has
    // completed, so no proxy fence is needed before the async-proxy writes.
    __syncwarp();
    if (!(loaded && has_diff)) issue(s);   // (a loaded diff block released s after S)
    if (has_diff) issue(s2);
    i += has_diff ? 2 : 1;
  }
  if (timed_out) {
    // the other stages may still have copies in flight: let them land (with
    // a limit) before the shared memory goes away
    for (int j = 1; j < S; ++j) mbar_drain(&bars[warp][(i + j) % S], ((i + j) / S) & 1);
  }
  if (cur >= 0) flush();
  // when this grid was launched behind the wide tile (programmatic dependent
  // launch) it must not complete before that grid has: the merge queued
  // behind this one reads both grids' splits (no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kMergeWarps = 8;
#ifndef KVS_MERGE_SLOTS_PER_WARP
#define KVS_MERGE_SLOTS_PER_WARP 64
#endif
// Four CTAs per SM (64 registers; batches of 8 split loads per lane, the
// most that fits without spills) keep the all-gather round's 320 merge CTAs
// in one wave: per layer 230.9 us with two CTAs per SM and batches of 12,
// 228.0 us with three, 228.6 us with four; the GQA fan-out took 21.2, 21.4
// and 20.7 us.
#ifndef KVS_MERGE_BATCH
#define KVS_MERGE_BATCH 8
#endif
#ifndef KVS_MERGE_MIN_CTAS
#define KVS_MERGE_MIN_CTAS 4
#endif
constexpr int kMergeBatch = KVS_MERGE_BATCH;

// Split merge, interleaved form.  The row's splits are dealt out round
// robin: warp wq of the row takes slots wq, wq + wpr, wq + 2 wpr, ...
// Existing splits sit in runs of consecutive slots (a sequence's chunks with
// unshared work, the chunks of its shared prefix), so every warp gets about
// the same number of them and loads them in one batch.  Each warp reads only
// its own slots' (m, l) and sums its splits relative to its own maximum; the
// row's warps then rescale their parts to the row's maximum and add them in
// a fixed order, so results are deterministic.

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32, KVS_MERGE_MIN_CTAS)
tm_merge_kernel(const __grid_constant__ TmParams p) {
  constexpr int CPL = D / 32;   // columns per lane
  __shared__ __align__(16) float sv[kMergeWarps][D];
  __shared__ float sL[kMergeWarps], sM[kMergeWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpr = p.mwpr;
  const int rl = warp / wpr, wq = warp - rl * wpr;
  const int row = blockIdx.x * (kMergeWarps / wpr) + rl;   // sequence * hq + query head
  const bool in_range = row < p.n_seq * p.hq;
  const int a = in_range ? row / p.hq : 0, qh = row - a * p.hq, h = qh / p.g, hh = qh - h * p.g;
  const size_t sbase = ((size_t)a * p.hkv + h) * p.n_chunks, sbase_s = ((size_t)a * p.hkv + h) * p.n_chunks_s;
  const int n_slots = in_range ? p.n_chunks + (p.SG > 1 ? p.n_chunks_s : 0) : 0;
  auto slot_off = [&](int sl) {   // split index of a slot
    return sl < p.n_chunks ? (sbase + sl) * p.g + hh : (sbase_s + (sl - p.n_chunks)) * p.g + hh;
  };
  // (m, l) index of a slot: a row's (m, l) are contiguous, so a warp reading
  // 32 consecutive slots touches two or three cache lines
  const size_t mrow = ((size_t)a * p.hkv + h) * p.g + hh;
  auto ml_off = [&](int sl) {
    return sl < p.n_chunks ? mrow * p.n_chunks + sl : mrow * p.n_chunks_s + (sl - p.n_chunks);
  };
  // Before the wait: this CTA is often resident well before the attention
  // grid completes, and what it reads below has usually left L2 (the (m, l)
  // of splits that no item writes were set by the plan once per step; early
  // splits were written long ago).  It fetches its row's lines into L2: every
  // slot's (m, l) line and, when the launch asks for it (p.merge_prefetch),
  // every slot's data.  A prefetch returns nothing to this program, and L2
  // is where every write lands, so everything is read after the wait and is
  // correct.
  for (int sl = wq + lane * wpr; sl < n_slots; sl += 32 * wpr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"((sl >= p.n_chunks ? p.p2_ml : p.p1_ml) + ml_off(sl) * 2));
    if (p.merge_prefetch) {
      const char* src = reinterpret_cast<const char*>((sl >= p.n_chunks ? p.p2 : p.p1) + slot_off(sl) * D);
#pragma unroll
      for (int j = 0; j < D * 4; j += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + j));
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // behind a wide tile the next call's first kernel (its tile) may be
  // scheduled now and do its set-up while this grid merges
  if (p.merge_trigger) asm volatile("griddepcontrol.launch_dependents;");
  // the token-major grid has completed: its claim counter starts the next call at zero
  if (p.dyn && blockIdx.x == 0 && threadIdx.x == 0) *p.claim_ctr = 0u;
  // a plan built for other shapes: the attention kernel computed nothing and
  // flagged it; the output is left untouched as well
  const bool plan_ok = tm_plan_ok(load_plan_hdr(p.hdr), p);
  // The plan set the (m, l) of splits that no item writes to (-inf, 0), so a
  // split exists exactly when its l is positive.
  auto load_ml = [&](int sl) {
    if (sl >= n_slots) return make_float2(-INFINITY, 0.f);
    const float* base = sl >= p.n_chunks ? p.p2_ml : p.p1_ml;
    return __ldcg(reinterpret_cast<const float2*>(base + ml_off(sl) * 2));
  };

  // 1. This warp's slots (lane k of pass j: slot 32 * wpr * j + k * wpr + wq)
  // and the warp's own maximum Mw over the splits among them.  The (m, l) of
  // the first two passes are loaded together and kept for step 2.
  const float2 own0 = load_ml(lane * wpr + wq), own1 = load_ml(32 * wpr + lane * wpr + wq);
  float Mw = -INFINITY;
  if (own0.y > 0.f) Mw = own0.x;
  if (own1.y > 0.f) Mw = fmaxf(Mw, own1.x);
  for (int base = 64 * wpr; base < n_slots; base += 32 * wpr) {   // rows of more than 64 * wpr slots
    const float2 ml = load_ml(base + lane * wpr + wq);
    if (ml.y > 0.f) Mw = fmaxf(Mw, ml.x);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, off));

  // 2. the warp's splits, weighted relative to Mw
  float v[CPL], Lw = 0.f;
#pragma unroll
  for (int j = 0; j < CPL; ++j) v[j] = 0.f;
  for (int base = 0; base < n_slots; base += 32 * wpr) {
    const int sl = base + lane * wpr + wq;
    const float2 ml = base == 0 ? own0 : base == 32 * wpr ? own1 : load_ml(sl);
    const bool ex = ml.y > 0.f;
    const float wk = ex ? fast_exp2(ml.x - Mw) : 0.f;
    Lw += wk * ml.y;
    unsigned mk = __ballot_sync(0xffffffffu, ex);
    while (mk) {   // warp-uniform: up to kMergeBatch splits, their loads all in flight
      float x[kMergeBatch][CPL];
      unsigned mq = mk;
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        if (!mq) continue;
        const int s2 = base + (__ffs(mq) - 1) * wpr + wq;
        mq &= mq - 1;
        const float* src = (s2 >= p.n_chunks ? p.p2 : p.p1) + slot_off(s2) * D + lane * CPL;
        if (CPL == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
          x[u][0] = t.x; x[u][1 % CPL] = t.y; x[u][2 % CPL] = t.z; x[u][3 % CPL] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
          x[u][0] = t.x; x[u][1 % CPL] = t.y;
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        if (!mk) continue;
        const float wgt = __shfl_sync(0xffffffffu, wk, __ffs(mk) - 1);
        mk &= mk - 1;
#pragma unroll
        for (int j = 0; j < CPL; ++j) v[j] += wgt * x[u][j];
      }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) Lw += __shfl_xor_sync(0xffffffffu, Lw, off);

  // 3. the row's warps add their parts in order, each rescaled from its own
  // maximum to the row's (a warp without splits adds nothing); the first
  // warp stores
  if (wpr > 1) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) sv[warp][lane * CPL + j] = v[j];
    if (lane == 0) {
      sL[warp] = Lw;
      sM[warp] = Mw;
    }
    __syncthreads();
    if (wq != 0) return;
    float M = Mw;
    for (int w = 1; w < wpr; ++w) M = fmaxf(M, sM[warp + w]);
    const float f0 = Mw == -INFINITY ? 0.f : fast_exp2(Mw - M);
#pragma unroll
    for (int j = 0; j < CPL; ++j) v[j] *= f0;
    Lw *= f0;
    for (int w = 1; w < wpr; ++w) {
      const float mw = sM[warp + w];
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
#pragma unroll
      for (int j = 0; j < CPL; ++j) v[j] += f * sv[warp + w][lane * CPL + j];
      Lw += f * sL[warp + w];
    }
  }
  if (!in_range || !plan_ok) return;
  // an empty context (no splits at all) gives a zero output
  const float inv = Lw > 0.f ? 1.f / Lw : 0.f;
  float* o = p.out + (size_t)row * D + lane * CPL;
  if (CPL == 4) {
    *reinterpret_cast<float4*>(o) = make_float4(v[0] * inv, v[1 % CPL] * inv, v[2 % CPL] * inv, v[3 % CPL] * inv);
  } else {
    *reinterpret_cast<float2*>(o) = make_float2(v[0] * inv, v[1 % CPL] * inv);
  }
}

template <int D>
static kvs_status launch_merge(const TmParams& prm, cudaStream_t st) {
  const int rows = prm.n_seq * prm.hq;
  cudaLaunchConfig_t cfg = {};
  const int rows_per_cta = kMergeWarps / prm.mwpr;
  cfg.gridDim = dim3((rows + rows_per_cta - 1) / rows_per_cta);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tm_merge_kernel<D>, prm) != cudaSuccess) {
    // the merge would have reset the token-major claim counter: do it here so
    // that the pool's next call starts from zero
    if (prm.dyn) cudaMemsetAsync(prm.claim_ctr, 0, sizeof(unsigned int), st);
    return fail(KVS_ERR_CUDA, "decode_attn: merge launch failed");
  }
  count_launch();
  return check_launch("decode_attn_merge");
}


template <int D, bool DIFF, bool ROPE>
static kvs_status launch_tm(TmParams& prm, const kvs_pool* pool, int layer, int max_claims, bool after_wide,
                            bool pdl, cudaStream_t st) {
  auto kern = attn_tm_kernel<D, DIFF, ROPE>;
  constexpr int smem = tm_smem_bytes<D>();
  // occupancy depends only on the kernel and the device type (one type of
  // device per process is assumed for the cached count)
  static std::atomic<int> occ{0};
  int blocks_per_sm = occ.load(std::memory_order_relaxed);
  if (!smem_limit_once<attn_tm_kernel<D, DIFF, ROPE>>(smem, pool->device))
    return fail(KVS_ERR_CUDA, "decode_attn: cannot raise the shared-memory limit");
  if (!blocks_per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kern, 128, smem) != cudaSuccess ||
        blocks_per_sm < 1)
      return fail(KVS_ERR_CUDA, "decode_attn: cannot configure the token-major kernel");
    occ.store(blocks_per_sm, std::memory_order_relaxed);
  }
  // persistent grid: every SM filled once, but never more warps than the
  // largest possible number of claims
  const int grid = std::max(1, std::min(pool->num_sms * blocks_per_sm, (max_claims + kTmWarps - 1) / kTmWarps));
  const CUtensorMap& dk = DIFF ? pool->tdk[layer] : pool->tk[layer];
  const CUtensorMap& dv = DIFF ? pool->tdv[layer] : pool->tv[layer];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;   // behind the wide tile: start on the SMs it leaves free
  prm.first_wait = after_wide ? 0 : 1;
  if (cudaLaunchKernelEx(&cfg, kern, (const TmParams)prm, pool->tk[layer], pool->tv[layer], dk, dv) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_attn: launch failed");
  count_launch();
  const kvs_status s = check_launch("decode_attn");
  if (s != KVS_OK) return s;
  return launch_merge<D>(prm, st);
}

// workspace pointers shared by the plan and the launch
struct TmPtrs {
  int* hdr;
  int4* items;
  int4* witems;
  int2* wsub;
  int2* wmem;
  int4* wclaims;
  uint32_t* gmask;
  int32_t* gphys;
  uint8_t* pne;
  uint32_t* spm;
  int32_t* bdelta;
  int32_t* bwin;
  int32_t* plist;
  int32_t* pcnt;
  float *p1, *p1_ml, *p2, *p2_ml;
};

static TmPtrs tm_ptrs(const TmLayout& L, const kvs_pool* pool, int n_seq, int g, void* ws) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t per_chunk = (size_t)n_seq * pool->desc.num_kv_heads * g * pool->desc.head_dim;
  const size_t split_vals = per_chunk * L.n_chunks, split_vals_s = per_chunk * L.n_chunks_s;
  TmPtrs t{};
  t.hdr = reinterpret_cast<int*>(w + L.off_hdr);
  t.items = reinterpret_cast<int4*>(w + L.off_items);
  t.gmask = reinterpret_cast<uint32_t*>(w + L.off_gmask);
  t.gphys = reinterpret_cast<int32_t*>(w + L.off_gphys);
  t.pne = w + L.off_pne;
  t.spm = reinterpret_cast<uint32_t*>(w + L.off_spm);
  t.witems = reinterpret_cast<int4*>(w + L.off_witems);
  t.wsub = reinterpret_cast<int2*>(w + L.off_wsub);
  t.wmem = reinterpret_cast<int2*>(w + L.off_wmem);
  t.wclaims = reinterpret_cast<int4*>(w + L.off_wclaims);
  t.bdelta = reinterpret_cast<int32_t*>(w + L.off_bdelta);
  t.bwin = reinterpret_cast<int32_t*>(w + L.off_bwin);
  t.plist = reinterpret_cast<int32_t*>(w + L.off_plist);
  t.pcnt = reinterpret_cast<int32_t*>(w + L.off_pcnt);
  t.p1 = reinterpret_cast<float*>(w + L.off_p1);
  t.p1_ml = t.p1 + split_vals;
  t.p2 = reinterpret_cast<float*>(w + L.off_p2);
  t.p2_ml = t.p2 + (L.SG > 1 ? split_vals_s : 0);
  return t;
}

kvs_status decode_plan_token_major(kvs_pool* pool, int n_q_heads, const int32_t* table, int max_blocks,
                                   const int32_t* seq_len, int n_seq, const int32_t* diff, const int32_t* rope_off,
                                   const kvs_seg_rope* rope_segs, void* ws, cudaStream_t stream) {
  const bool rope = rope_off != nullptr;
  const int g = n_q_heads / pool->desc.num_kv_heads;
  const TmLayout L = tm_layout(pool, n_seq, max_blocks, g, rope);
  const TmPtrs t = tm_ptrs(L, pool, n_seq, g, ws);
  PlanParams pp{};
  pp.block_table = table;
  pp.seq_len = seq_len;
  pp.diff_table = diff;
  pp.hdr = t.hdr;
  pp.items = t.items;
  pp.gmask = t.gmask;
  pp.gphys = t.gphys;
  pp.pne = t.pne;
  pp.spm = t.spm;
  pp.rope_off = rope_off;
  pp.rope_segs = reinterpret_cast<const int4*>(rope_segs);
  pp.bdelta = t.bdelta;
  pp.bwin = t.bwin;
  pp.status = pool->status;
  pp.p1_ml = t.p1_ml;
  pp.p2_ml = t.p2_ml;
  pp.n_seq = n_seq;
  pp.max_blocks = max_blocks;
  pp.R = L.R;
  pp.SG = L.SG;
  pp.wide = L.wide ? 1 : 0;
  pp.witems = t.witems;
  pp.wsub = t.wsub;
  pp.wmem = t.wmem;
  pp.wclaims = t.wclaims;
  pp.max_sub = L.max_sub;
  pp.runs = L.runs ? 1 : 0;
  pp.max_witems = (int)std::min<size_t>(L.max_witems, 0x7fffffff);
  pp.G = g;
  pp.ib = L.ib;
  pp.n_chunks = L.n_chunks;
  pp.ibs = L.ibs;
  pp.n_chunks_s = L.n_chunks_s;
  pp.n_groups = L.n_groups;
  pp.capacity = pool->desc.capacity_blocks;
  pp.hkv = pool->desc.num_kv_heads;
  pp.wide_ctas = L.runs ? runs_wide_ctas(pool) : pool->num_sms;   // the wide tile's grid
  pp.plist = t.plist;
  pp.pcnt = t.pcnt;
  pp.compact = L.compact ? 1 : 0;
  // item counters start at zero (several CTAs add to them)
  if (cudaMemsetAsync(t.hdr, 0, 64, stream) != cudaSuccess) return fail(KVS_ERR_CUDA, "decode_plan: memset failed");
  if (rope) {
    if (launch_pdl(tm_plan_shifts, dim3(std::max(1, std::min(n_seq, pool->num_sms * 8))), dim3(256), stream, pp) !=
        cudaSuccess)
      return fail(KVS_ERR_CUDA, "decode_plan: launch failed");
    count_launch();
    const kvs_status st0 = check_launch("decode_plan");
    if (st0 != KVS_OK) return st0;
  }
  const int g1 = std::max(1, std::min(L.n_groups, pool->num_sms * 4));
  if (launch_pdl(tm_plan_groups, dim3(g1), dim3(512), stream, pp) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_plan: launch failed");
  count_launch();
  kvs_status st = check_launch("decode_plan");
  if (st != KVS_OK) return st;
  const long long slots = (long long)(L.max_items + L.max_witems);
  const int g2 = (int)std::max<long long>(1, std::min<long long>((slots + 255) / 256, pool->num_sms * 8));
  if (launch_pdl(tm_plan_items, dim3(g2), dim3(256), stream, pp) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_plan: launch failed");
  count_launch();
  return check_launch("decode_plan");
}

kvs_status decode_attn_token_major(kvs_pool* pool, int layer, const void* q, int n_q_heads, const int32_t* table,
                                   int max_blocks, const int32_t* seq_len, int n_seq, const int32_t* diff,
                                   const int32_t* rope_off, const kvs_seg_rope* rope_segs, float theta,
                                   float scale, float* out, void* ws, cudaStream_t stream) {
  const kvs_pool_desc& d = pool->desc;
  const int g = n_q_heads / d.num_kv_heads;
  const bool rope = rope_off != nullptr, dif = diff != nullptr;
  const TmLayout L = tm_layout(pool, n_seq, max_blocks, g, rope);
  const TmPtrs t = tm_ptrs(L, pool, n_seq, g, ws);
  TmParams prm{};
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = table;
  prm.seq_len = seq_len;
  prm.diff_table = diff;
  prm.bdelta = rope ? t.bdelta : nullptr;
  prm.out = out;
  prm.p1 = t.p1;
  prm.p1_ml = t.p1_ml;
  prm.p2 = t.p2;
  prm.p2_ml = t.p2_ml;
  prm.hdr = t.hdr;
  prm.items = t.items;
  prm.gmask = t.gmask;
  prm.gphys = t.gphys;
  prm.plist = t.plist;
  prm.compact = L.compact ? 1 : 0;
  prm.status = pool->status;
  prm.max_blocks = max_blocks;
  prm.n_seq = n_seq;
  prm.hkv = d.num_kv_heads;
  prm.g = g;
  prm.hq = n_q_heads;
  prm.ib = L.ib;
  prm.n_chunks = L.n_chunks;
  prm.ibs = L.ibs;
  prm.n_chunks_s = L.n_chunks_s;
  prm.R = L.R;
  prm.SG = L.SG;
  prm.capacity = d.capacity_blocks;
  prm.diff_capacity = d.diff_capacity_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  // about two batches of split slots per merge warp (of which typically
  // fewer than half exist), so that the merge grid stays within one wave
  prm.mwpr = 1;
  prm.merge_prefetch = L.wide ? 0 : 1;
  prm.merge_trigger = (L.wide && !L.runs) ? 1 : 0;
  const int n_slots = L.n_chunks + (L.SG > 1 ? L.n_chunks_s : 0);
  if (L.compact) {
    // compact items fill only the first slots of a row (as many as its list
    // needs items): one warp per row while its range spans at most two
    // 32-slot windows (rows of such calls are many; 32 measured 0.5 % slower
    // on the all-gather round)
    while (prm.mwpr < kMergeWarps && (n_slots + prm.mwpr - 1) / prm.mwpr > KVS_MERGE_SLOTS_PER_WARP) prm.mwpr <<= 1;
  } else {
    while (prm.mwpr < kMergeWarps && prm.mwpr * 2 * kMergeBatch < n_slots) prm.mwpr <<= 1;
  }
  if (rope) rope_split_host(theta, d.head_dim, prm.rs.c);
  prm.claim_ctr = reinterpret_cast<unsigned int*>(pool->status) + 1;
  prm.stall_first = (pool->test_flags & KVS_TEST_STALL_ONE_STAGE) ? 1 : 0;
  pool->test_flags &= ~KVS_TEST_STALL_ONE_STAGE;   // one launch only
  const int max_claims = (int)std::min<size_t>(L.max_items * d.num_kv_heads, 0x7fffffff);
  bool wide_launched = false, runs_launched = false;
  if (L.wide) {
    // the shared chunks of every sharing group, on the tensor cores; they
    // write the shared splits, disjoint from what the token-major kernel writes
    WideParams wp{};
    wp.q = prm.q;
    wp.witems = t.witems;
    wp.hdr = t.hdr;
    wp.wsub = t.wsub;
    wp.wmem = t.wmem;
    wp.wclaims = t.wclaims;
    wp.max_sub = L.max_sub;
    wp.max_witems = (int)std::min<size_t>(L.max_witems, 0x7fffffff);
    wp.runs = L.runs ? 1 : 0;
    if (L.runs) std::memcpy(wp.rs, prm.rs.c, sizeof(wp.rs));
    wp.p2 = t.p2;
    wp.p2_ml = t.p2_ml;
    wp.status = pool->status;
    wp.n_seq = n_seq;
    wp.max_blocks = max_blocks;
    wp.hkv = d.num_kv_heads;
    wp.g = g;
    wp.hq = n_q_heads;
    wp.W = L.SG;
    wp.ib = L.ibs;
    wp.ibp = L.ib;
    wp.n_chunks = L.n_chunks_s;
    wp.R = L.R;
    wp.capacity = d.capacity_blocks;
    wp.magic = kPlanMagic;
    wp.scale_log2 = prm.scale_log2;
    const int wide_claims = (int)std::min<size_t>(L.max_witems * d.num_kv_heads, 0x7fffffff);
    const kvs_status ws_ = launch_wide_tile(wp, pool, layer, wide_claims, stream);
    if (ws_ != KVS_OK) return ws_;
    // rotation calls leave the token-major kernel the heavier part (private
    // blocks and mirror diffs); it runs after the tile at full occupancy
    // behind the tile (shared chunks: beside it on every SM; rotation calls:
    // on the SMs it leaves free), the merge waiting on both grids
    wide_launched = wide_claims > 0;
    runs_launched = wide_claims > 0 && L.runs;
  }
  const bool pdl = true;
  prm.dyn = runs_launched ? 1 : 0;
  if (d.head_dim == 128) {
    if (dif) return rope ? launch_tm<128, true, true>(prm, pool, layer, max_claims, wide_launched, pdl, stream)
                         : launch_tm<128, true, false>(prm, pool, layer, max_claims, wide_launched, pdl, stream);
    return rope ? launch_tm<128, false, true>(prm, pool, layer, max_claims, wide_launched, pdl, stream)
                : launch_tm<128, false, false>(prm, pool, layer, max_claims, wide_launched, pdl, stream);
  }
  if (dif) return rope ? launch_tm<64, true, true>(prm, pool, layer, max_claims, wide_launched, pdl, stream)
                       : launch_tm<64, true, false>(prm, pool, layer, max_claims, wide_launched, pdl, stream);
  return rope ? launch_tm<64, false, true>(prm, pool, layer, max_claims, wide_launched, pdl, stream)
              : launch_tm<64, false, false>(prm, pool, layer, max_claims, wide_launched, pdl, stream);
}

}  // namespace kvs
