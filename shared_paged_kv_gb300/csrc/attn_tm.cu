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
//  * Persistent warps claim items from an atomic counter over the plan's
//    compact item list; lane 0 runs a ring of TMA stages ahead of the warp's
//    compute across item boundaries.  Each item leaves one (m, l, acc) split
//    per sequence it touched; tm_merge_kernel, queued behind the attention
//    kernel as a programmatic dependent launch, merges them with one warp per
//    (sequence, query head).
//  * Rotation is applied to the query (R(-delta) q) whenever the RoPE segment
//    changes; the diff overlay adds DK / DV tiles through the same MMAs.
//    Calls with rotation use groups of one sequence.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr int kTmWarps = 4;
constexpr int kTmMaxIb = 32;
constexpr int kPlanMagic = 0x6b76730a;

#ifndef KVS_TM_STAGES_D128
#define KVS_TM_STAGES_D128 2
#endif
#ifndef KVS_TM_MIN_CTAS
#define KVS_TM_MIN_CTAS 3
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
struct TmLayout {
  int R, ib, n_chunks, n_groups, words;
  size_t max_entries;
  size_t off_hdr, off_items, off_shb, off_pne, off_spm, off_p1, off_p2, total;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Work-item size (blocks): about eight items per resident warp, at least
// max_blocks/64 (so one sequence never has more than ~64 splits per kind), at
// most 32 (one block-table entry per lane).
int tm_item_blocks(const kvs_pool* pool, int n_seq, int max_blocks) {
  const long long work = (long long)n_seq * pool->desc.num_kv_heads * max_blocks;
  const long long warps = (long long)pool->num_sms * KVS_TM_MIN_CTAS * kTmWarps;
  long long ib = work / (warps * 8);
  const long long min_ib = (max_blocks + 63) / 64;
  if (ib < min_ib) ib = min_ib;
  int r = 4;
  while (r < ib && r < kTmMaxIb) r <<= 1;
  return r;
}

static TmLayout tm_layout(const kvs_pool* pool, int n_seq, int max_blocks, int g, bool rope) {
  TmLayout L{};
  L.R = rope ? 1 : std::max(1, 8 / g);
  L.ib = tm_item_blocks(pool, n_seq, max_blocks);
  L.n_chunks = (max_blocks + L.ib - 1) / L.ib;
  L.n_groups = (n_seq + L.R - 1) / L.R;
  L.words = (max_blocks + 31) / 32;
  L.max_entries = (size_t)(n_seq + L.n_groups) * L.n_chunks;
  const size_t splits = (size_t)n_seq * pool->desc.num_kv_heads * L.n_chunks;
  const size_t split_bytes = splits * g * (pool->desc.head_dim + 2) * sizeof(float);
  size_t o = 0;
  L.off_hdr = o; o = align256(o + 64);
  L.off_items = o; o = align256(o + L.max_entries * sizeof(int2));
  L.off_shb = o; o = align256(o + (size_t)n_seq * L.words * 4);
  L.off_pne = o; o = align256(o + (size_t)n_seq * L.n_chunks);
  L.off_spm = o; o = align256(o + (size_t)L.n_groups * L.n_chunks);
  L.off_p1 = o; o = align256(o + split_bytes);
  L.off_p2 = o; o = align256(o + (L.R > 1 ? split_bytes : 0));
  L.total = o;
  return L;
}

size_t tm_workspace_bytes(const kvs_pool* pool, int n_seq, int max_blocks, int g) {
  // sized for grouping (no rotation), which is the larger layout
  return tm_layout(pool, n_seq, max_blocks, g, false).total + 256;
}

// ------------------------------------------------------------------- plan
struct PlanParams {
  const int32_t* block_table;
  const int32_t* seq_len;
  const int32_t* diff_table;
  int* hdr;
  int2* items;
  uint32_t* shb;
  uint8_t* pne;
  uint8_t* spm;
  int n_seq, max_blocks, R, G, ib, n_chunks, n_groups, words, capacity, diff_capacity, hkv;
};

__device__ __forceinline__ int plan_seq_blocks(const int32_t* seq_len, int a, int max_blocks) {
  int L = seq_len[a];
  if (L < 0) L = 0;
  if (L > max_blocks * 16) L = max_blocks * 16;
  return (L + 15) / 16;
}

// One CTA of 1024 threads builds the whole plan (it depends on the tables
// only, so one plan serves every layer of a decode step).
__global__ void __launch_bounds__(1024) tm_plan_kernel(PlanParams pp) {
  __shared__ int warp_sums[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < pp.n_seq * pp.words; i += nt) pp.shb[i] = 0u;
  __syncthreads();
  // 1. group-shared blocks: the same valid physical block for every member
  //    that reaches b (at least two), full blocks only, no mirror diff
  if (pp.R > 1) {
    for (int i = tid; i < pp.n_groups * pp.max_blocks; i += nt) {
      const int gi = i / pp.max_blocks, b = i - gi * pp.max_blocks;
      int cnt = 0, phys = -1;
      bool ok = true;
      uint32_t mask = 0;
      for (int r = 0; r < pp.R; ++r) {
        const int a = gi * pp.R + r;
        if (a >= pp.n_seq) break;
        const int L = min(max(pp.seq_len[a], 0), pp.max_blocks * 16);
        if (b * 16 >= L) continue;
        const int ph = pp.block_table[(size_t)a * pp.max_blocks + b];
        const bool full = (b + 1) * 16 <= L;
        const int d = pp.diff_table ? pp.diff_table[(size_t)a * pp.max_blocks + b] : -1;
        if (!full || d >= 0 || ph < 0 || ph >= pp.capacity) ok = false;
        if (cnt == 0) phys = ph;
        else if (ph != phys) ok = false;
        ++cnt;
        mask |= 1u << r;
      }
      if (ok && cnt >= 2)
        for (int r = 0; r < pp.R; ++r)
          if ((mask >> r) & 1u) atomicOr(pp.shb + (size_t)(gi * pp.R + r) * pp.words + (b >> 5), 1u << (b & 31));
    }
  }
  __syncthreads();
  // 2. chunk occupancy: private chunks with unshared work; shared-chunk
  //    participation per member
  for (int i = tid; i < pp.n_seq * pp.n_chunks; i += nt) {
    const int a = i / pp.n_chunks, c = i - a * pp.n_chunks;
    const int nb = plan_seq_blocks(pp.seq_len, a, pp.max_blocks);
    int any_priv = 0;
    for (int b = c * pp.ib; b < min((c + 1) * pp.ib, nb); ++b)
      any_priv |= !((pp.shb[(size_t)a * pp.words + (b >> 5)] >> (b & 31)) & 1u);
    pp.pne[i] = (uint8_t)any_priv;
  }
  for (int i = tid; i < pp.n_groups * pp.n_chunks; i += nt) {
    const int gi = i / pp.n_chunks, c = i - gi * pp.n_chunks;
    uint32_t m = 0;
    for (int r = 0; r < pp.R; ++r) {
      const int a = gi * pp.R + r;
      if (a >= pp.n_seq) break;
      const int nb = plan_seq_blocks(pp.seq_len, a, pp.max_blocks);
      for (int b = c * pp.ib; b < min((c + 1) * pp.ib, nb); ++b)
        if ((pp.shb[(size_t)a * pp.words + (b >> 5)] >> (b & 31)) & 1u) {
          m |= 1u << r;
          break;
        }
    }
    pp.spm[i] = (uint8_t)m;
  }
  __syncthreads();
  // 3. compact item list: shared items (group, chunk) first, then private
  //    items (sequence, chunk), chunk-major
  const int n_sh = pp.n_groups * pp.n_chunks, n_pr = pp.n_seq * pp.n_chunks;
  const int total = n_sh + n_pr;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  for (int base = 0; base < total; base += nt) {
    const int i = base + tid;
    int keep = 0;
    int2 item = make_int2(0, 0);
    if (i < n_sh) {
      const int c = i / pp.n_groups, gi = i - c * pp.n_groups;
      keep = pp.spm[gi * pp.n_chunks + c] != 0;
      item = make_int2((1 << 30) | gi, c);
    } else if (i < total) {
      const int j = i - n_sh;
      const int c = j / pp.n_seq, a = j - c * pp.n_seq;
      keep = pp.pne[a * pp.n_chunks + c];
      item = make_int2(a, c);
    }
    int x = keep;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int pos = s_carry + x - keep + (warp ? warp_sums[warp - 1] : 0);
    if (keep) pp.items[pos] = item;
    __syncthreads();
    if (tid == nt - 1) s_carry = pos + keep;
    __syncthreads();
  }
  if (tid == 0) {
    pp.hdr[0] = s_carry;
    pp.hdr[1] = kPlanMagic;
    pp.hdr[2] = pp.n_seq;
    pp.hdr[3] = pp.max_blocks;
    pp.hdr[4] = pp.R;
    pp.hdr[5] = pp.ib;
    pp.hdr[6] = pp.hkv;
  }
}

// -------------------------------------------------------------- attention
struct TmParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_len;
  const int32_t* diff_table;
  const int32_t* rope_off;
  const int4* rope_segs;
  float* out;
  float* p1;          // private splits [n_seq][hkv][n_chunks][g][D]
  float* p1_ml;       // [n_seq][hkv][n_chunks][g][2]
  float* p2;          // shared splits, same shape
  float* p2_ml;
  const int* hdr;
  const int2* items;
  const uint32_t* shb;
  const uint8_t* pne;
  const uint8_t* spm;
  int32_t* sched;     // [0] work counter, [1] finished-warp counter
  uint32_t* status;
  int max_blocks, n_seq, hkv, g, hq, ib, n_chunks, R, capacity, diff_capacity, total_warps, words;
  float scale_log2;
  RopeSplit rs;
};

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <int D, bool DIFF, bool ROPE>
__global__ void __launch_bounds__(128, KVS_TM_MIN_CTAS)
attn_tm_kernel(const __grid_constant__ TmParams p, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdk,
               const __grid_constant__ CUtensorMap tdv) {
  constexpr int B = 16, TILE = B * D * 2, KS = D / 16;
  constexpr int S = tm_stages<D>();
  constexpr int STAGE = 2 * TILE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kTmWarps][S];
  __shared__ int st_item[kTmWarps][S];
  // block index; bit 30: the next position holds the block's diff tiles;
  // bit 29: the block id was out of range and nothing was loaded
  __shared__ int st_block[kTmWarps][S];
  __shared__ int st_mask[kTmWarps][S];   // group members whose columns take this block

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // a merge kernel queued behind this one (programmatic dependent launch) may
  // be scheduled now; it waits for this grid to complete before reading
  asm volatile("griddepcontrol.launch_dependents;");
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* wbase = base + warp * S * STAGE;
  const uint32_t wbase_u32 = smem_u32(wbase);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // empty contexts produce zero output (they have no work items)
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < (size_t)p.n_seq * p.hq * D;
       e += (size_t)gridDim.x * blockDim.x)
    if (p.seq_len[e / ((size_t)p.hq * D)] <= 0) p.out[e] = 0.f;

  // the plan must have been built for this call's shapes
  const bool plan_ok = p.hdr[1] == kPlanMagic && p.hdr[2] == p.n_seq && p.hdr[3] == p.max_blocks &&
                       p.hdr[4] == p.R && p.hdr[5] == p.ib && p.hdr[6] == p.hkv;
  if (!plan_ok && threadIdx.x == 0 && blockIdx.x == 0) set_err(p.status, KVS_DEVERR_PLAN);
  const int n_claims = plan_ok ? p.hdr[0] * p.hkv : 0;
  const int R = p.R;
  auto seq_blocks = [&](int a) {
    int L = p.seq_len[a];
    if (L < 0 || L > p.max_blocks * B) L = L < 0 ? 0 : p.max_blocks * B;
    return (L + B - 1) / B;
  };

  // ------------------------------------------ producer state (warp-uniform)
  // The whole warp runs the producer logic; lane 0 alone issues the atomics
  // and the TMA copies.  When an item is claimed, lane j loads what block
  // b0 + j of the item needs (physical id, diff id, sharing), so issuing a
  // block costs shuffles instead of global loads.
  int p_claim = -1, p_kind = 0, p_h = 0, p_b = 0, p_b0 = 0, p_bend = 0, p_mask = 0;
  int tab_ent = -1, dif_ent = -1, aux_ent = 0;
  bool p_done = false;
  auto claim = [&]() {
    while (true) {
      int id = 0;
      if (lane == 0) id = atomicAdd(p.sched, 1);
      id = __shfl_sync(0xffffffffu, id, 0);
      if (id >= n_claims) {
        p_done = true;
        return;
      }
      const int2 it = p.items[id / p.hkv];
      const int h = id - (id / p.hkv) * p.hkv;
      const int b0 = it.y * p.ib;
      p_claim = id; p_h = h; p_b = b0; p_b0 = b0;
      if (it.x >> 30) {   // shared item of group it.x & mask
        const int gi = it.x & ((1 << 30) - 1);
        p_kind = 1;
        int nbmax = 0;
        for (int r = 0; r < R; ++r)
          if (gi * R + r < p.n_seq) nbmax = max(nbmax, seq_blocks(gi * R + r));
        p_bend = min(b0 + p.ib, nbmax);
        const int b = b0 + lane;
        int msk = 0, ph = -1;
        if (b < p_bend) {
          for (int r = 0; r < R; ++r) {
            const int a = gi * R + r;
            if (a >= p.n_seq) break;
            if ((p.shb[(size_t)a * p.words + (b >> 5)] >> (b & 31)) & 1u) {
              msk |= 1 << r;
              ph = p.block_table[(size_t)a * p.max_blocks + b];
            }
          }
        }
        tab_ent = ph;
        aux_ent = msk;
        dif_ent = -1;
      } else {           // private item of sequence it.x
        const int a = it.x;
        p_kind = 0;
        p_bend = min(b0 + p.ib, seq_blocks(a));
        p_mask = 1 << (a % R);
        const int b = b0 + lane;
        const bool in = b < p_bend;
        tab_ent = in ? __ldg(p.block_table + (size_t)a * p.max_blocks + b) : -1;
        aux_ent = in ? (int)((p.shb[(size_t)a * p.words + (b >> 5)] >> (b & 31)) & 1u) : 1;   // 1 = skip
        if (DIFF) dif_ent = in ? __ldg(p.diff_table + (size_t)a * p.max_blocks + b) : -1;
      }
      return;
    }
  };
  int pend_drow = -1;   // a diff tile pair still to issue for the last block
  auto issue = [&](int s) {   // whole warp; lane 0 issues
    uint64_t* bar = &bars[warp][s];
    uint8_t* st = wbase + s * STAGE;
    if (DIFF && pend_drow >= 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, 2 * TILE);
        tma_load_kv_tile<D>(st, &tdk, pend_drow, bar);
        tma_load_kv_tile<D>(st + TILE, &tdv, pend_drow, bar);
      }
      pend_drow = -1;
      return;
    }
    int phys = -1, did = -1, mask = 0, b = 0;
    while (true) {
      if (!p_done && p_b >= p_bend) claim();
      if (p_done) break;
      const int j = p_b - p_b0;
      b = p_b++;
      const int ent = __shfl_sync(0xffffffffu, tab_ent, j);
      const int aux = __shfl_sync(0xffffffffu, aux_ent, j);
      if (p_kind == 0) {
        if (aux) continue;          // computed by the group's shared item
        mask = p_mask;
        if (DIFF) did = __shfl_sync(0xffffffffu, dif_ent, j);
      } else {
        if (aux == 0) continue;     // not shared at this block
        mask = aux;
      }
      phys = ent;
      break;
    }
    if (p_done) {
      if (lane == 0) {
        st_item[warp][s] = -1;
        mbar_arrive(bar);
      }
      return;
    }
    const bool valid = phys >= 0 && phys < p.capacity;
    const bool dval = DIFF && valid && did >= 0 && did < p.diff_capacity;
    if (dval) pend_drow = (did * p.hkv + p_h) * B;
    if (lane != 0) return;
    st_item[warp][s] = p_claim;
    st_mask[warp][s] = mask;
    if (!valid) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      st_block[warp][s] = b | (1 << 29);   // nothing loaded: skip this block
      mbar_arrive(bar);
      return;
    }
    if (DIFF && did >= p.diff_capacity) set_err(p.status, KVS_DEVERR_DIFF_ID);
    st_block[warp][s] = dval ? (b | (1 << 30)) : b;
    mbar_arrive_expect_tx(bar, 2 * TILE);
    const int row = (phys * p.hkv + p_h) * B;
    tma_load_kv_tile<D>(st, &tk, row, bar);
    tma_load_kv_tile<D>(st + TILE, &tv, row, bar);
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
  int cur_delta = 0, seg_lo = 0, seg_hi = 0, seg_beg = 0, seg_end = 0;
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
  auto rotate_q = [&](int delta) {   // q' = R(-delta) q, as bf16 hi + lo
    q_has_lo = true;
#pragma unroll
    for (int kk = 0; kk < KS / 2; ++kk) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int col = kk * 16 + 2 * c + half * 8;
        float cs0, sn0, cs1, sn1;
        rope_cos_sin(p.rs, col, delta, cs0, sn0);
        rope_cos_sin(p.rs, col + 1, delta, cs1, sn1);
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
        const size_t it = (((size_t)a * p.hkv + ch_) * p.n_chunks + cchunk) * p.g + hh;
        float* pr = dst + it * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          __stcg(pr + mt * 16 + g, acc[mt][cc]);
          __stcg(pr + mt * 16 + g + 8, acc[mt][2 + cc]);
        }
        if (g == 0) __stcg(reinterpret_cast<float2*>(dml + it * 2), make_float2(m[cc], lt[cc]));
      }
    }
  };

  for (int i = 0;;) {
    const int s = i % S;
    if (!mbar_wait_bounded(&bars[warp][s], (i / S) & 1, p.status)) break;
    const int item = st_item[warp][s];
    const int bword = st_block[warp][s];
    const int emask = st_mask[warp][s];
    if (item < 0) break;
    const bool has_diff = DIFF && (bword >> 30) != 0;
    const int b = bword & ((1 << 29) - 1);
    const bool loaded = ((bword >> 29) & 1) == 0;
    const int s2 = (i + 1) % S;
    if (has_diff && !mbar_wait_bounded(&bars[warp][s2], ((i + 1) / S) & 1, p.status)) break;
    if (item != cur) {
      if (cur >= 0) flush();
      cur = item;
      const int2 it = p.items[item / p.hkv];
      ch_ = item - (item / p.hkv) * p.hkv;
      cchunk = it.y;
      ckind = it.x >> 30;
      cidx = it.x & ((1 << 30) - 1);
      int agent_of_col = -1;   // sequence of this lane's query column (n = g)
      if (ckind) {
        cact = p.spm[cidx * p.n_chunks + cchunk];
        const int slot = g / p.g;
        if (g < R * p.g && ((cact >> slot) & 1)) agent_of_col = cidx * R + slot;
      } else {
        const int slot = cidx % R;
        cact = 1 << slot;
        if (g / p.g == slot && g < R * p.g) agent_of_col = cidx;
      }
      qok = agent_of_col >= 0;
      qrow = p.q + ((size_t)(qok ? agent_of_col : 0) * p.hq + ch_ * p.g + (g % p.g)) * D;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int j = 2 * c + cc;
        const int slot = j / p.g;
        int a = -1;
        if (j < R * p.g && ((cact >> slot) & 1)) a = ckind ? cidx * R + slot : cidx;
        colslot[cc] = a >= 0 ? slot : 31;
        colL[cc] = a >= 0 ? min(max(p.seq_len[a], 0), p.max_blocks * B) : 0;
      }
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      load_q();
      cur_delta = 0;
      seg_lo = seg_hi = 0;
      if (ROPE) {
        seg_beg = p.rope_off[cidx];
        seg_end = p.rope_off[cidx + 1];
      }
    }
    if (loaded) {
      if (ROPE && (b < seg_lo || b >= seg_hi)) {
        // find the segment covering b; if none, the gap around b (delta 0)
        // is cached instead, so unrotated stretches are not rescanned
        int found = 0x7fffffff, fd = 0, flo = 0, fhi = 0, gap_lo = 0, gap_hi = 0x7fffffff;
        for (int e = seg_beg + lane; e < seg_end; e += 32) {
          const int4 sg = __ldg(p.rope_segs + e);
          if (b >= sg.x && b < sg.x + sg.y && e < found) {
            found = e; fd = sg.z; flo = sg.x; fhi = sg.x + sg.y;
          }
          if (sg.x > b) gap_hi = min(gap_hi, sg.x);
          if (sg.x + sg.y <= b) gap_lo = max(gap_lo, sg.x + sg.y);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const int f2 = __shfl_xor_sync(0xffffffffu, found, o);
          const int d2 = __shfl_xor_sync(0xffffffffu, fd, o);
          const int lo2 = __shfl_xor_sync(0xffffffffu, flo, o);
          const int hi2 = __shfl_xor_sync(0xffffffffu, fhi, o);
          if (f2 < found) { found = f2; fd = d2; flo = lo2; fhi = hi2; }
          gap_hi = min(gap_hi, __shfl_xor_sync(0xffffffffu, gap_hi, o));
          gap_lo = max(gap_lo, __shfl_xor_sync(0xffffffffu, gap_lo, o));
        }
        int nd = 0;
        if (found != 0x7fffffff) {
          nd = fd; seg_lo = flo; seg_hi = fhi;
        } else {
          seg_lo = gap_lo; seg_hi = gap_hi;
        }
        if (nd <= -(1 << 18) || nd >= (1 << 18)) {
          if (lane == 0) set_err(p.status, KVS_DEVERR_ROPE_RANGE);
          nd = 0;
        }
        if (nd != cur_delta) {
          if (nd == 0) load_q(); else rotate_q(nd);
          cur_delta = nd;
        }
      }
      const uint32_t tkb = wbase_u32 + s * STAGE, tvb = tkb + TILE;
      const uint32_t dkb = wbase_u32 + s2 * STAGE, dvb = dkb + TILE;   // diff tiles (if any)
      // S^T = K q^T : 16 tokens x 8 query columns, two accumulation chains
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        float* acc_s = (kk & 1) ? sd : sc;
        uint32_t a[4];
        ldsm_x4(tkb + koff[kk], a[0], a[1], a[2], a[3]);
        mma_bf16(acc_s, a, qb[kk][0], qb[kk][1]);
        if (ROPE && q_has_lo) mma_bf16(acc_s, a, qlo[ROPE ? kk : 0][0], qlo[ROPE ? kk : 0][1]);
        if (has_diff) {
          ldsm_x4(dkb + koff[kk], a[0], a[1], a[2], a[3]);
          mma_bf16(acc_s, a, qb[kk][0], qb[kk][1]);
          if (ROPE && q_has_lo) mma_bf16(acc_s, a, qlo[ROPE ? kk : 0][0], qlo[ROPE ? kk : 0][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] += sd[e];
      // sc: (t=g, col 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1); a column is live
      // if its member takes this block and the token is inside its context
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = g + ((e >> 1) << 3);
        const int cc = e & 1;
        const bool live = colslot[cc] != 31 && ((emask >> colslot[cc]) & 1) && b * B + t < colL[cc];
        sc[e] = live ? sc[e] * p.scale_log2 : -INFINITY;
      }
      float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      // a column with nothing live yet keeps (m, l, acc) = (-inf, 0, 0)
      const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m[0] - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m[1] - mn1);
      m[0] = mn0;
      m[1] = mn1;
      sc[0] = mn0 == -INFINITY ? 0.f : fast_exp2(sc[0] - mn0);
      sc[1] = mn1 == -INFINITY ? 0.f : fast_exp2(sc[1] - mn1);
      sc[2] = mn0 == -INFINITY ? 0.f : fast_exp2(sc[2] - mn0);
      sc[3] = mn1 == -INFINITY ? 0.f : fast_exp2(sc[3] - mn1);
      l[0] = l[0] * al0 + sc[0] + sc[2];
      l[1] = l[1] * al1 + sc[1] + sc[3];
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        acc[mt][0] *= al0; acc[mt][1] *= al1;
        acc[mt][2] *= al0; acc[mt][3] *= al1;
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
        if (has_diff) {
          ldsm_x4_t(dvb + voff[mt], a[0], a[1], a[2], a[3]);
          mma_bf16(acc[mt], a, bh0, bh1);
          mma_bf16(acc[mt], a, bl0, bl1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) fence_proxy_async_smem();
    issue(s);
    if (has_diff) issue(s2);
    i += has_diff ? 2 : 1;
  }
  if (cur >= 0) flush();
  // the last warp of the launch to finish resets the scheduler for the next one
  if (lane == 0) {
    __threadfence();
    const int done = atomicAdd(p.sched + 1, 1);
    if (done == p.total_warps - 1) {
      p.sched[0] = 0;
      p.sched[1] = 0;
    }
  }
}

// Split merge: one warp per (sequence, query head) row, so every row of every
// (sequence, kv head) merges in parallel, each lane keeping up to
// kMergeBatch independent split loads in flight.  The split order is fixed
// (chunk order, private then shared per 32-chunk window), so the result does
// not depend on which warp computed which split.
constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 12;   // independent split loads in flight per lane

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32, 2) tm_merge_kernel(const __grid_constant__ TmParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int CPL = D / 32;   // columns per lane
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);   // sequence * hq + query head
  if (row >= p.n_seq * p.hq) return;
  // the attention kernel has flagged a plan built for other shapes and
  // computed nothing; leave the output untouched as well
  if (!(p.hdr[1] == kPlanMagic && p.hdr[2] == p.n_seq && p.hdr[3] == p.max_blocks && p.hdr[4] == p.R &&
        p.hdr[5] == p.ib && p.hdr[6] == p.hkv))
    return;
  const int a = row / p.hq, qh = row - a * p.hq, h = qh / p.g, hh = qh - h * p.g;
  const int gi = a / p.R, slot = a - gi * p.R;
  const size_t sbase = ((size_t)a * p.hkv + h) * p.n_chunks;
  float* o = p.out + (size_t)row * D + lane * CPL;
  if (p.seq_len[a] <= 0) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) o[j] = 0.f;
    return;
  }
  // lane k owns chunks c0 + k of every 32-chunk window; the first two windows
  // keep their (m, l) in registers between the passes
  float2 cp0 = make_float2(0.f, 0.f), cs0 = cp0, cp1 = cp0, cs1 = cp0;
  bool hp0 = false, hs0 = false, hp1 = false, hs1 = false;
  auto own = [&](int c0, bool& pv, bool& sv, float2& mp, float2& ms) {
    const int ck = c0 + lane;
    pv = ck < p.n_chunks && p.pne[a * p.n_chunks + ck];
    sv = p.R > 1 && ck < p.n_chunks && ((p.spm[gi * p.n_chunks + ck] >> slot) & 1);
    mp = pv ? __ldcg(reinterpret_cast<const float2*>(p.p1_ml + ((sbase + ck) * p.g + hh) * 2)) : make_float2(0.f, 0.f);
    ms = sv ? __ldcg(reinterpret_cast<const float2*>(p.p2_ml + ((sbase + ck) * p.g + hh) * 2)) : make_float2(0.f, 0.f);
  };
  float M = -INFINITY;
  for (int c0 = 0, w = 0; c0 < p.n_chunks; c0 += 32, ++w) {
    bool pv, sv;
    float2 mp, ms;
    own(c0, pv, sv, mp, ms);
    if (pv && mp.y > 0.f) M = fmaxf(M, mp.x);
    if (sv && ms.y > 0.f) M = fmaxf(M, ms.x);
    if (w == 0) {
      hp0 = pv; hs0 = sv; cp0 = mp; cs0 = ms;
    } else if (w == 1) {
      hp1 = pv; hs1 = sv; cp1 = mp; cs1 = ms;
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float Ls = 0.f, v[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) v[j] = 0.f;
  for (int c0 = 0, w = 0; c0 < p.n_chunks; c0 += 32, ++w) {
    bool pv, sv;
    float2 mp, ms;
    if (w == 0) {
      pv = hp0; sv = hs0; mp = cp0; ms = cs0;
    } else if (w == 1) {
      pv = hp1; sv = hs1; mp = cp1; ms = cs1;
    } else {
      own(c0, pv, sv, mp, ms);
    }
    const float wp = pv && mp.y > 0.f ? fast_exp2(mp.x - M) : 0.f;
    const float ws = sv && ms.y > 0.f ? fast_exp2(ms.x - M) : 0.f;
    Ls += wp * mp.y + ws * ms.y;
#pragma unroll
    for (int kind = 0; kind < 2; ++kind) {
      const float* P = kind ? p.p2 : p.p1;
      const float wk = kind ? ws : wp;
      unsigned mk = __ballot_sync(0xffffffffu, kind ? sv : pv);
      while (mk) {   // warp-uniform
        int idx[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          idx[u] = -1;
          if (mk) {
            idx[u] = __ffs(mk) - 1;
            mk &= mk - 1;
          }
        }
        float x[kMergeBatch][CPL];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (idx[u] < 0) continue;
          const float* src = P + ((sbase + c0 + idx[u]) * p.g + hh) * D + lane * CPL;
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
          if (idx[u] < 0) continue;
          const float wgt = __shfl_sync(0xffffffffu, wk, idx[u]);
#pragma unroll
          for (int j = 0; j < CPL; ++j) v[j] += wgt * x[u][j];
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
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
  cfg.gridDim = dim3((rows + kMergeWarps - 1) / kMergeWarps);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tm_merge_kernel<D>, prm) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_attn: merge launch failed");
  count_launch();
  return check_launch("decode_attn_merge");
}

template <int D, bool DIFF, bool ROPE>
static kvs_status launch_tm(TmParams& prm, const kvs_pool* pool, int layer, int max_claims, cudaStream_t st) {
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
  // largest possible number of claims (idle warps would only contend)
  const int grid = std::max(1, std::min(pool->num_sms * blocks_per_sm, (max_claims + kTmWarps - 1) / kTmWarps));
  prm.total_warps = grid * kTmWarps;
  const CUtensorMap& dk = DIFF ? pool->tdk[layer] : pool->tk[layer];
  const CUtensorMap& dv = DIFF ? pool->tdv[layer] : pool->tv[layer];
  kern<<<grid, 128, smem, st>>>(prm, pool->tk[layer], pool->tv[layer], dk, dv);
  count_launch();
  const kvs_status s = check_launch("decode_attn");
  if (s != KVS_OK) return s;
  return launch_merge<D>(prm, st);
}

kvs_status decode_plan_token_major(kvs_pool* pool, int n_q_heads, const int32_t* table, int max_blocks,
                                   const int32_t* seq_len, int n_seq, const int32_t* diff, bool rope, void* ws,
                                   cudaStream_t stream) {
  const int g = n_q_heads / pool->desc.num_kv_heads;
  const TmLayout L = tm_layout(pool, n_seq, max_blocks, g, rope);
  uint8_t* w = static_cast<uint8_t*>(ws);
  PlanParams pp{};
  pp.block_table = table;
  pp.seq_len = seq_len;
  pp.diff_table = diff;
  pp.hdr = reinterpret_cast<int*>(w + L.off_hdr);
  pp.items = reinterpret_cast<int2*>(w + L.off_items);
  pp.shb = reinterpret_cast<uint32_t*>(w + L.off_shb);
  pp.pne = w + L.off_pne;
  pp.spm = w + L.off_spm;
  pp.n_seq = n_seq;
  pp.max_blocks = max_blocks;
  pp.R = L.R;
  pp.G = g;
  pp.ib = L.ib;
  pp.n_chunks = L.n_chunks;
  pp.n_groups = L.n_groups;
  pp.words = L.words;
  pp.capacity = pool->desc.capacity_blocks;
  pp.diff_capacity = pool->desc.diff_capacity_blocks;
  pp.hkv = pool->desc.num_kv_heads;
  tm_plan_kernel<<<1, 1024, 0, stream>>>(pp);
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
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t splits = (size_t)n_seq * d.num_kv_heads * L.n_chunks;
  TmParams prm{};
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = table;
  prm.seq_len = seq_len;
  prm.diff_table = diff;
  prm.rope_off = rope_off;
  prm.rope_segs = reinterpret_cast<const int4*>(rope_segs);
  prm.out = out;
  prm.p1 = reinterpret_cast<float*>(w + L.off_p1);
  prm.p1_ml = prm.p1 + splits * g * d.head_dim;
  prm.p2 = reinterpret_cast<float*>(w + L.off_p2);
  prm.p2_ml = prm.p2 + (L.R > 1 ? splits * g * d.head_dim : 0);
  prm.hdr = reinterpret_cast<const int*>(w + L.off_hdr);
  prm.items = reinterpret_cast<const int2*>(w + L.off_items);
  prm.shb = reinterpret_cast<const uint32_t*>(w + L.off_shb);
  prm.pne = w + L.off_pne;
  prm.spm = w + L.off_spm;
  prm.sched = pool->sched;
  prm.status = pool->status;
  prm.max_blocks = max_blocks;
  prm.n_seq = n_seq;
  prm.hkv = d.num_kv_heads;
  prm.g = g;
  prm.hq = n_q_heads;
  prm.ib = L.ib;
  prm.n_chunks = L.n_chunks;
  prm.R = L.R;
  prm.words = L.words;
  prm.capacity = d.capacity_blocks;
  prm.diff_capacity = d.diff_capacity_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  if (rope) rope_split_host(theta, d.head_dim, prm.rs.c);
  const int max_claims = (int)std::min<size_t>(L.max_entries * d.num_kv_heads, 0x7fffffff);
  if (d.head_dim == 128) {
    if (dif) return rope ? launch_tm<128, true, true>(prm, pool, layer, max_claims, stream)
                         : launch_tm<128, true, false>(prm, pool, layer, max_claims, stream);
    return rope ? launch_tm<128, false, true>(prm, pool, layer, max_claims, stream)
                : launch_tm<128, false, false>(prm, pool, layer, max_claims, stream);
  }
  if (dif) return rope ? launch_tm<64, true, true>(prm, pool, layer, max_claims, stream)
                       : launch_tm<64, true, false>(prm, pool, layer, max_claims, stream);
  return rope ? launch_tm<64, false, true>(prm, pool, layer, max_claims, stream)
              : launch_tm<64, false, false>(prm, pool, layer, max_claims, stream);
}

}  // namespace kvs
