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
//    the <= 8 query heads of a KV head are the N dimension: S^T = K q^T and
//    O^T = V^T P^T.  K is the A operand straight from shared memory
//    (ldmatrix), V^T too (ldmatrix.trans); P^T reaches the B operand through
//    movmatrix.  Per 16-token block this is 8 + 16 MMAs (P enters as a bf16
//    hi + lo pair) instead of padding the query group to 16 rows.
//  * Persistent warps: the grid fills every SM once; each warp claims work
//    items (sequence, kv head, run of IB logical blocks) from an atomic
//    counter in chunk-major, sequence-minor order, so the sequences sharing a
//    prefix stream the same physical blocks at about the same time and L2
//    serves the repeats.  Lane 0 runs ahead of the warp's own compute through
//    a ring of S TMA stages, claiming the next item as soon as it has issued
//    the current one, so the pipeline never drains between items.
//  * Each item leaves an (m, l, acc) split; the last warp to finish a
//    (sequence, kv head) merges its splits (arrival counter, no spinning).
//  * Rotation is applied to the query (R(-delta) q, as a bf16 hi + lo pair)
//    whenever the RoPE segment changes; the diff overlay adds DK / DV tiles
//    through the same MMAs (linearity).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace kvs {

struct TmParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_len;
  const int32_t* diff_table;
  const int32_t* rope_off;
  const int4* rope_segs;
  float* out;
  float* part;       // [n_items][g][D]
  float* part_ml;    // [n_items][g][2]
  int32_t* tickets;  // [n_seq * hkv]
  int32_t* sched;    // [0] work counter, [1] finished-warp counter
  uint32_t* status;
  int max_blocks, n_seq, hkv, g, hq, ib, n_chunks, n_items, capacity, diff_capacity, total_warps;
  float scale_log2;
  RopeSplit rs;
};

constexpr int kTmWarps = 4;

// Ring stages per warp.  A stage holds one block's K and V tiles; a block
// that carries a mirror diff takes two consecutive positions (K/V, then
// DK/DV), so diff blocks need no larger stages.
#ifndef KVS_TM_STAGES_D128
#define KVS_TM_STAGES_D128 2
#endif
#ifndef KVS_TM_MIN_CTAS
#define KVS_TM_MIN_CTAS 3
#endif
template <int D, bool DIFF>
__host__ __device__ constexpr int tm_stages() {
  return DIFF ? 3 : (D == 128 ? KVS_TM_STAGES_D128 : 4);
}

template <int D, bool DIFF>
__host__ __device__ constexpr int tm_smem_bytes() {
  return 1024 + kTmWarps * tm_stages<D, DIFF>() * 2 * (16 * D * 2);
}


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
  constexpr int S = tm_stages<D, DIFF>();
  constexpr int STAGE = 2 * TILE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[kTmWarps][S];
  __shared__ int st_item[kTmWarps][S];
  // block index; bit 30: the next position holds the block's diff tiles;
  // bit 29: the block id was out of range and nothing was loaded
  __shared__ int st_block[kTmWarps][S];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* wbase = base + warp * S * STAGE;
  const uint32_t wbase_u32 = smem_u32(wbase);
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ------------------------------------------ producer state (warp-uniform)
  // The whole warp runs the producer logic; lane 0 alone issues the atomics
  // and the TMA copies.  When an item is claimed, lane j loads the item's
  // j-th block-table (and diff-table) entry once, so issuing a block costs a
  // shuffle instead of a global load.
  int p_item = -1, p_a = 0, p_h = 0, p_b = 0, p_b0 = 0, p_bend = 0;
  int tab_ent = -1, dif_ent = -1;
  bool p_done = false;
  auto seq_blocks = [&](int a) {
    int L = p.seq_len[a];
    if (L < 0 || L > p.max_blocks * B) L = L < 0 ? 0 : p.max_blocks * B;
    return (L + B - 1) / B;
  };
  auto claim = [&]() {
    while (true) {
      int id = 0;
      if (lane == 0) id = atomicAdd(p.sched, 1);
      id = __shfl_sync(0xffffffffu, id, 0);
      if (id >= p.n_items) {
        p_done = true;
        return;
      }
      const int a = id % p.n_seq, rest = id / p.n_seq;
      const int h = rest % p.hkv, ch = rest / p.hkv;
      const int Lr = p.seq_len[a];
      if (lane == 0 && ch == 0 && (Lr < 0 || Lr > p.max_blocks * B)) set_err(p.status, KVS_DEVERR_SEQ_LEN);
      const int nb = seq_blocks(a);
      if (nb == 0) {
        if (ch == 0)
          for (int i = lane; i < p.g * D; i += 32) p.out[((size_t)a * p.hq + h * p.g) * D + i] = 0.f;
        continue;
      }
      const int b0 = ch * p.ib;
      if (b0 >= nb) continue;
      p_item = id; p_a = a; p_h = h; p_b = b0; p_b0 = b0; p_bend = min(b0 + p.ib, nb);
      tab_ent = lane < p_bend - b0 ? __ldg(p.block_table + (size_t)a * p.max_blocks + b0 + lane) : -1;
      if (DIFF) dif_ent = lane < p_bend - b0 ? __ldg(p.diff_table + (size_t)a * p.max_blocks + b0 + lane) : -1;
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
    if (!p_done && p_b >= p_bend) claim();
    if (p_done) {
      if (lane == 0) {
        st_item[warp][s] = -1;
        mbar_arrive(bar);
      }
      return;
    }
    const int b = p_b++;
    const int phys = __shfl_sync(0xffffffffu, tab_ent, b - p_b0);
    const int did = DIFF ? __shfl_sync(0xffffffffu, dif_ent, b - p_b0) : -1;
    if (lane != 0) {
      if (DIFF && phys >= 0 && phys < p.capacity && did >= 0 && did < p.diff_capacity)
        pend_drow = (did * p.hkv + p_h) * B;
      return;
    }
    st_item[warp][s] = p_item;
    st_block[warp][s] = b;
    if (phys < 0 || phys >= p.capacity) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      st_block[warp][s] = b | (1 << 29);   // nothing loaded: skip this block
      mbar_arrive(bar);
      return;
    }
    if (DIFF) {
      if (did >= p.diff_capacity) {
        set_err(p.status, KVS_DEVERR_DIFF_ID);
      } else if (did >= 0) {
        st_block[warp][s] = b | (1 << 30);
        pend_drow = (did * p.hkv + p_h) * B;
      }
    }
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
  int cur = -1, ca = 0, ch_ = 0, cL = 0;
  float m[2], l[2], acc[D / 16][4];
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

  // write the current item's split, count it, merge if this was the last one
  auto flush = [&]() {
    float lt0 = l[0], lt1 = l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
    }
    float* pr = p.part + (size_t)cur * p.g * D;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int r = 2 * c + cc;
      if (r < p.g) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          __stcg(pr + r * D + mt * 16 + g, acc[mt][cc]);
          __stcg(pr + r * D + mt * 16 + g + 8, acc[mt][2 + cc]);
        }
        if (g == 0) __stcg(reinterpret_cast<float2*>(p.part_ml + ((size_t)cur * p.g + r) * 2), make_float2(m[cc], cc ? lt1 : lt0));
      }
    }
    __syncwarp();
    const int nb = seq_blocks(ca);
    const int nch = (nb + p.ib - 1) / p.ib;
    int last = 0;
    if (lane == 0) {
      __threadfence();   // the warp's split stores (ordered by __syncwarp) before the arrival
      const int t = atomicAdd(p.tickets + ca * p.hkv + ch_, 1);
      last = (t == nch - 1);
      if (last) p.tickets[ca * p.hkv + ch_] = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();   // acquire side: other warps' splits are visible
    // merge the nch splits of (ca, ch_): chunk k's split is item ((k*hkv + ch_)*n_seq + ca).
    // Lanes first take one split each for the max and the normaliser; then
    // every lane owns D/32 consecutive columns and walks the splits with
    // several independent loads in flight.
    constexpr int CPL = D / 32;                 // columns per lane
    const size_t kstride = (size_t)p.hkv * p.n_seq;
    const size_t it0 = (size_t)ch_ * p.n_seq + ca;
    for (int r = 0; r < p.g; ++r) {
      float M = -INFINITY;
      for (int k = lane; k < nch; k += 32) M = fmaxf(M, __ldcg(p.part_ml + ((it0 + k * kstride) * p.g + r) * 2));
#pragma unroll
      for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float Ls = 0.f;
      float v[CPL];
#pragma unroll
      for (int j = 0; j < CPL; ++j) v[j] = 0.f;
      // no shuffles in this loop: every lane reads the (m, l) of split k
      // itself (one broadcast transaction), so the loads of several splits
      // can be in flight at once
#pragma unroll 8
      for (int k = 0; k < nch; ++k) {
        const size_t it = (it0 + k * kstride) * p.g + r;
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + it * 2));
        const float* src = p.part + it * D + lane * CPL;
        float x[CPL];
        if (CPL == 4) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
          x[0] = t.x; x[1 % CPL] = t.y; x[2 % CPL] = t.z; x[3 % CPL] = t.w;
        } else {
          const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
          x[0] = t.x; x[1 % CPL] = t.y;
        }
        const float wgt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
        Ls += wgt * ml.y;
#pragma unroll
        for (int j = 0; j < CPL; ++j) v[j] += wgt * x[j];
      }
      float* o = p.out + ((size_t)ca * p.hq + ch_ * p.g + r) * D + lane * CPL;
#pragma unroll
      for (int j = 0; j < CPL; ++j) o[j] = Ls > 0.f ? v[j] / Ls : 0.f;
    }
  };

  for (int i = 0;;) {
    const int s = i % S;
    if (!mbar_wait_bounded(&bars[warp][s], (i / S) & 1, p.status)) break;
    const int item = st_item[warp][s];
    const int bword = st_block[warp][s];
    if (item < 0) break;
    const bool has_diff = DIFF && (bword >> 30) != 0;
    const int b = bword & ((1 << 29) - 1);
    const bool loaded = ((bword >> 29) & 1) == 0;
    const int s2 = (i + 1) % S;
    if (has_diff && !mbar_wait_bounded(&bars[warp][s2], ((i + 1) / S) & 1, p.status)) break;
    if (item != cur) {
      if (cur >= 0) flush();
      cur = item;
      ca = item % p.n_seq;
      ch_ = (item / p.n_seq) % p.hkv;
      int L = p.seq_len[ca];
      cL = L < 0 ? 0 : min(L, p.max_blocks * B);
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      qok = g < p.g;
      qrow = p.q + ((size_t)ca * p.hq + ch_ * p.g + g) * D;
      load_q();
      cur_delta = 0;
      seg_lo = seg_hi = 0;
      if (ROPE) {
        seg_beg = p.rope_off[ca];
        seg_end = p.rope_off[ca + 1];
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
      // S^T = K q^T : 16 tokens x 8 query heads
      // two independent accumulation chains (even / odd k-steps)
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
      const int nv = min(B, cL - b * B);
      // sc: (t=g, r=2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = g + ((e >> 1) << 3);
        sc[e] = t < nv ? sc[e] * p.scale_log2 : -INFINITY;
      }
      float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
      m[0] = mn0;
      m[1] = mn1;
      sc[0] = fast_exp2(sc[0] - mn0);
      sc[1] = fast_exp2(sc[1] - mn1);
      sc[2] = fast_exp2(sc[2] - mn0);
      sc[3] = fast_exp2(sc[3] - mn1);
      l[0] = l[0] * al0 + sc[0] + sc[2];
      l[1] = l[1] * al1 + sc[1] + sc[3];
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        acc[mt][0] *= al0; acc[mt][1] *= al1;
        acc[mt][2] *= al0; acc[mt][3] *= al1;
      }
      // P^T as the B operand (k = token, n = query head), bf16 hi + lo
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

template <int D, bool DIFF, bool ROPE>
static kvs_status launch_tm(TmParams& prm, const kvs_pool* pool, int layer, cudaStream_t st) {
  auto kern = attn_tm_kernel<D, DIFF, ROPE>;
  constexpr int smem = tm_smem_bytes<D, DIFF>();
  static int blocks_per_sm = 0;
  if (!blocks_per_sm) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kern, 128, smem) != cudaSuccess ||
        blocks_per_sm < 1)
      return fail(KVS_ERR_CUDA, "decode_attn: cannot configure the token-major kernel");
  }
  // persistent grid: every SM filled once, but never more warps than items
  // (idle warps would only contend on the work counter)
  const int grid = std::max(1, std::min(pool->num_sms * blocks_per_sm, (prm.n_items + kTmWarps - 1) / kTmWarps));
  prm.total_warps = grid * kTmWarps;
  const CUtensorMap& dk = DIFF ? pool->tdk[layer] : pool->tk[layer];
  const CUtensorMap& dv = DIFF ? pool->tdv[layer] : pool->tv[layer];
  kern<<<grid, 128, smem, st>>>(prm, pool->tk[layer], pool->tv[layer], dk, dv);
  count_launch();
  return check_launch("decode_attn");
}

// Work-item size (blocks): about eight items per resident warp so the dynamic
// schedule balances ragged contexts, but at least max_blocks/64 so one
// (sequence, kv head) never has more than ~64 splits to merge, and at most
// 32 (one block-table entry per lane).
int tm_item_blocks(const kvs_pool* pool, int n_seq, int max_blocks) {
  const long long work = (long long)n_seq * pool->desc.num_kv_heads * max_blocks;
  const long long warps = (long long)pool->num_sms * KVS_TM_MIN_CTAS * kTmWarps;
  long long ib = work / (warps * 8);
  const long long min_ib = (max_blocks + 63) / 64;
  if (ib < min_ib) ib = min_ib;
  int r = 4;
  while (r < ib && r < 32) r <<= 1;
  return r;
}

kvs_status decode_attn_token_major(kvs_pool* pool, int layer, const void* q, int n_q_heads, const int32_t* table,
                                   int max_blocks, const int32_t* seq_len, int n_seq, const int32_t* diff,
                                   const int32_t* rope_off, const kvs_seg_rope* rope_segs, float theta,
                                   float scale, float* out, void* ws, cudaStream_t stream) {
  const kvs_pool_desc& d = pool->desc;
  const int g = n_q_heads / d.num_kv_heads;
  TmParams prm{};
  prm.q = static_cast<const uint16_t*>(q);
  prm.block_table = table;
  prm.seq_len = seq_len;
  prm.diff_table = diff;
  prm.rope_off = rope_off;
  prm.rope_segs = reinterpret_cast<const int4*>(rope_segs);
  prm.out = out;
  prm.ib = tm_item_blocks(pool, n_seq, max_blocks);
  prm.n_chunks = (max_blocks + prm.ib - 1) / prm.ib;
  prm.n_items = n_seq * d.num_kv_heads * prm.n_chunks;
  prm.part = static_cast<float*>(ws);
  prm.part_ml = prm.part + (size_t)prm.n_items * g * d.head_dim;
  prm.tickets = pool->tickets;
  prm.sched = pool->sched;
  prm.status = pool->status;
  prm.max_blocks = max_blocks;
  prm.n_seq = n_seq;
  prm.hkv = d.num_kv_heads;
  prm.g = g;
  prm.hq = n_q_heads;
  prm.capacity = d.capacity_blocks;
  prm.diff_capacity = d.diff_capacity_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const bool rope = rope_off != nullptr, dif = diff != nullptr;
  if (rope) rope_split_host(theta, d.head_dim, prm.rs.c);
  if (d.head_dim == 128) {
    if (dif) return rope ? launch_tm<128, true, true>(prm, pool, layer, stream) : launch_tm<128, true, false>(prm, pool, layer, stream);
    return rope ? launch_tm<128, false, true>(prm, pool, layer, stream) : launch_tm<128, false, false>(prm, pool, layer, stream);
  }
  if (dif) return rope ? launch_tm<64, true, true>(prm, pool, layer, stream) : launch_tm<64, true, false>(prm, pool, layer, stream);
  return rope ? launch_tm<64, false, true>(prm, pool, layer, stream) : launch_tm<64, false, false>(prm, pool, layer, stream);
}

size_t tm_workspace_bytes(const kvs_pool* pool, int n_seq, int max_blocks, int g) {
  const int ib = tm_item_blocks(pool, n_seq, max_blocks);
  const size_t items = (size_t)n_seq * pool->desc.num_kv_heads * ((max_blocks + ib - 1) / ib);
  return items * g * (pool->desc.head_dim + 2) * sizeof(float) + 256;
}

}  // namespace kvs
