// Wide shared tile: decode attention of a whole sharing group over the blocks
// its members share, on the fifth-generation tensor cores.
//
// What it computes is one split per (member, query head) of a shared chunk:
// m = max_t s_t, l = sum_t 2^(s_t - m), acc = sum_t 2^(s_t - m) V_t with
// s_t = scale * log2(e) * <q, K_t> (MemDecay post §4.2 weighting; INMS
// walkthrough §6.1: attention work on a common prefix done once for all
// agents that share it).  The split merge combines it with the private
// splits exactly as the token-major kernel's.
//
// GB300 layout of the work:
//  * A group holds W = min(32, 128 / G) sequences; its W * G query rows are
//    the M = 128 rows of tcgen05 MMAs (row r = member r / G, head r % G of
//    the KV head).  A sub-tile is 8 logical blocks (128 tokens), staged by
//    TMA as [64-column half][token][64] with the 128-byte swizzle.
//  * S = Q K^T (M 128, N 128, K 128) lands in tensor memory; each of the four
//    row warps reads its 32 rows (one row per thread: no shuffles in the
//    softmax), writes P = 2^(s - m) back into the same columns as bf16 hi + lo
//    halves, and O += P V is issued with A = P from tensor memory and B = V
//    (MN-major) from shared memory.  O stays in tensor memory across the
//    chunk; a row whose maximum moves is rescaled in place.
//  * Warp 4 issues the MMAs (one thread), warp 5 the TMA copies; two S/P
//    buffers and two K/V stages let S of the next sub-tile and the copies run
//    under the softmax of the current one.
//  * Rows whose member does not share a block see it masked (p = 0); blocks
//    nobody in the group shares are neither loaded nor multiplied.
#include <algorithm>

#include "tcgen05.cuh"
#include "internal.h"

namespace kvs {

namespace {

// Row warps: four (one per 32-lane quadrant of tensor memory), or eight for
// rotation calls, where warps w and w + 4 share a quadrant and split its 128
// columns (their rows' softmax, the query rotation and the epilogue); then
// the MMA warp and the TMA warp.
template <bool RUNS>
__host__ __device__ constexpr int wd_row_warps() { return RUNS ? 8 : 4; }
template <bool RUNS>
__host__ __device__ constexpr int wd_threads() { return 32 * (wd_row_warps<RUNS>() + 2); }
constexpr int kWdSubBlocks = 8;          // blocks per sub-tile (128 tokens)
constexpr int kWdHalf = 128 * 128;       // one [128][64] bf16 half of a 128-row tile, bytes
constexpr int kWdTile = 2 * kWdHalf;     // a 128 x 128 bf16 tile
// Q + ST stages of K and V (one stage when every item is a single sub-tile)
// (rotation calls: Q hi and Q lo tiles)
template <int ST, bool RUNS>
constexpr int wd_smem() { return 1024 + kWdTile * ((RUNS ? 2 : 1) + 2 * ST); }
constexpr uint32_t kWdCols = 512;        // S/P buffers at 0 and 128, O at 256
// rotation calls: per row warp, (cos, sin) of a run's shift for each member
// slot of its 32 rows (at most 8 for G >= 4), for its 32 of the 64
// frequencies; the row stride is padded by 16 bytes so that slots fall in
// different banks
constexpr int kWdTblSlots = 8, kWdTblStride = 34;

__device__ __forceinline__ bool wd_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const bool ok = mbar_wait_bounded(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

// Position in this CTA's work: claim cl (KV head cl % hkv) and sub-tile j.
//  * Shared chunks: the claim is item cl / hkv, its sub-tiles the 8-block
//    pieces of the item's chunk.
//  * Rotation calls: the claim is range cl / hkv of a group's run items
//    (cr = {group, first item, items | split slot << 16, members}), sub-tile
//    j is item cr.y + j (one 8-block run).
// Lane k < 8 holds block k's record {sharing members, physical block}
// (members 0 past the chunk end).  The next position's item and record are
// loaded one position ahead.
struct WdCursor {
  int cl, j, n_cl, n_j;
  int4 cr, n_cr;   // rotation calls: the claim's range
  int4 it, n_it;   // the sub-tile's item
  int2 rec, n_rec;
};

template <bool RUNS>
__device__ __forceinline__ int wd_nsub(const WideParams& p, const WdCursor& c) {
  return RUNS ? (c.cr.z & 0xffff) : (c.it.z - c.it.y * p.ib + kWdSubBlocks - 1) / kWdSubBlocks;
}

// the item index of a position
template <bool RUNS>
__device__ __forceinline__ int wd_item(const WideParams& p, int cl, const int4& cr, int j) {
  return RUNS ? cr.y + j : cl / p.hkv;
}

template <bool RUNS>
__device__ __forceinline__ int2 wd_rec(const WideParams& p, int item, int j, int lane) {
  const size_t o = RUNS ? (size_t)item * kWdSubBlocks : ((size_t)item * p.max_sub + j) * kWdSubBlocks;
  return lane < kWdSubBlocks ? __ldg(p.wsub + o + lane) : make_int2(0, -1);
}

template <bool RUNS>
__device__ __forceinline__ void wd_start(const WideParams& p, WdCursor& c, int lane) {
  c.cl = blockIdx.x;
  c.j = 0;
  c.cr = RUNS ? __ldg(p.wclaims + blockIdx.x / p.hkv) : make_int4(0, 0, 0, 0);
  // speculative (before the plan check): keep the index inside the arrays
  const int item = RUNS ? min(max(c.cr.y, 0), p.max_witems - 1) : wd_item<RUNS>(p, c.cl, c.cr, 0);
  c.it = __ldg(p.witems + item);
  c.rec = wd_rec<RUNS>(p, item, 0, lane);
}

template <bool RUNS>
__device__ __forceinline__ void wd_prefetch(const WideParams& p, WdCursor& c, int n_claims, int lane) {
  c.n_cl = c.cl;
  c.n_j = c.j + 1;
  c.n_cr = c.cr;
  if (c.n_j >= wd_nsub<RUNS>(p, c)) {
    c.n_cl = c.cl + gridDim.x;
    c.n_j = 0;
    if (RUNS && c.n_cl < n_claims) c.n_cr = __ldg(p.wclaims + c.n_cl / p.hkv);
  }
  c.n_it = c.it;
  c.n_rec = make_int2(0, -1);
  if (c.n_cl < n_claims) {
    const int item = wd_item<RUNS>(p, c.n_cl, c.n_cr, c.n_j);
    if (RUNS || c.n_cl != c.cl) c.n_it = __ldg(p.witems + item);
    c.n_rec = wd_rec<RUNS>(p, item, c.n_j, lane);
  }
}

template <bool RUNS>
__device__ __forceinline__ void wd_advance(const WideParams& p, WdCursor& c, int n_claims, int lane) {
  c.cl = c.n_cl;
  c.j = c.n_j;
  c.cr = c.n_cr;
  c.it = c.n_it;
  c.rec = c.n_rec;
  if (c.cl < n_claims) wd_prefetch<RUNS>(p, c, n_claims, lane);
}

// blocks of the sub-tile that somebody shares (bit j: block j is loaded)
__device__ __forceinline__ uint32_t wd_loaded(const int2& rec) {
  return __ballot_sync(0xffffffffu, rec.x != 0) & 0xffu;
}

// kv_full / kv_empty: the ST K/V stages (rotation calls: the two K buffers,
// with v_full / v_empty for the two V buffers, so that a K buffer is refilled
// as soon as S has read it).
// pair[i] (rotation calls): the two row warps of quadrant i exchange their
// halves' row maxima (every run) and row sums (every split).
struct WdBars {
  uint64_t kv_full[2], kv_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2], q_full, o_free, fin;
  uint64_t pair[4];
};

}  // namespace

template <int ST, bool RUNS>
__global__ void __launch_bounds__(wd_threads<RUNS>(), 1)
attn_wide_kernel(const __grid_constant__ WideParams p, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ WdBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float rsc[RUNS ? 4 * 64 : 1];   // RoPE frequency pieces (rotation calls)
  __shared__ __align__(16) float2 tbl[RUNS ? 8 * kWdTblSlots * kWdTblStride : 2];
  __shared__ float xch[RUNS ? 2 * 2 * 128 : 1];   // [run parity][column half][row] row maxima
  __shared__ float xl[RUNS ? 2 * 128 : 1];        // [column half][row] row sums of a split
  constexpr int QT = RUNS ? 2 : 1;           // query tiles: Q (or Q hi, Q lo)
  constexpr int RW = wd_row_warps<RUNS>();   // row warps
  constexpr int NQ = 16 / RW;                // 32-column slices per row warp
  // launched as a programmatic dependent of the kernel before it (the
  // previous layer's merge, which reads the same split slots): nothing is
  // read before that kernel has completed.  Then the token-major kernel
  // queued behind this one (it computes other splits) may start on the SMs
  // left free.
  if (threadIdx.x == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = base;                                   // [2][128][64] (rotation calls: then Q lo)
  auto sK = [&](int s) { return base + kWdTile * (QT + 2 * s); };
  auto sV = [&](int s) { return base + kWdTile * (QT + 1 + 2 * s); };
  static_assert(!RUNS || ST == 2, "rotation calls use two K and two V buffers");

  // the plan header, the first item and its first record are independent
  // loads: issue them together (the grid never exceeds the item capacity)
  WdCursor cur;
  wd_start<RUNS>(p, cur, lane);
  // every compare evaluated (no short circuit): the header's loads are all
  // in flight together
  const PlanHdr ph = load_plan_hdr(p.hdr);
  const bool plan_ok = (ph.v[1] == p.magic) & (ph.v[2] == p.n_seq) & (ph.v[3] == p.max_blocks) & (ph.v[4] == p.R) &
                       (ph.v[5] == p.ibp) & (ph.v[6] == p.hkv) & (ph.v[7] == p.W) & (ph.v[9] == p.ib);
  const int n_claims = plan_ok ? min(ph.v[RUNS ? 10 : 8], p.max_witems) * p.hkv : 0;
  if ((int)blockIdx.x >= n_claims) return;   // uniform over the CTA: nothing allocated yet
  wd_prefetch<RUNS>(p, cur, n_claims, lane);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 32 * RW);
      mbar_init(&bars.pv_done[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    mbar_init(&bars.q_full, 32 * RW);
    mbar_init(&bars.o_free, 32 * RW);
    for (int i = 0; i < 4; ++i) mbar_init(&bars.pair[i], 64);
    mbar_init(&bars.fin, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (RUNS)
    for (int i = threadIdx.x; i < 4 * 64; i += blockDim.x) rsc[i] = p.rs[i >> 6][i & 63];
  if (warp == 0) {
    tmem_alloc(&s_tmem, kWdCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // warp-uniform view of the abort flag
  auto stop = [&]() { return __any_sync(0xffffffffu, s_abort != 0); };

  if (warp == RW + 1) {
    // ------------------------------------------------------ TMA producer
    // lane k < 8 copies block k of the sub-tile: both 64-column halves of K
    // and of V into the [half][token][64] stage
    int n = 0;
    int armed[2] = {-1, -1}, armed_v[2] = {-1, -1};   // parity of the last arming of kv_full / v_full [s]
    bool quit = false;
    // lanes k < 8 (bit k of lm) copy block k's two halves of K or V
    auto copy = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int h, uint32_t lm) {
      if ((lm >> lane) & 1u) {
        int ph = cur.rec.y;
        if (ph < 0 || ph >= p.capacity) {   // the plan shares valid blocks only
          set_err(p.status, KVS_DEVERR_BLOCK_ID);
          ph = 0;
        }
        const int row = (ph * p.hkv + h) * 16;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) tma_load_3d(dst + hf * kWdHalf + lane * 2048, map, 0, row, hf, bar);
      }
      __syncwarp();
    };
    for (; cur.cl < n_claims; wd_advance<RUNS>(p, cur, n_claims, lane)) {
      if (stop()) { quit = true; break; }
      const uint32_t lm = wd_loaded(cur.rec);
      if (!lm) continue;
      const int s = n % ST, h = cur.cl % p.hkv;
      // rotation calls: K buffer s is free once S of position n - 2 has
      // completed, V buffer s once P V of n - 2 has; otherwise the stage is
      // free once P V of n - ST has completed
      if (n >= ST && !wd_wait(&bars.kv_empty[s], ((n - ST) / ST) & 1, p.status)) {
        s_abort = 1;
        quit = true;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars.kv_full[s], (uint32_t)__popc(lm) * (RUNS ? 2u : 4u) * 2048u);
        armed[s] = (n / ST) & 1;
      }
      __syncwarp();
      copy(&tk, sK(s), &bars.kv_full[s], h, lm);
      if constexpr (RUNS) {
        if (n >= ST && !wd_wait(&bars.v_empty[s], ((n - ST) / ST) & 1, p.status)) {
          s_abort = 1;
          quit = true;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.v_full[s], (uint32_t)__popc(lm) * 2u * 2048u);
          armed_v[s] = (n / ST) & 1;
        }
        __syncwarp();
        copy(&tv, sV(s), &bars.v_full[s], h, lm);
      } else {
        copy(&tv, sV(s), &bars.kv_full[s], h, lm);
      }
      ++n;
    }
    if (quit) {   // copies still in flight land before the shared memory goes away
      for (int s = 0; s < 2; ++s) {
        if (armed[s] >= 0) mbar_drain(&bars.kv_full[s], (uint32_t)armed[s]);
        if (armed_v[s] >= 0) mbar_drain(&bars.v_full[s], (uint32_t)armed_v[s]);
      }
    }
  } else if (warp == RW) {
    // ----------------------------------------------------------- MMA issue
    constexpr uint32_t idS = umma_idesc_bf16(128, 128, false, false);
    constexpr uint32_t idO = umma_idesc_bf16(128, 128, false, true);
    const uint32_t tO = tmem + 256;
    int n = 0, k = -1, qn = 0;
    bool first_pv = true;
    int pend = -1;
    uint32_t pend_lm = 0;
    bool ok = true;
    auto issue_pv = [&](int m, uint32_t lmm) {
      if (first_pv && k >= 1 && !wd_wait(&bars.o_free, (k - 1) & 1, p.status)) return false;
      if (!wd_wait(&bars.p_full[m & 1], (m >> 1) & 1, p.status)) return false;
      if (RUNS && !wd_wait(&bars.v_full[m % ST], (m / ST) & 1, p.status)) return false;   // V of position m
      tc_fence_after();
      if (lane == 0) {
        const uint32_t tP = tmem + 128u * (m & 1);
        bool acc = !first_pv;
#pragma unroll
        for (int j = 0; j < kWdSubBlocks; ++j) {
          if (!((lmm >> j) & 1u)) continue;
          const uint64_t bv = umma_desc_sw128(smem_u32(sV(m % ST)) + j * 2048, kWdHalf, 1024);
          const uint32_t pj = tP + 32 * (j >> 1) + 8 * (j & 1);   // block j's P hi; its lo 16 columns on
          umma_ts(tO, pj, bv, idO, acc ? 1u : 0u);
          umma_ts(tO, pj + 16, bv, idO, 1u);
          acc = true;
        }
        umma_commit(&bars.pv_done[m & 1]);
        umma_commit(RUNS ? &bars.v_empty[m % ST] : &bars.kv_empty[m % ST]);
      }
      __syncwarp();
      first_pv = false;
      return true;
    };
    for (; cur.cl < n_claims; wd_advance<RUNS>(p, cur, n_claims, lane)) {
      if (stop()) { ok = false; break; }
      if (cur.j == 0) {   // a new claim: its query tile must be in place
        ++k;
        if (!RUNS && !wd_wait(&bars.q_full, (qn++) & 1, p.status)) { ok = false; break; }
        first_pv = true;
        pend = -1;
      }
      const uint32_t lm = wd_loaded(cur.rec);
      if (lm) {
        // rotation calls: every run has its own (rotated) query tile
        if (RUNS && !wd_wait(&bars.q_full, (qn++) & 1, p.status)) { ok = false; break; }
        const int s = n & 1, ks = n % ST;   // TMEM buffer, shared-memory stage
        if (!wd_wait(&bars.kv_full[ks], (n / ST) & 1, p.status)) { ok = false; break; }
        if (n >= 2 && !wd_wait(&bars.pv_done[s], ((n - 2) >> 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 8 * QT; ++kk) {   // rotation calls: Q hi, then Q lo
            const uint64_t a =
                umma_desc_sw128(smem_u32(sQ) + (kk >> 3) * kWdTile + ((kk >> 2) & 1) * kWdHalf + (kk & 3) * 32, 16, 1024);
            const uint64_t b =
                umma_desc_sw128(smem_u32(sK(ks)) + ((kk >> 2) & 1) * kWdHalf + (kk & 3) * 32, 16, 1024);
            umma_ss(tmem + 128u * s, a, b, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars.s_full[s]);
          if (RUNS) umma_commit(&bars.kv_empty[ks]);   // K buffer ks may be refilled
        }
        __syncwarp();
        if (pend >= 0 && !issue_pv(pend, pend_lm)) { ok = false; break; }
        pend = n;
        pend_lm = lm;
        ++n;
      }
      if (cur.n_cl != cur.cl) {   // the claim's last sub-tile
        if (pend >= 0) {
          if (!issue_pv(pend, pend_lm)) { ok = false; break; }
          pend = -1;
        } else if (k >= 1 && !wd_wait(&bars.o_free, (k - 1) & 1, p.status)) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) s_abort = 1;
    // every MMA issued has completed before the tensor memory is released
    if (lane == 0) umma_commit(&bars.fin);
    __syncwarp();
    mbar_wait_bounded(&bars.fin, 0, p.status);
  } else {
    // ------------------------------------------------------------ row warps
    const int qd = warp & 3, ch = warp >> 2;   // TMEM lane quadrant, column half (rotation calls)
    const int r = qd * 32 + lane;              // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    const int slot = r / p.g, hh = r - slot * p.g;
    const float sl2 = p.scale_log2;
    // 4 KB of the Q (hi) tile per row warp, reused to stage O
    uint8_t* stg = sQ + warp * 4096;
    int pu = 0;   // uses of this quadrant's pair barrier
    // rotation calls: the two warps of the quadrant exchange a value per row
    auto pair_sync = [&]() {
      mbar_arrive(&bars.pair[qd]);
      return wd_wait(&bars.pair[qd], (pu++) & 1, p.status);
    };
    int n = 0, k = -1;
    bool ok = true, pend_epi = false;
    int e_gw = 0, e_h = 0, e_c = 0, e_last = 0;
    uint32_t e_spm = 0;
    float e_m = 0.f, e_l = 0.f;
    float m = -INFINITY, l = 0.f;
    bool first = true, row_ok = false;
    // rotation calls: this row's query (the claim's KV head; the warp's
    // half of the dims and their rotation partners), loaded once per claim
    // and rotated from registers for each of its runs
    uint4 qreg[RUNS ? 8 : 1];
    // The finished chunk's splits of this warp's 32 rows.  Each 32-column
    // slice of O goes from tensor memory through shared memory (128-byte
    // rows, XOR-swizzled) so that stores cover whole row segments.
    auto epilogue = [&]() {
      float l_tot = e_l;
      if (RUNS) {   // the row sum over both column halves
        xl[ch * 128 + r] = e_l;
        if (!pair_sync()) return false;
        l_tot = xl[r] + xl[128 + r];
      }
#pragma unroll 1
      for (int qq = 0; qq < NQ; ++qq) {
        const int q = ch * NQ + qq;
        uint32_t v[32];
        tmem_ld32(tO + 32 * q, v);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((e ^ (lane & 7)) << 4)) =
              make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int jr = 4 * t + (lane >> 3), e = lane & 7;
          const int r2 = qd * 32 + jr, sl = r2 / p.g, h2 = r2 - sl * p.g, a2 = e_gw * p.W + sl;
          if (sl < p.W && a2 < p.n_seq && ((e_spm >> sl) & 1u)) {
            const size_t it2 = (((size_t)a2 * p.hkv + e_h) * p.n_chunks + e_c) * p.g + h2;
            // evict-last, as the token-major kernel's splits: the merge reads it back
            st_hint_v4u32(p.p2 + it2 * 128 + 32 * q + 4 * e,
                          *reinterpret_cast<const uint4*>(stg + jr * 128 + ((e ^ (jr & 7)) << 4)), l2_policy_evict_last());
          }
        }
        __syncwarp();
      }
      const int a = e_gw * p.W + slot;
      if (ch == 0 && slot < p.W && a < p.n_seq && ((e_spm >> slot) & 1u)) {
        const size_t im = (((size_t)a * p.hkv + e_h) * p.g + hh) * p.n_chunks + e_c;
        __stcg(reinterpret_cast<float2*>(p.p2_ml + im * 2), make_float2(e_m, l_tot));
      }
      return true;
    };
    // The query rows of a claim (a rotation call: of one run item) into the
    // Q tile ([half][row][64], 128-byte swizzle); the S MMAs that read the
    // previous contents have completed.
    auto load_q = [&](int gw, int h, const int4& it, int item) {
      const int a = gw * p.W + slot;
      row_ok = slot < p.W && a < p.n_seq;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)(row_ok ? a : 0) * p.hq + h * p.g + hh) * 128);
      if constexpr (RUNS) {
        // this member's query rotated back by its shift on this run,
        // q' = R(-delta) q (rotate-half pairs i, i + 64), as bf16 hi (first
        // tile) + lo (second tile); rows of non-members are zero.  The
        // angles are computed once per member slot of the warp's rows.
        const bool mem = row_ok && ((((uint32_t)it.w) >> slot) & 1u);
        const int s_lo = (qd * 32) / p.g;
        const int n_s = min((qd * 32 + 31) / p.g - s_lo + 1, kWdTblSlots);
        int dl_own = 0;
        if (lane < n_s) {
          const int sl = s_lo + lane;
          const bool mm = sl < p.W && gw * p.W + sl < p.n_seq && ((((uint32_t)it.w) >> sl) & 1u);
          dl_own = mm ? __ldg(p.wmem + (size_t)item * 32 + sl).y : 0;
        }
        // this warp's frequencies 32 ch + lane, one table row per slot
        float2* tb = tbl + warp * (kWdTblSlots * kWdTblStride);
        __syncwarp();   // the previous run's table has been read
        for (int k = 0; k < n_s; ++k) {
          const int dl = __shfl_sync(0xffffffffu, dl_own, k);
          float cs, sn;
          rope_cos_sin(rsc, 32 * ch + lane, dl, cs, sn);
          tb[k * kWdTblStride + lane] = make_float2(cs, sn);
        }
        __syncwarp();
        const float2* mine = tb + min(max(slot - s_lo, 0), kWdTblSlots - 1) * kWdTblStride;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {   // dims 8c..8c+7 (c = 4 ch + cc) and their partners 64 + 8c..
          const int c = 4 * ch + cc;
          const uint4 xv = mem ? qreg[cc] : z, yv = mem ? qreg[4 + cc] : z;
          const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ys[4] = {yv.x, yv.y, yv.z, yv.w};
          uint32_t xh[4], xlo[4], yh[4], ylo[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float x0 = bf16_lo(xs[u]), x1 = bf16_hi(xs[u]), y0 = bf16_lo(ys[u]), y1 = bf16_hi(ys[u]);
            const float4 cs = *reinterpret_cast<const float4*>(mine + 8 * cc + 2 * u);   // (c0, s0, c1, s1)
            split_bf16(x0 * cs.x + y0 * cs.y, x1 * cs.z + y1 * cs.w, xh[u], xlo[u]);
            split_bf16(y0 * cs.x - x0 * cs.y, y1 * cs.z - x1 * cs.w, yh[u], ylo[u]);
          }
          const uint32_t off = r * 128 + ((c ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(sQ + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
          *reinterpret_cast<uint4*>(sQ + kWdHalf + off) = make_uint4(yh[0], yh[1], yh[2], yh[3]);
          *reinterpret_cast<uint4*>(sQ + kWdTile + off) = make_uint4(xlo[0], xlo[1], xlo[2], xlo[3]);
          *reinterpret_cast<uint4*>(sQ + kWdTile + kWdHalf + off) = make_uint4(ylo[0], ylo[1], ylo[2], ylo[3]);
        }
      } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint4 qv[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) qv[c] = row_ok ? __ldg(src + hf * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(sQ + hf * kWdHalf + r * 128 + ((c ^ (r & 7)) << 4)) = qv[c];
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars.q_full);
    };
    for (; cur.cl < n_claims; wd_advance<RUNS>(p, cur, n_claims, lane)) {
      if (stop()) { ok = false; break; }
      const int gw = cur.it.x & ((1 << 30) - 1), h = cur.cl % p.hkv;
      if (cur.j == 0) {   // a new claim
        ++k;
        if (k >= 1) {
          if (pend_epi) {
            if (!wd_wait(&bars.pv_done[e_last & 1], (e_last >> 1) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
            if (!epilogue()) { ok = false; break; }
            pend_epi = false;
          }
          tc_fence_before();
          mbar_arrive(&bars.o_free);
        }
        const int a = gw * p.W + slot;
        row_ok = slot < p.W && a < p.n_seq;
        if constexpr (RUNS) {
          const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)(row_ok ? a : 0) * p.hq + h * p.g + hh) * 128);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            qreg[cc] = row_ok ? __ldg(src + 4 * ch + cc) : make_uint4(0u, 0u, 0u, 0u);
            qreg[4 + cc] = row_ok ? __ldg(src + 8 + 4 * ch + cc) : make_uint4(0u, 0u, 0u, 0u);
          }
        } else {
          load_q(gw, h, cur.it, 0);
        }
        m = -INFINITY;
        l = 0.f;
        first = true;
      }
      const uint32_t lm = wd_loaded(cur.rec);
      if (lm) {
        // rotation calls: the claim's first run is rotated here, every later
        // one once S of the run before it has read the query tile (below)
        if (RUNS && cur.j == 0) load_q(gw, h, cur.it, cur.cr.y);
        const int s = n & 1;
        uint32_t rl = 0;   // blocks this row takes
#pragma unroll
        for (int j = 0; j < kWdSubBlocks; ++j) {
          const uint32_t gm = (uint32_t)__shfl_sync(0xffffffffu, cur.rec.x, j);
          rl |= ((row_ok && ((gm >> slot) & 1u)) ? 1u : 0u) << j;
        }
        if (!wd_wait(&bars.s_full[s], (n >> 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        // the next run's query, so that its S runs under this run's softmax
        if (RUNS && cur.n_cl == cur.cl) load_q(gw, h, cur.n_it, cur.cr.y + cur.j + 1);
        const uint32_t tS = tmem + lane_off + 128u * s;
        // two passes over the S row in tensor memory (32 columns at a time):
        // its maximum, then P; only one slice is held in registers
        // (rotation calls: over this warp's column half, then combined with
        // the other half's through the quadrant's pair barrier)
        float mx = -INFINITY;
#pragma unroll 1
        for (int qq = 0; qq < NQ; qq += 2) {   // two slices under one wait
          const int q = ch * NQ + qq;
          uint32_t v[64];
          tmem_ld64(tS + 32 * q, v);
          const uint32_t lq = (rl >> (2 * q)) & 15u;
#pragma unroll
          for (int t = 0; t < 64; ++t)
            if ((lq >> (t >> 4)) & 1u) mx = fmaxf(mx, __uint_as_float(v[t]));
        }
        mx = mx == -INFINITY ? mx : mx * sl2;
        if (RUNS) {
          xch[((n & 1) * 2 + ch) * 128 + r] = mx;
          if (!pair_sync()) { ok = false; break; }
          mx = fmaxf(mx, xch[((n & 1) * 2 + (ch ^ 1)) * 128 + r]);
        }
        // The reference point moves only on a row's first live values or when
        // the new maximum exceeds it by more than 8 (so P < 2^8 and O is
        // rescaled rarely); m, l and O stay relative to the same reference,
        // so the split is exact either way.
        const float mn = (m == -INFINITY || mx > m + 8.f) ? fmaxf(m, mx) : m;
        // nothing live yet: reference point 0, so that 2^(-inf - 0) = 0
        const float ref = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m - ref);
        float sum = 0.f;
#pragma unroll 1
        for (int qq = 0; qq < NQ; ++qq) {
          const int q = ch * NQ + qq;
          uint32_t v[32], hi[16], lo[16];
          tmem_ld32(tS + 32 * q, v);
          const uint32_t lq = (rl >> (2 * q)) & 3u;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const bool live = (lq >> (e >> 3)) & 1u;
            const float p0 = live ? fast_exp2(__uint_as_float(v[2 * e]) * sl2 - ref) : 0.f;
            const float p1 = live ? fast_exp2(__uint_as_float(v[2 * e + 1]) * sl2 - ref) : 0.f;
            sum += p0 + p1;
            split_bf16(p0, p1, hi[e], lo[e]);
          }
          // P of tokens 32q..32q+31 as packed bf16 pairs, hi then lo, in the
          // slice's own (already read) columns
          tmem_st16(tS + 32 * q, hi);
          tmem_st16(tS + 32 * q + 16, lo);
        }
        // a row whose maximum moved rescales its O once the previous P V is done
        const bool need = !first && m != -INFINITY && mn > m;
        if (__any_sync(0xffffffffu, need)) {
          if (!wd_wait(&bars.pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, p.status)) { ok = false; break; }
          tc_fence_after();
          const float f = need ? alpha : 1.f;
#pragma unroll 1
          for (int qq = 0; qq < NQ; ++qq) {
            const int q = ch * NQ + qq;
            uint32_t v[32];
            tmem_ld32(tO + 32 * q, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
            tmem_st32(tO + 32 * q, v);
          }
        }
        l = l * alpha + sum;
        m = mn;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_full[s]);
        first = false;
        ++n;
      }
      if (cur.n_cl != cur.cl && !first) {   // the claim's last sub-tile: its split is pending
        pend_epi = true;
        e_gw = gw;
        e_h = h;
        e_c = RUNS ? (cur.cr.z >> 16) : cur.it.y;   // the claim's split slot
        e_spm = (uint32_t)(RUNS ? cur.cr.w : cur.it.w);
        e_last = n - 1;
        e_m = m;
        e_l = l;
      }
    }
    if (ok && pend_epi) {
      if (wd_wait(&bars.pv_done[e_last & 1], (e_last >> 1) & 1, p.status)) {
        tc_fence_after();
        if (!epilogue()) ok = false;
      } else {
        ok = false;
      }
    }
    if (!ok) s_abort = 1;
  }
  // teardown: every role has finished with the tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kWdCols);
  }
}

template <int ST, bool RUNS>
static kvs_status launch_wide(const WideParams& p, const kvs_pool* pool, int layer, int grid, cudaStream_t stream) {
  if (!smem_limit_once<attn_wide_kernel<ST, RUNS>>(wd_smem<ST, RUNS>(), pool->device))
    return fail(KVS_ERR_CUDA, "decode_attn: cannot raise the shared-memory limit (wide tile)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(wd_threads<RUNS>());
  cfg.dynamicSmemBytes = wd_smem<ST, RUNS>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // a rotation-call tile fills its SM's shared memory: launched early it
  // would hold SMs that the previous layer's merge still needs
  cfg.numAttrs = RUNS ? 0 : 1;
  if (cudaLaunchKernelEx(&cfg, attn_wide_kernel<ST, RUNS>, p, pool->tk1[layer], pool->tv1[layer]) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_attn: wide tile launch failed");
  count_launch();
  return check_launch("decode_attn_wide");
}

kvs_status launch_wide_tile(const WideParams& p, const kvs_pool* pool, int layer, int max_claims,
                            cudaStream_t stream) {
  if (max_claims <= 0) return KVS_OK;
  // one CTA per SM (its 512 TMEM columns), claims taken round-robin; CTAs
  // beyond the plan's item count return at once.  Items of one sub-tile need
  // no second stage, which leaves room on the SM for a token-major CTA.
  // (rotation calls: on part of the SMs, the token-major kernel on the rest)
  const int grid = std::max(1, std::min(p.runs ? runs_wide_ctas(pool) : pool->num_sms, max_claims));
  // the MMA thread issues S of the next sub-tile before P V of the current
  // one, so claims of several sub-tiles (and rotation ranges) need two stages
  if (p.runs) return launch_wide<2, true>(p, pool, layer, grid, stream);
  return p.max_sub > 1 ? launch_wide<2, false>(p, pool, layer, grid, stream)
                      : launch_wide<1, false>(p, pool, layer, grid, stream);
}

}  // namespace kvs
