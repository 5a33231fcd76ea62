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

constexpr int kWdThreads = 192;          // 4 row warps, MMA warp, TMA warp
constexpr int kWdSubBlocks = 8;          // blocks per sub-tile (128 tokens)
constexpr int kWdHalf = 128 * 128;       // one [128][64] bf16 half of a 128-row tile, bytes
constexpr int kWdTile = 2 * kWdHalf;     // a 128 x 128 bf16 tile
constexpr int kWdSmem = 1024 + kWdTile * 5;   // Q + 2 stages of K and V
constexpr uint32_t kWdCols = 512;        // S/P buffers at 0 and 128, O at 256

__device__ __forceinline__ bool wd_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const bool ok = mbar_wait_bounded(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

// Sharing members of the blocks of one sub-tile (gm[j], 0 past the chunk
// end); bit j of the result: block j is loaded (somebody shares it).
__device__ __forceinline__ uint32_t wd_masks(const WideParams& p, int gw, int b0, int nb, uint32_t (&gm)[kWdSubBlocks]) {
  uint32_t lm = 0;
#pragma unroll
  for (int j = 0; j < kWdSubBlocks; ++j) {
    gm[j] = j < nb ? __ldg(p.gmask + (size_t)gw * p.max_blocks + b0 + j) : 0u;
    lm |= (gm[j] != 0u ? 1u : 0u) << j;
  }
  return lm;
}

struct WdBars {
  uint64_t kv_full[2], kv_empty[2], s_full[2], p_full[2], pv_done[2], q_full, o_free, fin;
};

}  // namespace

__global__ void __launch_bounds__(kWdThreads, 1)
attn_wide_kernel(const __grid_constant__ WideParams p, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ WdBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = base;                                   // [2][128][64]
  auto sK = [&](int s) { return base + kWdTile * (1 + 2 * s); };
  auto sV = [&](int s) { return base + kWdTile * (2 + 2 * s); };

  const bool plan_ok = p.hdr[1] == p.magic && p.hdr[2] == p.n_seq && p.hdr[3] == p.max_blocks &&
                       p.hdr[4] == p.R && p.hdr[5] == p.ib && p.hdr[6] == p.hkv && p.hdr[7] == p.W;
  const int n_claims = plan_ok ? p.hdr[8] * p.hkv : 0;
  if ((int)blockIdx.x >= n_claims) return;   // uniform over the CTA: nothing allocated yet

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_full[s], 128);
      mbar_init(&bars.pv_done[s], 1);
    }
    mbar_init(&bars.q_full, 128);
    mbar_init(&bars.o_free, 128);
    mbar_init(&bars.fin, 1);
    s_abort = 0;
    fence_barrier_init();
  }
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

  if (warp == 5) {
    // ------------------------------------------------------ TMA producer
    int n = 0;
    int armed[2] = {-1, -1};
    bool quit = false;
    for (int cl = blockIdx.x; cl < n_claims && !quit; cl += gridDim.x) {
      const int4 it = __ldg(p.witems + cl / p.hkv);
      const int h = cl % p.hkv, gw = it.x & ((1 << 30) - 1);
      for (int b0 = it.y * p.ib; b0 < it.z; b0 += kWdSubBlocks) {
        if (stop()) { quit = true; break; }
        const int nb = min(kWdSubBlocks, it.z - b0);
        uint32_t gm[kWdSubBlocks];
        const uint32_t lm = wd_masks(p, gw, b0, nb, gm);
        if (!lm) continue;
        const int s = n & 1;
        if (n >= 2 && !wd_wait(&bars.kv_empty[s], ((n - 2) >> 1) & 1, p.status)) {
          s_abort = 1;
          quit = true;
          break;
        }
        int phys = lane < nb ? __ldg(p.gphys + (size_t)gw * p.max_blocks + b0 + lane) : 0;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars.kv_full[s], (uint32_t)__popc(lm) * 4u * 2048u);
          armed[s] = n;
        }
#pragma unroll
        for (int j = 0; j < kWdSubBlocks; ++j) {
          int ph = __shfl_sync(0xffffffffu, phys, j);
          if (lane == 0 && ((lm >> j) & 1u)) {
            if (ph < 0 || ph >= p.capacity) {   // the plan shares valid blocks only
              set_err(p.status, KVS_DEVERR_BLOCK_ID);
              ph = 0;
            }
            const int row = (ph * p.hkv + h) * 16;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              tma_load_3d(sK(s) + hf * kWdHalf + j * 2048, &tk, 0, row, hf, &bars.kv_full[s]);
              tma_load_3d(sV(s) + hf * kWdHalf + j * 2048, &tv, 0, row, hf, &bars.kv_full[s]);
            }
          }
        }
        __syncwarp();
        ++n;
      }
    }
    if (quit) {   // copies still in flight land before the shared memory goes away
      for (int s = 0; s < 2; ++s)
        if (armed[s] >= 0) mbar_drain(&bars.kv_full[s], (armed[s] >> 1) & 1);
    }
  } else if (warp == 4) {
    // ----------------------------------------------------------- MMA issue
    constexpr uint32_t idS = umma_idesc_bf16(128, 128, false, false);
    constexpr uint32_t idO = umma_idesc_bf16(128, 128, false, true);
    const uint32_t tO = tmem + 256;
    int n = 0, k = 0;
    bool first_pv = true;
    int pend = -1;
    uint32_t pend_lm = 0;
    bool ok = true;
    auto issue_pv = [&](int m, uint32_t lmm) {
      if (first_pv && k >= 1 && !wd_wait(&bars.o_free, (k - 1) & 1, p.status)) return false;
      if (!wd_wait(&bars.p_full[m & 1], (m >> 1) & 1, p.status)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t tP = tmem + 128u * (m & 1);
        bool acc = !first_pv;
#pragma unroll
        for (int j = 0; j < kWdSubBlocks; ++j) {
          if (!((lmm >> j) & 1u)) continue;
          const uint64_t bv = umma_desc_sw128(smem_u32(sV(m & 1)) + j * 2048, kWdHalf, 1024);
          umma_ts(tO, tP + 8 * j, bv, idO, acc ? 1u : 0u);
          umma_ts(tO, tP + 64 + 8 * j, bv, idO, 1u);
          acc = true;
        }
        umma_commit(&bars.pv_done[m & 1]);
        umma_commit(&bars.kv_empty[m & 1]);
      }
      __syncwarp();
      first_pv = false;
      return true;
    };
    for (int cl = blockIdx.x; cl < n_claims; cl += gridDim.x, ++k) {
      if (stop()) { ok = false; break; }
      if (!wd_wait(&bars.q_full, k & 1, p.status)) { ok = false; break; }
      const int4 it = __ldg(p.witems + cl / p.hkv);
      const int gw = it.x & ((1 << 30) - 1);
      first_pv = true;
      pend = -1;
      for (int b0 = it.y * p.ib; b0 < it.z; b0 += kWdSubBlocks) {
        const int nb = min(kWdSubBlocks, it.z - b0);
        uint32_t gm[kWdSubBlocks];
        const uint32_t lm = wd_masks(p, gw, b0, nb, gm);
        if (!lm) continue;
        const int s = n & 1;
        if (!wd_wait(&bars.kv_full[s], (n >> 1) & 1, p.status)) { ok = false; break; }
        if (n >= 2 && !wd_wait(&bars.pv_done[s], ((n - 2) >> 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t a = umma_desc_sw128(smem_u32(sQ) + (kk >> 2) * kWdHalf + (kk & 3) * 32, 16, 1024);
            const uint64_t b = umma_desc_sw128(smem_u32(sK(s)) + (kk >> 2) * kWdHalf + (kk & 3) * 32, 16, 1024);
            umma_ss(tmem + 128u * s, a, b, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars.s_full[s]);
        }
        __syncwarp();
        if (pend >= 0 && !issue_pv(pend, pend_lm)) { ok = false; break; }
        pend = n;
        pend_lm = lm;
        ++n;
      }
      if (!ok) break;
      if (pend >= 0) {
        if (!issue_pv(pend, pend_lm)) { ok = false; break; }
      } else if (k >= 1 && !wd_wait(&bars.o_free, (k - 1) & 1, p.status)) {
        ok = false;
        break;
      }
    }
    if (!ok) s_abort = 1;
    // every MMA issued has completed before the tensor memory is released
    if (lane == 0) umma_commit(&bars.fin);
    __syncwarp();
    mbar_wait_bounded(&bars.fin, 0, p.status);
  } else {
    // ------------------------------------------------------------ row warps
    const int r = threadIdx.x;   // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    const int slot = r / p.g, hh = r - slot * p.g;
    const float sl2 = p.scale_log2;
    int n = 0, k = 0;
    bool ok = true, pend_epi = false, e_ok = false;
    int e_a = 0, e_h = 0, e_c = 0, e_last = 0;
    float e_m = 0.f, e_l = 0.f;
    // the finished chunk's split of this row: O from tensor memory, (m, l)
    auto epilogue = [&]() {
      const size_t it = (((size_t)e_a * p.hkv + e_h) * p.n_chunks + e_c) * p.g + hh;
      float* dst = p.p2 + it * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld32(tO + 32 * q, v);
        if (e_ok) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            __stcg(reinterpret_cast<float4*>(dst + 32 * q + 4 * e),
                   make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                               __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3])));
        }
      }
      if (e_ok) __stcg(reinterpret_cast<float2*>(p.p2_ml + it * 2), make_float2(e_m, e_l));
    };
    for (int cl = blockIdx.x; cl < n_claims; cl += gridDim.x, ++k) {
      if (stop()) { ok = false; break; }
      const int4 it = __ldg(p.witems + cl / p.hkv);
      const int h = cl % p.hkv, gw = it.x & ((1 << 30) - 1);
      const int a = gw * p.W + slot;
      const bool row_ok = slot < p.W && a < p.n_seq;
      // this claim's query rows into the Q tile ([half][row][64], 128-byte
      // swizzle); every S of the previous claim has completed
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)(row_ok ? a : 0) * p.hq + h * p.g + hh) * 128);
#pragma unroll
        for (int c16 = 0; c16 < 16; ++c16) {
          const uint4 v = row_ok ? __ldg(src + c16) : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(sQ + (c16 >> 3) * kWdHalf + r * 128 + (((c16 & 7) ^ (r & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars.q_full);
      if (k >= 1) {
        if (pend_epi) {
          if (!wd_wait(&bars.pv_done[e_last & 1], (e_last >> 1) & 1, p.status)) { ok = false; break; }
          tc_fence_after();
          epilogue();
          pend_epi = false;
        }
        tc_fence_before();
        mbar_arrive(&bars.o_free);
      }
      float m = -INFINITY, l = 0.f;
      bool first = true;
      for (int b0 = it.y * p.ib; b0 < it.z; b0 += kWdSubBlocks) {
        const int nb = min(kWdSubBlocks, it.z - b0);
        uint32_t gm[kWdSubBlocks];
        const uint32_t lm = wd_masks(p, gw, b0, nb, gm);
        if (!lm) continue;
        const int s = n & 1;
        if (!wd_wait(&bars.s_full[s], (n >> 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t rl = 0;   // blocks this row takes
#pragma unroll
        for (int j = 0; j < kWdSubBlocks; ++j) rl |= ((row_ok && ((gm[j] >> slot) & 1u)) ? 1u : 0u) << j;
        const uint32_t tS = tmem + lane_off + 128u * s;
        uint32_t sv[128];
        tmem_ld32(tS, sv);
        tmem_ld32(tS + 32, sv + 32);
        tmem_ld32(tS + 64, sv + 64);
        tmem_ld32(tS + 96, sv + 96);
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < 128; ++t)
          if ((rl >> (t >> 4)) & 1u) mx = fmaxf(mx, __uint_as_float(sv[t]) * sl2);
        const float mn = fmaxf(m, mx);
        // nothing live yet: reference point 0, so that 2^(-inf - 0) = 0
        const float ref = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m - ref);
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int t = 32 * q + 2 * e;
            const bool live = (rl >> (t >> 4)) & 1u;
            const float p0 = live ? fast_exp2(__uint_as_float(sv[t]) * sl2 - ref) : 0.f;
            const float p1 = live ? fast_exp2(__uint_as_float(sv[t + 1]) * sl2 - ref) : 0.f;
            sum += p0 + p1;
            split_bf16(p0, p1, hi[e], lo[e]);
          }
          tmem_st16(tS + 16 * q, hi);        // P hi: tokens 32q.. as packed pairs
          tmem_st16(tS + 64 + 16 * q, lo);   // P lo
        }
        // a row whose maximum moved rescales its O once the previous P V is done
        const bool need = !first && m != -INFINITY && mn > m;
        if (__any_sync(0xffffffffu, need)) {
          if (!wd_wait(&bars.pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, p.status)) { ok = false; break; }
          tc_fence_after();
          const float f = need ? alpha : 1.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
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
      if (!ok) break;
      if (!first) {
        pend_epi = true;
        e_ok = row_ok && ((((uint32_t)it.w) >> slot) & 1u);
        e_a = a;
        e_h = h;
        e_c = it.y;
        e_last = n - 1;
        e_m = m;
        e_l = l;
      }
    }
    if (ok && pend_epi) {
      if (wd_wait(&bars.pv_done[e_last & 1], (e_last >> 1) & 1, p.status)) {
        tc_fence_after();
        epilogue();
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

kvs_status launch_wide_tile(const WideParams& p, const kvs_pool* pool, int layer, int max_claims,
                            cudaStream_t stream) {
  if (max_claims <= 0) return KVS_OK;
  if (!smem_limit_once<attn_wide_kernel>(kWdSmem, pool->device))
    return fail(KVS_ERR_CUDA, "decode_attn: cannot raise the shared-memory limit (wide tile)");
  // one CTA per SM (its shared memory and 512 TMEM columns), claims taken
  // round-robin; CTAs beyond the plan's item count return at once
  const int grid = std::max(1, std::min(pool->num_sms, max_claims));
  attn_wide_kernel<<<grid, kWdThreads, kWdSmem, stream>>>(p, pool->tk1[layer], pool->tv1[layer]);
  count_launch();
  return check_launch("decode_attn_wide");
}

}  // namespace kvs
