// Block-granular MemDecay eviction scoring (MemDecay post §3.2: a token's
// current score is its region's initial score times exp(-decay * steps since
// it was stored), lowest evicted first; §4.1 scoring code: times
// (1 + 0.1 ln(1 + accesses)) for an accessed token; §5.3: eviction by whole
// blocks, judged by the mean score of their tokens).
//
// One CTA of 1024 threads per sequence:
//  1. block scores: a half-warp per block, one lane per token, reduced with
//     shuffles in a fixed order (deterministic), divided by the block's
//     stored token count;
//  2. the k lowest: a radix select over the float bit patterns (scores are
//     non-negative, so bit order is numeric order), 8 bits at a time;
//  3. ordered emission of the victims: scores below the k-th, then equal
//     ones in block order until k are taken (ties go to the lower block).
#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr int kEvMaxRegions = 16;
constexpr int kEvUnroll = 4;   // blocks per half-warp whose loads are in flight together

struct EvictParams {
  const uint8_t* region;
  const int32_t* created;
  const int32_t* access;
  const int32_t* seq_len;
  const int32_t* k;
  float* scores;
  int32_t* victims;
  int64_t* victims_off;
  uint32_t* status;
  int n_seq, max_blocks, B, n_regions;
  long long step;
  float init[kEvMaxRegions], decay[kEvMaxRegions];
};

__device__ __forceinline__ int ev_blocks(const EvictParams& p, int a) {
  int L = p.seq_len[a];
  if (L < 0) L = 0;
  if (L > p.max_blocks * p.B) L = p.max_blocks * p.B;
  return (L + p.B - 1) / p.B;
}

__device__ __forceinline__ int ev_k(const EvictParams& p, int a) {
  const int nb = ev_blocks(p, a);
  const int k = p.k[a];
  return k < 0 ? 0 : (k > nb ? nb : k);
}

__global__ void __launch_bounds__(1024) evict_kernel(const __grid_constant__ EvictParams p) {
  __shared__ unsigned hist[256];
  __shared__ int warp_sums[32];
  __shared__ unsigned s_prefix;
  __shared__ int s_remaining;
  __shared__ long long s_out0;
  __shared__ long long s_part[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int a = blockIdx.x; a < p.n_seq; a += gridDim.x) {
    int L = p.seq_len[a];
    if (L < 0 || L > p.max_blocks * p.B) {
      if (threadIdx.x == 0) set_err(p.status, KVS_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : p.max_blocks * p.B;
    }
    const int nb = (L + p.B - 1) / p.B;
    float* srow = p.scores + (size_t)a * p.max_blocks;
    // ---- 1. block scores: a half-warp per block (B <= 16), one lane per token;
    // the loads of kEvUnroll blocks per half-warp go out before any is used
    const int half = lane >> 4, hl = lane & 15;
    for (int b0 = warp * 2; b0 < p.max_blocks; b0 += 64 * kEvUnroll) {
      int rg[kEvUnroll], cr[kEvUnroll], ac[kEvUnroll];
      bool on[kEvUnroll];
#pragma unroll
      for (int j = 0; j < kEvUnroll; ++j) {
        const int b = b0 + 64 * j + half, t = b * p.B + hl;
        on[j] = b < nb && hl < p.B && t < L;
        const size_t o = (size_t)a * p.max_blocks * p.B + t;
        rg[j] = on[j] ? (int)p.region[o] : -1;
        cr[j] = on[j] ? p.created[o] : 0;
        ac[j] = on[j] ? p.access[o] : 0;
      }
#pragma unroll
      for (int j = 0; j < kEvUnroll; ++j) {
        const int b = b0 + 64 * j + half;
        float s = 0.f;
        int r = rg[j];
        if (r >= p.n_regions) {
          set_err(p.status, KVS_DEVERR_JOB);
          r = -1;
        }
        if (r >= 0) {
          const float age = (float)(p.step - (long long)cr[j]);
          s = p.init[r] * expf(-p.decay[r] * age);
          if (ac[j] > 0) s *= 1.f + 0.1f * log1pf((float)ac[j]);
        }
        int cnt = on[j] ? 1 : 0;
#pragma unroll
        for (int off = 8; off; off >>= 1) {
          s += __shfl_xor_sync(0xffffffffu, s, off);
          cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        }
        if (hl == 0 && b < p.max_blocks) srow[b] = b < nb ? s / (float)cnt : INFINITY;
      }
    }
    // ---- 2. the k-th lowest bit pattern.  The output offset of this
    // sequence's victims is the sum of the counts of the sequences before it,
    // summed by all threads.
    const int k = ev_k(p, a);
    {
      long long part = 0;
      for (int c = threadIdx.x; c < a; c += blockDim.x) part += ev_k(p, c);
#pragma unroll
      for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) s_part[warp] = part;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long o = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) o += s_part[w];
      s_out0 = o;
      p.victims_off[a] = o;
      if (a == p.n_seq - 1) p.victims_off[p.n_seq] = o + k;
      s_prefix = 0u;
      s_remaining = k;
    }
    __syncthreads();
    const long long out0 = s_out0;
    if (k > 0) {
      const unsigned* sb = reinterpret_cast<const unsigned*>(srow);
      unsigned mask = 0u;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        const unsigned pre = s_prefix;
        for (int i = threadIdx.x; i < nb; i += blockDim.x) {
          const unsigned v = sb[i];
          if ((v & mask) == pre) atomicAdd(&hist[(v >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
          // the digit: the first bin whose running count reaches the
          // remaining rank (bin 255 if none does); lane l scans bins 8l..8l+7
          // after a prefix sum of the lanes' totals
          unsigned c8[8], lsum = 0u;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            c8[j] = hist[lane * 8 + j];
            lsum += c8[j];
          }
          unsigned incl = lsum;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
          }
          const unsigned excl = incl - lsum;
          const unsigned rem0 = (unsigned)s_remaining;
          const bool mine = excl < rem0 && rem0 <= incl;
          const unsigned who = __ballot_sync(0xffffffffu, mine);
          if (mine) {
            unsigned r = rem0 - excl;
            int digit = lane * 8 + 7;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (c8[j] >= r) { digit = lane * 8 + j; break; }
              r -= c8[j];
            }
            s_prefix = pre | ((unsigned)digit << shift);
            s_remaining = (int)r;
          } else if (who == 0u && lane == 31) {
            s_prefix = pre | (255u << shift);
            s_remaining = (int)(rem0 - (incl - c8[7]));
          }
        }
        __syncthreads();
        mask |= 255u << shift;
      }
      const unsigned thr = s_prefix;
      const int need_eq = s_remaining;
      // ---- 3. ordered emission
      int base_out = 0, eq_seen = 0;
      for (int c0 = 0; c0 < nb; c0 += blockDim.x) {
        const int i = c0 + threadIdx.x;
        const unsigned v = i < nb ? sb[i] : 0xffffffffu;
        const int is_eq = (i < nb && v == thr) ? 1 : 0;
        int eq_total;
        const int eq_rank = block_exclusive_scan(is_eq, warp_sums, eq_total) + eq_seen;
        const int take = (i < nb && (v < thr || (is_eq && eq_rank < need_eq))) ? 1 : 0;
        int take_total;
        const int pos = block_exclusive_scan(take, warp_sums, take_total);
        if (take) p.victims[out0 + base_out + pos] = i;
        base_out += take_total;
        eq_seen += eq_total;
      }
    }
    __syncthreads();
  }
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_evict_score(kvs_pool* pool, const uint8_t* region_dev, const int32_t* created_dev,
                                      const int32_t* access_dev, const int32_t* seq_len_dev, int32_t n_seq,
                                      int32_t max_blocks, const float* init, const float* decay, int32_t n_regions,
                                      int64_t step, const int32_t* k_dev, float* scores_dev, int32_t* victims_dev,
                                      int64_t* victims_off_dev, cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "evict_score: null pool");
  if (n_seq < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "evict_score: bad sizes");
  if (n_regions < 1 || n_regions > kEvMaxRegions || !init || !decay)
    return fail(KVS_ERR_INVALID_ARG, "evict_score: 1 to 16 regions with host init/decay arrays");
  for (int r = 0; r < n_regions; ++r)
    if (!(init[r] >= 0.f) || !(decay[r] >= 0.f) || init[r] > 3.0e38f || decay[r] > 3.0e38f)
      return fail(KVS_ERR_INVALID_ARG, "evict_score: initial scores and decays must be finite and >= 0");
  if (pool->desc.block_tokens > 16) return fail(KVS_ERR_UNSUPPORTED, "evict_score: block_tokens above 16");
  if (n_seq == 0) return KVS_OK;
  if (!region_dev || !created_dev || !access_dev || !seq_len_dev || !k_dev || !scores_dev || !victims_dev ||
      !victims_off_dev)
    return fail(KVS_ERR_INVALID_ARG, "evict_score: null pointer");
  EvictParams p{};
  p.region = region_dev;
  p.created = created_dev;
  p.access = access_dev;
  p.seq_len = seq_len_dev;
  p.k = k_dev;
  p.scores = scores_dev;
  p.victims = victims_dev;
  p.victims_off = victims_off_dev;
  p.status = pool->status;
  p.n_seq = n_seq;
  p.max_blocks = max_blocks;
  p.B = pool->desc.block_tokens;
  p.n_regions = n_regions;
  p.step = step;
  for (int r = 0; r < n_regions; ++r) {
    p.init[r] = init[r];
    p.decay[r] = decay[r];
  }
  evict_kernel<<<std::min(n_seq, pool->num_sms * 2), 1024, 0, stream>>>(p);
  count_launch();
  return check_launch("evict_score");
}
