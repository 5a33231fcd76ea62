// Split-K merge of online-softmax partial states, shared by the decode
// attention kernels.  Each split s holds (m_s, l_s, acc_s[d]) in the log2
// domain; the merged output is
//   out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
// The caller is the last CTA of a (sequence, kv head) to arrive (see
// arrive_last); splits are read from L2 (__ldcg) in a fixed order, so results
// do not depend on which CTA merges.
#pragma once

#include "common.cuh"

namespace kvs {

// Arrival counter: returns true in exactly one CTA — the last of `expected`
// CTAs to call it for this counter — and resets the counter for the next
// launch.  Call after the CTA's partial results are written.
__device__ __forceinline__ bool arrive_last(int32_t* counter, int expected, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atomicAdd(counter, 1);
    *s_flag = (t == expected - 1);
    if (*s_flag) *counter = 0;
  }
  __syncthreads();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// 128-thread CTA merge of nsplit splits for g rows of width D: one warp per
// row finds the max and the normaliser with its lanes spread over the
// splits; then every thread accumulates a 4-column slice of a row, walking the
// splits with the loop unrolled so several loads are in flight.
template <int D>
__device__ __forceinline__ void merge_splits(const float* part, const float* part_ml, size_t s0, int nsplit, int g,
                                             float* out_rows, float* sM, float* sL) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < g; r += 4) {
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, __ldcg(part_ml + ((s0 + s) * g + r) * 2));
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Ls = 0.f;
    for (int s = lane; s < nsplit; s += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(part_ml + ((s0 + s) * g + r) * 2));
      Ls += ml.y > 0.f ? fast_exp2(ml.x - M) * ml.y : 0.f;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) {
      sM[r] = M;
      sL[r] = Ls;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < g * (D / 4); e += blockDim.x) {
    const int r = e / (D / 4), col = (e - r * (D / 4)) * 4;
    const float M = sM[r];
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < nsplit; ++s) {
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(part_ml + ((s0 + s) * g + r) * 2));
      const float4 x = __ldcg(reinterpret_cast<const float4*>(part + ((s0 + s) * g + r) * D + col));
      const float ws = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
      v.x += ws * x.x; v.y += ws * x.y; v.z += ws * x.z; v.w += ws * x.w;
    }
    const float Ls = sL[r];
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    *reinterpret_cast<float4*>(out_rows + (size_t)r * D + col) = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
  }
}

}  // namespace kvs
