// Critical-position selection by K difference (TokenDance summary, section 2:
// at check layers one batched difference computation finds, per request, the
// positions whose cached and newly computed K differ most).
//
// Pass 1 (HBM-bound): one warp per position row streams both bf16 rows with
// 16-byte loads and reduces sum((a-b)^2) in fp32 — the squared L2 norm, whose
// order equals the norm's.  Pass 2: one CTA per agent finds the k-th largest
// score by a 4 x 8-bit radix select on the float bits (scores are >= 0, so
// the bit pattern orders them), then emits, in ascending position order, every
// position above the threshold and the lowest-positioned ones equal to it.
#include <string>

#include "common.cuh"
#include "internal.h"

namespace kvs {

// The rows sel_scores writes: [row_off[0], row_off[n_agents]) clipped to the
// score buffer [0, cap_rows).
__device__ __forceinline__ long long rows_lo(const int64_t* row_off) { return row_off[0] > 0 ? row_off[0] : 0; }
__device__ __forceinline__ long long rows_hi(const int64_t* row_off, int n_agents, long long cap_rows) {
  return row_off[n_agents] < cap_rows ? row_off[n_agents] : cap_rows;
}

// Rows of agent a, or 0 when its range is malformed: a range that ends
// before it starts or leaves the scored rows [lo, hi) selects nothing, so
// every score the selection reads was written by sel_scores in the same call.
__device__ __forceinline__ int agent_rows(const int64_t* row_off, int a, long long lo, long long hi) {
  const long long r0 = row_off[a], r1 = row_off[a + 1];
  if (r0 < lo || r1 < r0 || r1 > hi) return 0;
  return static_cast<int>(r1 - r0);
}

__global__ void sel_scores(const uint16_t* __restrict__ kc, const uint16_t* __restrict__ kn,
                           const int64_t* __restrict__ row_off, int n_agents, int row_elems,
                           long long cap_rows, float* __restrict__ scores) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row < rows_lo(row_off) || row >= rows_hi(row_off, n_agents, cap_rows)) return;
  const uint4* a = reinterpret_cast<const uint4*>(kc + row * row_elems);
  const uint4* b = reinterpret_cast<const uint4*>(kn + row * row_elems);
  float acc = 0.f;
  for (int v = lane; v < row_elems / 8; v += 32) {
    const uint4 x = __ldg(a + v), y = __ldg(b + v);
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float d0 = bf16_lo(xs[e]) - bf16_lo(ys[e]);
      const float d1 = bf16_hi(xs[e]) - bf16_hi(ys[e]);
      acc = fmaf(d0, d0, acc);
      acc = fmaf(d1, d1, acc);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) scores[row] = acc;
}

__device__ __forceinline__ int count_for(float ratio, int n) {
  double k = ceil(static_cast<double>(ratio) * static_cast<double>(n));
  if (k < 0) k = 0;
  if (k > n) k = n;
  return static_cast<int>(k);
}

constexpr int kSelUnroll = 8;   // scores a thread loads at once in a radix pass

__global__ void __launch_bounds__(1024) sel_topk(const float* __restrict__ scores, const int64_t* __restrict__ row_off,
                                                 int n_agents, float ratio, long long cap_rows,
                                                 int32_t* __restrict__ idx_out, int64_t* __restrict__ idx_off) {
  __shared__ unsigned hist[256];
  __shared__ int warp_sums[32];
  __shared__ unsigned s_prefix;
  __shared__ int s_remaining;
  const int a = blockIdx.x;
  const long long lo = rows_lo(row_off), hi = rows_hi(row_off, n_agents, cap_rows);
  const int n = agent_rows(row_off, a, lo, hi);
  const int64_t r0 = n > 0 ? row_off[a] : 0;   // rows [r0, r0 + n) lie in [lo, hi) when n > 0
  const int k = count_for(ratio, n);
  // exclusive prefix of k over agents: the earlier agents' counts, summed
  // over the CTA
  {
    long long part = 0;
    for (int b = threadIdx.x; b < a; b += blockDim.x) part += count_for(ratio, agent_rows(row_off, b, lo, hi));
    __shared__ long long s_part[32];
#pragma unroll
    for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t o = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) o += s_part[w];
      idx_off[a] = o;
      if (a == n_agents - 1) idx_off[n_agents] = o + k;
      s_prefix = 0u;
      s_remaining = k;
    }
  }
  __syncthreads();
  const int64_t out0 = idx_off[a];
  if (k == 0) return;
  const unsigned* sb = reinterpret_cast<const unsigned*>(scores + r0);
  // radix select of the k-th largest bit pattern, 8 bits at a time from the top
  unsigned mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    const unsigned pre = s_prefix;
    // kSelUnroll scores per thread at a time, their loads in flight together
    for (int i0 = threadIdx.x; i0 < n; i0 += kSelUnroll * blockDim.x) {
      unsigned v[kSelUnroll];
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u) {
        const int i = i0 + u * blockDim.x;
        v[u] = i < n ? sb[i] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u)
        if (i0 + u * (int)blockDim.x < n && (v[u] & mask) == pre) atomicAdd(&hist[(v[u] >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the digit: from the top, the first bin whose running count reaches
      // the remaining rank (bin 0 if none does before it); lane l scans bins
      // 255 - 8l .. 248 - 8l after a prefix sum of the lanes' totals
      const int lane = threadIdx.x;
      unsigned c8[8], lsum = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c8[j] = hist[255 - (lane * 8 + j)];
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
        int digit = 255 - (lane * 8 + 7);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (c8[j] >= r) { digit = 255 - (lane * 8 + j); break; }
          r -= c8[j];
        }
        s_prefix = pre | ((unsigned)digit << shift);
        s_remaining = (int)r;
      } else if (who == 0u && lane == 31) {
        s_prefix = pre;   // digit 0
        s_remaining = (int)(rem0 - (incl - c8[7]));
      }
    }
    __syncthreads();
    mask |= 255u << shift;
  }
  const unsigned thr = s_prefix;
  const int need_eq = s_remaining;    // how many positions equal to thr to keep
  // ordered emission (the next chunk's score is loaded before this one's scans)
  int base_out = 0, eq_seen = 0;
  unsigned v_next = (int)threadIdx.x < n ? sb[threadIdx.x] : 0u;
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const unsigned v = v_next;
    v_next = i + (int)blockDim.x < n ? sb[i + blockDim.x] : 0u;
    const int is_eq = (i < n && v == thr) ? 1 : 0;
    int eq_total;
    const int eq_rank = block_exclusive_scan(is_eq, warp_sums, eq_total) + eq_seen;
    const int take = (i < n && (v > thr || (is_eq && eq_rank < need_eq))) ? 1 : 0;
    int take_total;
    const int pos = block_exclusive_scan(take, warp_sums, take_total);
    if (take) idx_out[out0 + base_out + pos] = i;
    base_out += take_total;
    eq_seen += eq_total;
  }
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_select_critical(const void* k_cached_dev, const void* k_new_dev, const int64_t* row_off_dev,
                                          int32_t n_agents, int32_t max_rows_per_agent, int32_t row_elems, float ratio,
                                          int32_t* idx_out_dev, int64_t* idx_off_dev, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
  if (n_agents < 0 || max_rows_per_agent < 0 || max_rows_per_agent > 65536 || row_elems < 8 || row_elems % 8)
    return fail(KVS_ERR_INVALID_ARG, "select_critical: bad sizes (row_elems must be a positive multiple of 8)");
  if (!row_off_dev || !idx_off_dev) return fail(KVS_ERR_INVALID_ARG, "select_critical: null pointer");
  if (n_agents == 0) return KVS_OK;
  if (!k_cached_dev || !k_new_dev || !idx_out_dev || !ws) return fail(KVS_ERR_INVALID_ARG, "select_critical: null pointer");
  if (!aligned16(k_cached_dev) || !aligned16(k_new_dev) || !aligned16(ws))
    return fail(KVS_ERR_INVALID_ARG, "select_critical: K buffers and ws must be 16-byte aligned");
  if (!(ratio >= 0.f)) return fail(KVS_ERR_INVALID_ARG, "select_critical: ratio must be >= 0");
  const long long rows = (long long)n_agents * max_rows_per_agent;
  if ((size_t)rows * sizeof(float) > ws_bytes) return fail(KVS_ERR_CAPACITY, "select_critical: workspace too small");
  float* scores = static_cast<float*>(ws);
  const long long threads = rows * 32;
  const int tb = 256;
  if (rows > 0) {
    sel_scores<<<(unsigned)((threads + tb - 1) / tb), tb, 0, stream>>>(
        static_cast<const uint16_t*>(k_cached_dev), static_cast<const uint16_t*>(k_new_dev), row_off_dev, n_agents,
        row_elems, rows, scores);
    count_launch();
  }
  sel_topk<<<n_agents, 1024, 0, stream>>>(scores, row_off_dev, n_agents, ratio, rows, idx_out_dev, idx_off_dev);
  count_launch();
  return check_launch("select_critical");
}

// ---------------------------------------------------------------------------
// kvs_select_critical_noalloc: the same selection for callers that cannot
// allocate device memory on the call path.  Its only scratch (one fp32 score
// per position row) lives in this file-scope device array, reserved on every
// device where the library's device code is loaded and held until the
// process exits.  Host code never uses the array's name as a pointer: every
// call asks the runtime for the array's device address in the current context
// (cudaGetSymbolAddress, a lookup that allocates nothing).  The address is not
// cached, because a device reset or a new primary context reloads the device
// code at another address.
namespace kvs {
constexpr long long kSelNoallocMaxRows = 1ll << 20;   // 4 MiB of scores
static __device__ __align__(256) float g_sel_scores[kSelNoallocMaxRows];
}  // namespace kvs

extern "C" kvs_status kvs_select_critical_noalloc(const void* k_cached_dev, const void* k_new_dev,
                                                  const int64_t* row_off_dev, int32_t n_agents,
                                                  int32_t max_rows_per_agent, int32_t row_elems, float ratio,
                                                  int32_t* idx_out_dev, int64_t* idx_off_dev,
                                                  cudaStream_t stream) {
  if (n_agents < 0 || max_rows_per_agent < 0 || max_rows_per_agent > 65536 || row_elems < 8 || row_elems % 8)
    return fail(KVS_ERR_INVALID_ARG, "select_critical_noalloc: bad sizes (row_elems must be a positive multiple of 8)");
  const long long rows = (long long)n_agents * max_rows_per_agent;
  if (rows > kSelNoallocMaxRows)
    return fail(KVS_ERR_CAPACITY, "select_critical_noalloc: n_agents * max_rows_per_agent exceeds the fixed scratch "
                                  "of 1048576 rows; use kvs_select_critical with a caller workspace");
  if (!row_off_dev || !idx_off_dev) return fail(KVS_ERR_INVALID_ARG, "select_critical_noalloc: null pointer");
  if (n_agents == 0) return KVS_OK;
  if (!k_cached_dev || !k_new_dev || !idx_out_dev) return fail(KVS_ERR_INVALID_ARG, "select_critical_noalloc: null pointer");
  if (!aligned16(k_cached_dev) || !aligned16(k_new_dev))
    return fail(KVS_ERR_INVALID_ARG, "select_critical_noalloc: K buffers must be 16-byte aligned");
  if (!(ratio >= 0.f)) return fail(KVS_ERR_INVALID_ARG, "select_critical_noalloc: ratio must be >= 0");
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_sel_scores);
  if (e != cudaSuccess || !ptr)
    return fail(KVS_ERR_CUDA, std::string("select_critical_noalloc: cudaGetSymbolAddress failed: ") +
                                  cudaGetErrorString(e));
  float* scores = static_cast<float*>(ptr);
  // Every score the selection reads is written by sel_scores in this call
  // (rows [row_off[0], row_off[n_agents]) below the capacity; an agent whose
  // range is malformed or leaves those rows reads nothing), so nothing in the
  // array has to start at zero.
  const long long threads = rows * 32;
  const int tb = 256;
  if (rows > 0) {
    sel_scores<<<(unsigned)((threads + tb - 1) / tb), tb, 0, stream>>>(
        static_cast<const uint16_t*>(k_cached_dev), static_cast<const uint16_t*>(k_new_dev), row_off_dev, n_agents,
        row_elems, rows, scores);
    count_launch();
  }
  sel_topk<<<n_agents, 1024, 0, stream>>>(scores, row_off_dev, n_agents, ratio, rows, idx_out_dev, idx_off_dev);
  count_launch();
  return check_launch("select_critical_noalloc");
}
