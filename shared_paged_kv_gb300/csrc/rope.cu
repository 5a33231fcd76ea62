// Batched RoPE re-rotation of reused K blocks (INMS walkthrough §3.2: a
// block stored from p_s and reused at p_t is rotated by an angle depending
// only on p_t - p_s; V untouched; TokenDance summary section 2: one batched
// RoPE call per layer for the whole group of requests).
//
// Rotate-half pairing (i, i + d/2), frequency theta^(-2i/d), angles by the
// Cody-Waite reduced evaluation of common.cuh.  One CTA = one job x 64
// tokens, four warps.  Lane (token tl, vector v) of a warp step holds head
// dims [8v, 8v+8) and [d/2 + 8v, d/2 + 8v+8) of one token as two 16-byte
// vectors, so the 8 cos/sin pairs it needs depend on v only and stay in
// registers for the whole job; each token's low and high halves are 128-byte
// (d = 128) coalesced runs.  A lane walks all KV heads of its token: the
// block-table lookups and the index arithmetic are done once per token, and
// the heads are loaded in batches before any of them is stored (the stores
// go to the same slab, so the compiler could not move later loads above
// them).  The rotated rows are written with streaming stores: a layer's
// destinations are far larger than L2.  Rotation in fp32, rounding to bf16
// (RNE).
#include "common.cuh"
#include "internal.h"

namespace kvs {

struct RopeParams {
  uint16_t* slab;             // this layer's K slab, bf16 [cap][hkv][16][D]
  const int4* jobs;           // pairs of int4: (src_row, src_tok0, dst_row, dst_tok0), (n_tok, src_pos, dst_pos, -)
  const int32_t* src_table;
  const int32_t* dst_table;
  uint32_t* status;
  int n_jobs, max_blocks, hkv, capacity, tok_per_cta;
  RopeSplit rs;
};

constexpr int kRopeWarps = 4;
#ifndef KVS_ROPE_TOK_PER_CTA
#define KVS_ROPE_TOK_PER_CTA 64
#endif
constexpr int kRopeTokPerCta = KVS_ROPE_TOK_PER_CTA;
constexpr int kRopeB = 16;          // tokens per block of a bf16 pool
// Measured on the all-gather layer (524,288 rows, 8 KV heads): batches of
// 4 / 8 heads took 176 / 171 us with plain stores; streaming (evict-first)
// stores took the 8-head batch to 160 us.  64 tokens per CTA beat 32 and
// 128; capping registers for more CTAs per SM (spills, or 2-head batches)
// was slower.
#ifndef KVS_ROPE_HEAD_BATCH
#define KVS_ROPE_HEAD_BATCH 8
#endif
#ifndef KVS_ROPE_MIN_CTAS
#define KVS_ROPE_MIN_CTAS 1
#endif
constexpr int kRopeHeadBatch = KVS_ROPE_HEAD_BATCH;   // KV heads loaded before any is stored

template <int D>
__global__ void __launch_bounds__(kRopeWarps * 32, KVS_ROPE_MIN_CTAS) rope_rerotate_kernel(const __grid_constant__ RopeParams p) {
  constexpr int VEC = 8;                 // bf16 per 16-byte vector
  constexpr int NV = D / 2 / VEC;        // vectors per half row
  constexpr int TPW = 32 / NV;           // tokens per warp step
  constexpr int B = kRopeB, HB = kRopeHeadBatch;
  __shared__ float rsc[4 * 64];          // RoPE frequency pieces (lanes index them differently)
  const int job = blockIdx.x;
  const int4 j0 = __ldg(p.jobs + 2 * job), j1 = __ldg(p.jobs + 2 * job + 1);
  const int n_tok = j1.x;
  const int t0 = blockIdx.y * p.tok_per_cta;
  if (t0 >= n_tok) return;
  const int delta = j1.z - j1.y;
  if (delta <= -(1 << 18) || delta >= (1 << 18)) {
    if (threadIdx.x == 0) set_err(p.status, KVS_DEVERR_ROPE_RANGE);
    return;
  }
  for (int i = threadIdx.x; i < 4 * 64; i += blockDim.x) rsc[i] = p.rs.c[i >> 6][i & 63];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v = lane % NV, tl = lane / NV;
  float cs[VEC], sn[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) rope_cos_sin(rsc, v * VEC + e, delta, cs[e], sn[e]);
  const int t1 = min(n_tok, t0 + p.tok_per_cta);
  const long long lim = (long long)p.max_blocks * B;
  const size_t hstride = (size_t)B * D;   // elements between the KV heads of one token
  for (int t = t0 + warp * TPW + tl; t < t1; t += kRopeWarps * TPW) {
    const int ts = j0.y + t, td = j0.w + t;
    if (ts < 0 || td < 0 || ts >= lim || td >= lim) {
      set_err(p.status, KVS_DEVERR_JOB);
      continue;
    }
    const int bs = ts / B, bd = td / B;
    const int ps = __ldg(p.src_table + (size_t)j0.x * p.max_blocks + bs);
    const int pd = __ldg(p.dst_table + (size_t)j0.z * p.max_blocks + bd);
    if (ps < 0 || ps >= p.capacity || pd < 0 || pd >= p.capacity) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      continue;
    }
    const uint16_t* src = p.slab + ((size_t)ps * p.hkv * B + (ts - bs * B)) * D + v * VEC;
    uint16_t* dst = p.slab + ((size_t)pd * p.hkv * B + (td - bd * B)) * D + v * VEC;
    for (int h0 = 0; h0 < p.hkv; h0 += HB) {
      uint4 lo[HB], hi[HB];
#pragma unroll
      for (int k = 0; k < HB; ++k) {
        if (h0 + k < p.hkv) {
          lo[k] = __ldg(reinterpret_cast<const uint4*>(src + (h0 + k) * hstride));
          hi[k] = __ldg(reinterpret_cast<const uint4*>(src + (h0 + k) * hstride + D / 2));
        }
      }
#pragma unroll
      for (int k = 0; k < HB; ++k) {
        if (h0 + k >= p.hkv) break;
        const uint32_t lw[4] = {lo[k].x, lo[k].y, lo[k].z, lo[k].w};
        const uint32_t hw[4] = {hi[k].x, hi[k].y, hi[k].z, hi[k].w};
        uint32_t ol[4], oh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = bf16_lo(lw[e]), a1 = bf16_hi(lw[e]);
          const float b0 = bf16_lo(hw[e]), b1 = bf16_hi(hw[e]);
          ol[e] = pack_bf16(a0 * cs[2 * e] - b0 * sn[2 * e], a1 * cs[2 * e + 1] - b1 * sn[2 * e + 1]);
          oh[e] = pack_bf16(b0 * cs[2 * e] + a0 * sn[2 * e], b1 * cs[2 * e + 1] + a1 * sn[2 * e + 1]);
        }
        uint16_t* o = dst + (h0 + k) * hstride;
        __stcs(reinterpret_cast<uint4*>(o), make_uint4(ol[0], ol[1], ol[2], ol[3]));
        __stcs(reinterpret_cast<uint4*>(o + D / 2), make_uint4(oh[0], oh[1], oh[2], oh[3]));
      }
    }
  }
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_rope_rerotate(kvs_pool* pool, int32_t layer, const kvs_rope_job* jobs_dev, int32_t n_jobs,
                                        int32_t max_job_tokens, float theta, const int32_t* src_table_dev,
                                        const int32_t* dst_table_dev, int32_t max_blocks, cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: null pool");
  const kvs_pool_desc& d = pool->desc;
  if (d.dtype != KVS_DTYPE_BF16 || d.block_tokens != kRopeB)
    return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: bf16 pools (16-token blocks) only");
  if (layer < 0 || layer >= d.num_layers) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: layer out of range");
  if (n_jobs < 0 || max_job_tokens < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: bad sizes");
  if (!(theta > 0.f)) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: theta must be positive");
  if (n_jobs == 0 || max_job_tokens == 0) return KVS_OK;
  if (!jobs_dev || !src_table_dev || !dst_table_dev) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: null pointer");
  if (!aligned16(jobs_dev)) return fail(KVS_ERR_INVALID_ARG, "rope_rerotate: jobs must be 16-byte aligned");
  RopeParams p{};
  p.slab = static_cast<uint16_t*>(pool->k[layer]);
  p.jobs = reinterpret_cast<const int4*>(jobs_dev);
  p.src_table = src_table_dev;
  p.dst_table = dst_table_dev;
  p.status = pool->status;
  p.n_jobs = n_jobs;
  p.max_blocks = max_blocks;
  p.hkv = d.num_kv_heads;
  p.capacity = d.capacity_blocks;
  p.tok_per_cta = kRopeTokPerCta;
  rope_split_host(theta, d.head_dim, p.rs.c);
  dim3 grid(n_jobs, (max_job_tokens + p.tok_per_cta - 1) / p.tok_per_cta);
  if (grid.y > 65535) return fail(KVS_ERR_CAPACITY, "rope_rerotate: max_job_tokens too large");
  if (d.head_dim == 128)
    rope_rerotate_kernel<128><<<grid, kRopeWarps * 32, 0, stream>>>(p);
  else
    rope_rerotate_kernel<64><<<grid, kRopeWarps * 32, 0, stream>>>(p);
  count_launch();
  return check_launch("rope_rerotate");
}
