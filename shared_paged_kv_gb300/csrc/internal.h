// Host-side internals of libkvs shared by the translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <string>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kvs.h"

struct kvs_pool {
  kvs_pool_desc desc;
  int device = 0;
  int num_sms = 0;
  std::vector<void*> k, v, ksb, vsb, dk, dv;    // per-layer device slabs (not owned)
  std::vector<CUtensorMap> tk, tv, tdk, tdv;    // TMA maps per layer
  std::vector<CUtensorMap> tk1, tv1;           // bf16 head_dim 128: one 64-column half of a block per copy
  uint32_t* status = nullptr;                   // device status word [0] and token-major claim counter [1] (owned)
  int32_t* tickets = nullptr;                   // split-K arrival counters (owned)
  size_t n_tickets = 0;
  // every per-layer slab that holds block contents (K, V and, for Q4, the
  // scale/bias slabs) with its bytes per physical block, on the device
  // (owned): what a block copy must move
  void** blk_slabs = nullptr;
  long long* blk_bytes = nullptr;
  long long* blk_offs = nullptr;   // offset of each slab's bytes inside one packed block record
  int n_blk_slabs = 0;
  long long blk_record = 0;        // bytes of one packed block record (all slabs)
  uint32_t test_flags = 0;         // KVS_TEST_* (tests only)
};

namespace kvs {

void set_error(const std::string& msg);
kvs_status fail(kvs_status st, const std::string& msg);
kvs_status check_launch(const char* what);
void count_launch(uint64_t n = 1);
bool aligned16(const void* p);

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute belongs to the device's context).  Safe to call from several
// threads: a repeated set is harmless.  Returns false on a CUDA error.
template <auto Kern>
bool smem_limit_once(int smem, int device) {
  static std::atomic<uint64_t> done{0};   // bit d: set on device d < 64
  const uint64_t bit = device >= 0 && device < 64 ? (uint64_t{1} << device) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
  if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

// RoPE frequency split (see common.cuh): c[piece][i] for i < head_dim/2.
void rope_split_host(float theta, int head_dim, float out[4][64]);

// Split-K plan for decode attention: blocks per CTA chunk and chunk count.
struct AttnPlan {
  int bpc;        // logical blocks per CTA
  int n_chunks;   // CTAs per (sequence, kv head)
};
AttnPlan attn_plan(const kvs_pool* pool, int n_seq, int max_blocks);   // bf16 path
AttnPlan q4_plan(const kvs_pool* pool, int n_seq, int max_blocks);     // Q4 path
constexpr int kAttnWarps = 4;

// Token-major persistent decode attention (query group <= 8), attn_tm.cu.
kvs_status decode_attn_token_major(kvs_pool* pool, int layer, const void* q, int n_q_heads, const int32_t* table,
                                   int max_blocks, const int32_t* seq_len, int n_seq, const int32_t* diff,
                                   const int32_t* rope_off, const kvs_seg_rope* rope_segs, float theta,
                                   float scale, float* out, void* ws, cudaStream_t stream);
size_t tm_workspace_bytes(const kvs_pool* pool, int n_seq, int max_blocks, int g);
bool tm_wide_tile(const kvs_pool* pool, int g, bool rope);
kvs_status decode_plan_token_major(kvs_pool* pool, int n_q_heads, const int32_t* table, int max_blocks,
                                   const int32_t* seq_len, int n_seq, const int32_t* diff, const int32_t* rope_off,
                                   const kvs_seg_rope* rope_segs, void* ws, cudaStream_t stream);
constexpr int kTmMaxGroup = 8;
// Small calls: up to this many (sequence, KV head, logical block) triples a
// call with a query group <= 8 runs on the 16-row kernel alone (attn.cu: one
// launch, no plan, no separate merge), whose fixed cost is lower than the
// planned token-major path's three launches.  The 4-agent, 24-block layer
// (192 triples) took 12.9 us per layer there against 17.0 us planned; 16,384
// sequences of that shape (786,432 triples) took 2.31 ms against 0.70 ms.
constexpr long long kSmallCallWork = 2048;
// small calls whose block tables are at most this long run one chunk per
// (sequence, KV head): at most 8 blocks per warp, no split merge
constexpr int kSmallOneChunk = 32;
inline bool small_call(int n_seq, int num_kv_heads, int max_blocks, int g) {
  return g <= kTmMaxGroup && (long long)n_seq * num_kv_heads * max_blocks <= kSmallCallWork;
}

// Wide shared tile (attn_wide.cu): tcgen05 attention of a sharing group's
// W * G query rows over the blocks the group shares.  Writes the shared splits
// (p2, p2_ml) of the token-major plan; the split merge combines them.
struct WideParams {
  const uint16_t* q;        // [n_seq][hq][128] bf16
  const int4* witems;       // {kind | group, chunk, end block, member mask}
  const int* hdr;           // plan header ([8]: number of wide items)
  const int2* wsub;        // [item][max_sub][8] {sharing members, physical block} per block
  const int2* wmem;        // rotation calls: [item][32] {split slot, RoPE shift} per member
  const int4* wclaims;     // rotation calls: claims {group, first item, items | slot << 16, members}
  float* p2;                // [n_seq][hkv][n_chunks][g][128]
  float* p2_ml;             // [n_seq][hkv][g][n_chunks][2]
  uint32_t* status;
  int n_seq, max_blocks, hkv, g, hq, W, ib, n_chunks, R, capacity, max_sub;   // ib, n_chunks: shared chunks
  int ibp;                  // private chunk blocks (plan header check)
  int max_witems;           // item capacity (the plan's counter may run past it)
  int runs;                 // rotation call: items are 8-block runs, per-member shift and slot
  int magic;                // plan header check: magic, n_seq, max_blocks, R, ibp, hkv, W, ib
  float scale_log2;
  float rs[4][64];          // RoPE frequency pieces (rotation calls), as RopeSplit::c
};
// The plan header (the first 12 of its 16 ints), read with three 16-byte
// loads that are all in flight at once.  A check written as a chain of
// short-circuit compares on the header would make each load wait for the
// compare before it.  The loads are plain (L1-cached) loads: every warp of
// every CTA reads the same line, and loads that bypass L1 would queue all of
// those requests at one L2 slice.
struct PlanHdr {
  int v[12];
};
__device__ __forceinline__ PlanHdr load_plan_hdr(const int* hdr) {
  const int4* h4 = reinterpret_cast<const int4*>(hdr);
  const int4 a = h4[0], b = h4[1], c = h4[2];
  return PlanHdr{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w}};
}

// CTAs of the wide tile's grid for rotation calls (attn_tm.cu)
int runs_wide_ctas(const kvs_pool* pool);
kvs_status launch_wide_tile(const WideParams& p, const kvs_pool* pool, int layer, int max_claims,
                            cudaStream_t stream);

// Mirror construction (mirror.cu).
size_t mirror_workspace_bytes(int n_seq, int max_blocks);

// Block lifetime (blocks.cu).
size_t blocks_workspace_bytes(int capacity, int n_items);

}  // namespace kvs
