// libkvs host side: pool lifetime, TMA tensor maps, workspace sizing, status
// and statistics.  No kernels of the hot path live here.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "internal.h"

namespace kvs {

static thread_local std::string g_last_error = "no error";
static std::atomic<uint64_t> g_launches{0};

void set_error(const std::string& msg) { g_last_error = msg; }

kvs_status fail(kvs_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

kvs_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return KVS_OK;
}

void count_launch(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void rope_split_host(float theta, int head_dim, float out[4][64]) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int p = 0; p < 4; ++p)
    for (int i = 0; i < 64; ++i) out[p][i] = 0.f;
  for (int i = 0; i < head_dim / 2; ++i) {
    const double w = std::pow(static_cast<double>(theta), -2.0 * i / head_dim);
    double f = w / two_pi;                       // turns per position
    const double c0 = std::floor(f * 64.0) / 64.0;
    f -= c0;
    const double c1 = std::floor(f * 4096.0) / 4096.0;
    f -= c1;
    const double c2 = std::floor(f * 262144.0) / 262144.0;
    f -= c2;
    out[0][i] = static_cast<float>(c0);
    out[1][i] = static_cast<float>(c1);
    out[2][i] = static_cast<float>(c2);
    out[3][i] = static_cast<float>(f);
  }
}

AttnPlan attn_plan(const kvs_pool* pool, int n_seq, int max_blocks) {
  // Aim at ~8 CTAs per SM over the whole grid (2 resident, 4 waves) so that
  // ragged contexts balance; chunks are a multiple of the warp count.
  const long long work = static_cast<long long>(n_seq) * pool->desc.num_kv_heads * max_blocks;
  const long long target = static_cast<long long>(pool->num_sms) * 8;
  long long bpc = (work + target - 1) / target;
  bpc = ((bpc + kAttnWarps - 1) / kAttnWarps) * kAttnWarps;
  if (bpc < 8) bpc = 8;
  if (bpc > 256) bpc = 256;
  AttnPlan p;
  p.bpc = static_cast<int>(bpc);
  p.n_chunks = (max_blocks + p.bpc - 1) / p.bpc;
  if (p.n_chunks < 1) p.n_chunks = 1;
  return p;
}

// ------------------------------------------------------------ tensor maps ---
static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 slab [rows][head_dim] seen as a 3-D tensor {64 elements, rows,
// head_dim/64 halves} (row stride head_dim*2 bytes, half stride 128 bytes), so
// one box {64, block_tokens, head_dim/64} with 128-byte swizzle brings a whole
// block tile in one copy, laid out in shared memory as [half][row][64]: each
// half is a 16-row x 128-byte swizzled panel, which keeps ldmatrix free of
// bank conflicts.
// With halves = 1 the box takes one 64-column half of a block (used where a
// tile of several blocks is laid out as [half][token][64]).
static bool encode_bf16_slab(CUtensorMap* m, void* base, long long rows, int head_dim, int box_rows,
                             int halves = 0) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(head_dim / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(halves > 0 ? halves : head_dim / 64)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Q4 code slab [rows][64 bytes] (head_dim 128) as uint8 {64, rows}; box
// {64, block_tokens}; 64-byte swizzle.
static bool encode_q4_slab(CUtensorMap* m, void* base, long long rows, int row_bytes, int box_rows) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace kvs

using namespace kvs;

extern "C" {

const char* kvs_last_error_string(void) { return g_last_error.c_str(); }

uint64_t kvs_launch_count(void) { return g_launches.load(); }

kvs_status kvs_pool_create(const kvs_pool_desc* d, void* const* k_layers, void* const* v_layers,
                           void* const* k_sb_layers, void* const* v_sb_layers, void* const* dk_layers,
                           void* const* dv_layers, kvs_pool** out) {
  if (!d || !out || !k_layers || !v_layers) return fail(KVS_ERR_INVALID_ARG, "pool_create: null argument");
  *out = nullptr;
  if (d->num_layers < 1 || d->num_kv_heads < 1 || d->capacity_blocks < 1 || d->max_seqs < 1 ||
      d->diff_capacity_blocks < 0)
    return fail(KVS_ERR_INVALID_ARG, "pool_create: sizes must be positive");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(KVS_ERR_UNSUPPORTED, "pool_create: head_dim must be 64 or 128");
  const bool q4 = d->dtype == KVS_DTYPE_Q4G64;
  if (d->dtype != KVS_DTYPE_BF16 && !q4) return fail(KVS_ERR_INVALID_ARG, "pool_create: unknown dtype");
  if (!q4 && d->block_tokens != 16)
    return fail(KVS_ERR_UNSUPPORTED, "pool_create: bf16 pools use 16-token blocks");
  if (q4 && (d->block_tokens != 256 || d->head_dim != 128))
    return fail(KVS_ERR_UNSUPPORTED, "pool_create: Q4G64 pools use 256-token blocks and head_dim 128");
  if (q4 && (!k_sb_layers || !v_sb_layers))
    return fail(KVS_ERR_INVALID_ARG, "pool_create: Q4G64 needs scale/bias slabs");
  if (!q4 && (k_sb_layers || v_sb_layers))
    return fail(KVS_ERR_INVALID_ARG, "pool_create: scale/bias slabs are for Q4G64 pools only");
  if (d->diff_capacity_blocks > 0 && (!dk_layers || !dv_layers))
    return fail(KVS_ERR_INVALID_ARG, "pool_create: diff slabs missing");
  const long long rows = static_cast<long long>(d->capacity_blocks) * d->num_kv_heads * d->block_tokens;
  // Q4 pools keep mirror diffs per 16-token sub-block of their 256-token blocks
  const long long drows = static_cast<long long>(d->diff_capacity_blocks) * d->num_kv_heads * (q4 ? 16 : d->block_tokens);
  if (rows > 0x7FFFFFFFll || drows > 0x7FFFFFFFll)
    return fail(KVS_ERR_CAPACITY, "pool_create: capacity * kv_heads * block_tokens must fit in int32");

  kvs_pool* p = new kvs_pool();
  p->desc = *d;
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return fail(KVS_ERR_CUDA, "pool_create: cannot query the current device");
  }
  const int L = d->num_layers;
  for (int l = 0; l < L; ++l) {
    const bool bad = !k_layers[l] || !v_layers[l] || !aligned16(k_layers[l]) || !aligned16(v_layers[l]) ||
                     (q4 && (!k_sb_layers[l] || !v_sb_layers[l] || !aligned16(k_sb_layers[l]) ||
                             !aligned16(v_sb_layers[l]))) ||
                     (d->diff_capacity_blocks > 0 &&
                      (!dk_layers[l] || !dv_layers[l] || !aligned16(dk_layers[l]) || !aligned16(dv_layers[l])));
    if (bad) {
      delete p;
      return fail(KVS_ERR_INVALID_ARG, "pool_create: a layer slab pointer is null or not 16-byte aligned");
    }
    p->k.push_back(k_layers[l]);
    p->v.push_back(v_layers[l]);
    if (q4) {
      p->ksb.push_back(k_sb_layers[l]);
      p->vsb.push_back(v_sb_layers[l]);
    }
    if (d->diff_capacity_blocks > 0) {
      p->dk.push_back(dk_layers[l]);
      p->dv.push_back(dv_layers[l]);
    }
  }
  p->tk.resize(L);
  p->tv.resize(L);
  if (d->diff_capacity_blocks > 0) {
    p->tdk.resize(L);
    p->tdv.resize(L);
  }
  for (int l = 0; l < L; ++l) {
    bool ok;
    if (q4) {
      ok = encode_q4_slab(&p->tk[l], p->k[l], rows, d->head_dim / 2, d->block_tokens) &&
           encode_q4_slab(&p->tv[l], p->v[l], rows, d->head_dim / 2, d->block_tokens);
    } else {
      ok = encode_bf16_slab(&p->tk[l], p->k[l], rows, d->head_dim, d->block_tokens) &&
           encode_bf16_slab(&p->tv[l], p->v[l], rows, d->head_dim, d->block_tokens);
      if (ok && d->head_dim == 128 && d->block_tokens == 16) {
        if (p->tk1.empty()) {
          p->tk1.resize(L);
          p->tv1.resize(L);
        }
        ok = encode_bf16_slab(&p->tk1[l], p->k[l], rows, d->head_dim, d->block_tokens, 1) &&
             encode_bf16_slab(&p->tv1[l], p->v[l], rows, d->head_dim, d->block_tokens, 1);
      }
      if (ok && d->diff_capacity_blocks > 0)
        ok = encode_bf16_slab(&p->tdk[l], p->dk[l], drows, d->head_dim, d->block_tokens) &&
             encode_bf16_slab(&p->tdv[l], p->dv[l], drows, d->head_dim, d->block_tokens);
    }
    if (!ok) {
      delete p;
      return fail(KVS_ERR_CUDA, "pool_create: cuTensorMapEncodeTiled failed");
    }
  }
  // slabs a block copy moves, with their bytes per physical block
  std::vector<void*> slabs;
  std::vector<long long> sbytes;
  const long long per_block_rows = static_cast<long long>(d->num_kv_heads) * d->block_tokens;
  for (int l = 0; l < L; ++l) {
    const long long row = q4 ? d->head_dim / 2 : d->head_dim * 2;
    slabs.push_back(p->k[l]); sbytes.push_back(per_block_rows * row);
    slabs.push_back(p->v[l]); sbytes.push_back(per_block_rows * row);
    if (q4) {
      const long long sb = (d->head_dim / 64) * 4;   // fp16 scale + bias per 64-element group
      slabs.push_back(p->ksb[l]); sbytes.push_back(per_block_rows * sb);
      slabs.push_back(p->vsb[l]); sbytes.push_back(per_block_rows * sb);
    }
  }
  std::vector<long long> soffs(sbytes.size());
  long long rec = 0;
  for (size_t i = 0; i < sbytes.size(); ++i) {
    soffs[i] = rec;
    rec += sbytes[i];
  }
  p->n_blk_slabs = static_cast<int>(slabs.size());
  p->blk_record = rec;
  if (cudaMalloc(&p->blk_slabs, slabs.size() * sizeof(void*)) != cudaSuccess ||
      cudaMalloc(&p->blk_bytes, sbytes.size() * sizeof(long long)) != cudaSuccess ||
      cudaMalloc(&p->blk_offs, soffs.size() * sizeof(long long)) != cudaSuccess ||
      cudaMemcpy(p->blk_slabs, slabs.data(), slabs.size() * sizeof(void*), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(p->blk_bytes, sbytes.data(), sbytes.size() * sizeof(long long), cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemcpy(p->blk_offs, soffs.data(), soffs.size() * sizeof(long long), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(p->blk_slabs);
    cudaFree(p->blk_bytes);
    cudaFree(p->blk_offs);
    delete p;
    return fail(KVS_ERR_CUDA, "pool_create: cannot allocate the slab list");
  }
  p->n_tickets = static_cast<size_t>(d->max_seqs) * d->num_kv_heads;
  if (cudaMalloc(&p->status, 16) != cudaSuccess ||
      cudaMalloc(&p->tickets, p->n_tickets * sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(p->status, 0, 16) != cudaSuccess ||
      cudaMemset(p->tickets, 0, p->n_tickets * sizeof(int32_t)) != cudaSuccess) {
    cudaFree(p->status);
    cudaFree(p->tickets);
    cudaFree(p->blk_slabs);
    cudaFree(p->blk_bytes);
    cudaFree(p->blk_offs);
    delete p;
    return fail(KVS_ERR_CUDA, "pool_create: cannot allocate the status word / counters");
  }
  *out = p;
  return KVS_OK;
}

kvs_status kvs_pool_destroy(kvs_pool* p) {
  if (!p) return fail(KVS_ERR_INVALID_ARG, "pool_destroy: null pool");
  cudaFree(p->status);
  cudaFree(p->tickets);
  cudaFree(p->blk_slabs);
  cudaFree(p->blk_bytes);
  cudaFree(p->blk_offs);
  delete p;
  return KVS_OK;
}

kvs_status kvs_workspace_size(const kvs_pool* p, int32_t op, int32_t n_seq, int32_t max_blocks,
                              int32_t n_q_heads, size_t* bytes) {
  if (!p || !bytes || n_seq < 0 || max_blocks < 0) return fail(KVS_ERR_INVALID_ARG, "workspace_size: bad argument");
  size_t b = 0;
  switch (op) {
    case KVS_OP_DEDUP: {
      // hash table (16 B per entry, power of two >= 2 x slots) + per-slot
      // arrays: key (8), rep (4), segstart (4), flag/id (4), + scan scratch
      const size_t slots = static_cast<size_t>(n_seq) * max_blocks;
      size_t t = 1024;
      while (t < 2 * slots) t <<= 1;
      // + per-chunk reference counts of the optional CSR (32 x min(capacity, slots))
      b = t * 16 + slots * (8 + 4 + 4 + 4 + 4) + 64 * 1024 + 256 +
          32ull * std::min<size_t>(p->desc.capacity_blocks, slots) * 4 + 256;
      break;
    }
    case KVS_OP_DECODE_ATTN:
    case KVS_OP_DECODE_ATTN_Q4: {
      if (n_q_heads < 1 || n_q_heads % p->desc.num_kv_heads) return fail(KVS_ERR_INVALID_ARG, "workspace_size: n_q_heads");
      const int g = n_q_heads / p->desc.num_kv_heads;
      const AttnPlan plan = op == KVS_OP_DECODE_ATTN ? attn_plan(p, n_seq, max_blocks) : q4_plan(p, n_seq, max_blocks);
      const size_t splits = static_cast<size_t>(n_seq) * p->desc.num_kv_heads * plan.n_chunks * kAttnWarps;
      b = splits * g * (p->desc.head_dim + 2) * sizeof(float) + 256;
      // query groups <= 8: the planned token-major path, and for small calls
      // also the 16-row kernel (either may run: see KVS_TEST_TOKEN_MAJOR)
      if (op == KVS_OP_DECODE_ATTN && g <= kTmMaxGroup) {
        const size_t tm = tm_workspace_bytes(p, n_seq, max_blocks, g);
        b = small_call(n_seq, p->desc.num_kv_heads, max_blocks, g) ? std::max(b, tm) : tm;
      }
      break;
    }
    case KVS_OP_SELECT: {
      // one float score per row; bound rows by n_seq * max_blocks (callers pass
      // n_agents and max_rows_per_agent here)
      b = static_cast<size_t>(n_seq) * max_blocks * sizeof(float) + 256;
      break;
    }
    case KVS_OP_MIRROR:
      b = mirror_workspace_bytes(n_seq, max_blocks);
      break;
    case KVS_OP_BLOCKS:
      b = blocks_workspace_bytes(p->desc.capacity_blocks, n_seq);
      break;
    default:
      return fail(KVS_ERR_INVALID_ARG, "workspace_size: unknown op");
  }
  *bytes = b;
  return KVS_OK;
}

kvs_status kvs_pool_set_test_flags(kvs_pool* p, uint32_t flags) {
  if (!p) return fail(KVS_ERR_INVALID_ARG, "pool_set_test_flags: null pool");
  p->test_flags = flags;
  return KVS_OK;
}

kvs_status kvs_pool_check(kvs_pool* p, cudaStream_t s, uint32_t* flags) {
  if (!p || !flags) return fail(KVS_ERR_INVALID_ARG, "pool_check: null argument");
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, p->status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(p->status, 0, 4, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return fail(KVS_ERR_CUDA, std::string("pool_check: ") + cudaGetErrorString(cudaGetLastError()));
  *flags = h;
  if (h) return fail(KVS_ERR_DEVICE_BOUNDS, "pool_check: the device recorded errors");
  return KVS_OK;
}

kvs_status kvs_pool_stats(const kvs_pool* p, const int32_t* refcount_dev, const int32_t* n_phys_dev,
                          cudaStream_t s, kvs_stats* out) {
  if (!p || !refcount_dev || !n_phys_dev || !out) return fail(KVS_ERR_INVALID_ARG, "pool_stats: null argument");
  int32_t n = 0;
  if (cudaMemcpyAsync(&n, n_phys_dev, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "pool_stats: copy failed");
  if (n < 0 || n > p->desc.capacity_blocks) return fail(KVS_ERR_CAPACITY, "pool_stats: n_phys out of range");
  std::vector<int32_t> rc(static_cast<size_t>(n));
  if (n > 0 && (cudaMemcpyAsync(rc.data(), refcount_dev, n * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess))
    return fail(KVS_ERR_CUDA, "pool_stats: copy failed");
  kvs_stats st{};
  st.unique_blocks = n;
  for (int32_t r : rc) {
    st.total_refs += r;
    if (r > 1) st.shared_blocks++;
  }
  const int64_t per_block = p->desc.dtype == KVS_DTYPE_BF16
                                ? 2ll * p->desc.num_kv_heads * p->desc.block_tokens * p->desc.head_dim * 2
                                : 2ll * p->desc.num_kv_heads * p->desc.block_tokens * (p->desc.head_dim / 2 + p->desc.head_dim / 16);
  st.pool_bytes = st.unique_blocks * per_block * p->desc.num_layers;
  st.dense_bytes = st.total_refs * per_block * p->desc.num_layers;
  *out = st;
  return KVS_OK;
}

}  // extern "C"
