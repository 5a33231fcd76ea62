// Block lifetime on the device: copy-on-write and release of shared physical
// blocks (INMS walkthrough §2.2: shared blocks are read-only; a sequence about
// to write into a block others also reference gets a private copy and the old
// block's reference count drops, else it writes in place; §3.3: destroying a
// sequence decrements its blocks' counts and reclaims what becomes unused;
// §5.3: every path must bring the counts back to zero).
//
// Unused blocks sit on a free stack (free_ids[0 .. n_free), top at
// n_free - 1).  Pushes go in descending block id order, so the smallest id
// ends on top and is taken first.  Every step is deterministic: a write batch
// has the result of applying the writes one after the other; a release has
// the result of decrementing first and then pushing the blocks that reached
// zero.
//
// Copy-on-write of a batch, all on the device:
//  bw_dups     a write whose (sequence, block) appeared earlier in the batch
//              targets that earlier write's private block: it writes in place;
//  bw_rank     among the other writes, the k-th one (list order) to the same
//              physical block X sees a count of refcount[X] - k, so it copies
//              exactly when k < refcount[X] - 1;
//  bw_alloc    one CTA: copies take blocks off the top of the stack in list
//              order;
//  bw_apply    redirect the table entries, count 1 on the copies, one less on
//              the old blocks;
//  bw_copy     every layer's K and V (and Q4 scale/bias) of the old block into
//              the copy, 16-byte vectors.
#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr int kBlkChunk = 2048;   // blocks per CTA in the free-stack compaction
constexpr int kBlkTile = 256;     // writes staged in shared memory at a time

static size_t blk_align(size_t x) { return (x + 255) & ~size_t(255); }

struct BlkLayout {
  int n_chunks;
  size_t off_flags, off_counts, off_wold, off_wdup, off_wcow, off_wnew, off_seqf, total;
};

static BlkLayout blk_layout(int capacity, int n_items) {
  BlkLayout L{};
  L.n_chunks = (capacity + kBlkChunk - 1) / kBlkChunk;
  const size_t n = n_items > 0 ? (size_t)n_items : 1;
  size_t o = 0;
  L.off_flags = o; o = blk_align(o + (size_t)capacity);
  L.off_counts = o; o = blk_align(o + (size_t)(L.n_chunks + 2) * sizeof(int32_t));
  L.off_wold = o; o = blk_align(o + n * sizeof(int32_t));
  L.off_wdup = o; o = blk_align(o + n * sizeof(int32_t));
  L.off_wcow = o; o = blk_align(o + n * sizeof(int32_t));
  L.off_wnew = o; o = blk_align(o + n * sizeof(int32_t));
  L.off_seqf = o; o = blk_align(o + n);
  L.total = o;
  return L;
}

size_t blocks_workspace_bytes(int capacity, int n_items) { return blk_layout(capacity, n_items).total + 256; }

// ------------------------------------------------ free-stack compaction ---
struct PushParams {
  const uint8_t* flags;   // [capacity] 1 = push this block
  int32_t* counts;        // [n_chunks + 2]: per-chunk counts -> offsets; [n_chunks] total; [n_chunks + 1] old n_free
  int32_t* free_ids;
  int32_t* n_free;
  uint32_t* status;
  int capacity, n_chunks;
};

// chunk c covers the reversed indices [c * kBlkChunk, ...): block id
// capacity - 1 - i, so the scan order is descending block id
__global__ void __launch_bounds__(256) blk_count(const __grid_constant__ PushParams q) {
  __shared__ int warp_sums[32];
  for (int c = blockIdx.x; c < q.n_chunks; c += gridDim.x) {
    int cnt = 0;
    for (int i = c * kBlkChunk + threadIdx.x; i < min(q.capacity, (c + 1) * kBlkChunk); i += blockDim.x)
      cnt += q.flags[q.capacity - 1 - i];
    int total;
    block_exclusive_scan(cnt, warp_sums, total);
    if (threadIdx.x == 0) q.counts[c] = total;
  }
}

__global__ void __launch_bounds__(1024) blk_scan(const __grid_constant__ PushParams q) {
  __shared__ int warp_sums[32];
  int carry = 0;
  for (int base = 0; base < q.n_chunks; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int x = i < q.n_chunks ? q.counts[i] : 0;
    int total;
    const int ex = block_exclusive_scan(x, warp_sums, total);
    if (i < q.n_chunks) q.counts[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) {
    const int old = *q.n_free;
    q.counts[q.n_chunks] = carry;
    q.counts[q.n_chunks + 1] = old;
    *q.n_free = min(old + carry, q.capacity);
  }
}

__global__ void __launch_bounds__(256) blk_push(const __grid_constant__ PushParams q) {
  __shared__ int warp_sums[32];
  const int base0 = q.counts[q.n_chunks + 1];
  for (int c = blockIdx.x; c < q.n_chunks; c += gridDim.x) {
    int carry = base0 + q.counts[c];
    for (int i0 = c * kBlkChunk; i0 < min(q.capacity, (c + 1) * kBlkChunk); i0 += blockDim.x) {
      const int i = i0 + threadIdx.x;
      const int f = i < min(q.capacity, (c + 1) * kBlkChunk) ? q.flags[q.capacity - 1 - i] : 0;
      int total;
      const int ex = block_exclusive_scan(f, warp_sums, total);
      if (f) {
        // a consistent stack never overflows; an inconsistent one (a block
        // pushed while already free) is reported instead of written past
        if (carry + ex < q.capacity) q.free_ids[carry + ex] = q.capacity - 1 - i;
        else set_err(q.status, KVS_DEVERR_CAPACITY);
      }
      carry += total;
    }
  }
}

static kvs_status push_flagged(const kvs_pool* pool, const uint8_t* flags, int32_t* counts, int32_t* free_ids,
                               int32_t* n_free, int n_chunks, cudaStream_t st) {
  PushParams q{flags, counts, free_ids, n_free, pool->status, pool->desc.capacity_blocks, n_chunks};
  const int grid = std::max(1, std::min(n_chunks, pool->num_sms * 8));
  blk_count<<<grid, 256, 0, st>>>(q);
  blk_scan<<<1, 1024, 0, st>>>(q);
  blk_push<<<grid, 256, 0, st>>>(q);
  count_launch(3);
  return check_launch("block free stack");
}

// ------------------------------------------------------------ init free ---
__global__ void blk_zero_flags(const int32_t* __restrict__ refcount, uint8_t* flags, int32_t* n_free, int capacity) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p == 0) *n_free = 0;
  if (p < capacity) flags[p] = refcount[p] == 0 ? 1 : 0;
}

// --------------------------------------------------------- copy on write ---
struct WriteParams {
  int32_t* table;
  const int32_t* wseq;
  const int32_t* wblk;
  int32_t* refcount;
  int32_t* free_ids;
  int32_t* n_free;
  int32_t* w_old;   // physical block targeted (-1: invalid write)
  int32_t* w_dup;   // 1: the same (sequence, block) was written earlier in the batch
  int32_t* w_cow;   // 1: this write copies
  int32_t* w_new;   // the copy's block (-1: none)
  void** slabs;
  const long long* sbytes;
  uint32_t* status;
  int n_seq, max_blocks, n_writes, capacity, n_slabs;
};

__global__ void __launch_bounds__(kBlkTile) bw_dups(const __grid_constant__ WriteParams p) {
  __shared__ int ta[kBlkTile], tb[kBlkTile];
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  int a = -1, b = -1, old = -1;
  if (w < p.n_writes) {
    a = p.wseq[w];
    b = p.wblk[w];
    if (a < 0 || a >= p.n_seq || b < 0 || b >= p.max_blocks) {
      set_err(p.status, KVS_DEVERR_JOB);
      a = b = -1;
    } else {
      old = p.table[(size_t)a * p.max_blocks + b];
      if (old < 0 || old >= p.capacity) {
        set_err(p.status, KVS_DEVERR_BLOCK_ID);
        old = -1;
      }
    }
  }
  int dup = 0;
  const int last = min(p.n_writes, (int)(blockIdx.x + 1) * (int)blockDim.x);
  for (int t0 = 0; t0 < last; t0 += kBlkTile) {
    __syncthreads();
    const int i = t0 + threadIdx.x;
    ta[threadIdx.x] = i < p.n_writes ? p.wseq[i] : -2;
    tb[threadIdx.x] = i < p.n_writes ? p.wblk[i] : -2;
    __syncthreads();
    if (a >= 0)
      for (int j = 0; j < kBlkTile && t0 + j < w; ++j) dup |= (ta[j] == a && tb[j] == b);
  }
  if (w < p.n_writes) {
    p.w_old[w] = old;
    p.w_dup[w] = dup;
  }
}

__global__ void __launch_bounds__(kBlkTile) bw_rank(const __grid_constant__ WriteParams p) {
  __shared__ int told[kBlkTile];
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  const int old = w < p.n_writes ? p.w_old[w] : -1;
  const int dup = w < p.n_writes ? p.w_dup[w] : 1;
  int rank = 0;
  const int last = min(p.n_writes, (int)(blockIdx.x + 1) * (int)blockDim.x);
  for (int t0 = 0; t0 < last; t0 += kBlkTile) {
    __syncthreads();
    const int i = t0 + threadIdx.x;
    told[threadIdx.x] = (i < p.n_writes && !p.w_dup[i]) ? p.w_old[i] : -1;
    __syncthreads();
    if (old >= 0 && !dup)
      for (int j = 0; j < kBlkTile && t0 + j < w; ++j) rank += told[j] == old;
  }
  if (w < p.n_writes) p.w_cow[w] = (old >= 0 && !dup && rank < p.refcount[old] - 1) ? 1 : 0;
}

__global__ void __launch_bounds__(1024) bw_alloc(const __grid_constant__ WriteParams p) {
  __shared__ int warp_sums[32];
  const int avail = *p.n_free;
  int carry = 0;
  for (int base = 0; base < p.n_writes; base += blockDim.x) {
    const int w = base + threadIdx.x;
    const int c = w < p.n_writes ? p.w_cow[w] : 0;
    int total;
    const int k = carry + block_exclusive_scan(c, warp_sums, total);
    if (w < p.n_writes) {
      int nw = -1;
      if (c) {
        if (k < avail) nw = p.free_ids[avail - 1 - k];
        else set_err(p.status, KVS_DEVERR_CAPACITY);   // no free block: this write keeps the shared block
      }
      p.w_new[w] = nw;
    }
    carry += total;
  }
  if (threadIdx.x == 0) *p.n_free = avail - min(carry, avail);
}

__global__ void bw_apply(const __grid_constant__ WriteParams p) {
  const int w = blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= p.n_writes) return;
  const int nw = p.w_new[w];
  if (nw < 0) return;
  const int a = p.wseq[w], b = p.wblk[w];
  p.table[(size_t)a * p.max_blocks + b] = nw;
  p.refcount[nw] = 1;
  atomicSub(p.refcount + p.w_old[w], 1);
}

// blockIdx.x: write; blockIdx.y: slab
__global__ void __launch_bounds__(256) bw_copy(const __grid_constant__ WriteParams p) {
  const int w = blockIdx.x;
  const int nw = p.w_new[w];
  if (nw < 0) return;
  const int old = p.w_old[w];
  const long long nb = p.sbytes[blockIdx.y];
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.slabs[blockIdx.y]) + (long long)old * nb);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.slabs[blockIdx.y]) + (long long)nw * nb);
  for (long long i = threadIdx.x; i < nb / 16; i += blockDim.x) dst[i] = __ldg(src + i);
}

// --------------------------------------------------------------- release ---
struct RelParams {
  int32_t* table;
  int32_t* seq_len;
  const int32_t* rel;
  int32_t* refcount;
  uint8_t* seqf;    // [n_seq] 1 = released by this call
  uint8_t* freed;   // [capacity] 1 = reached zero in this call
  uint32_t* status;
  int n_seq, max_blocks, n_release, capacity, block_tokens;
};

__global__ void rel_mark(const __grid_constant__ RelParams p) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.n_release) return;
  const int a = p.rel[i];
  if (a < 0 || a >= p.n_seq) {
    set_err(p.status, KVS_DEVERR_JOB);
    return;
  }
  p.seqf[a] = 1;   // a sequence listed twice is released once
}

__global__ void __launch_bounds__(256) rel_dec(const __grid_constant__ RelParams p) {
  for (int a = blockIdx.x; a < p.n_seq; a += gridDim.x) {
    if (!p.seqf[a]) continue;
    int L = p.seq_len[a];
    if (L < 0 || L > p.max_blocks * p.block_tokens) {
      if (threadIdx.x == 0) set_err(p.status, KVS_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : p.max_blocks * p.block_tokens;
    }
    const int nb = (L + p.block_tokens - 1) / p.block_tokens;
    int32_t* row = p.table + (size_t)a * p.max_blocks;
    for (int b = threadIdx.x; b < p.max_blocks; b += blockDim.x) {
      if (b < nb) {
        const int ph = row[b];
        if (ph < 0 || ph >= p.capacity) {
          set_err(p.status, KVS_DEVERR_BLOCK_ID);
        } else {
          const int before = atomicSub(p.refcount + ph, 1);
          if (before == 1) p.freed[ph] = 1;
          if (before <= 0) set_err(p.status, KVS_DEVERR_REFCOUNT);
        }
      }
      row[b] = -1;
    }
    if (threadIdx.x == 0) p.seq_len[a] = 0;
  }
}

// ---------------------------------------------------------- export/import ---
// blockIdx.x: listed block i; blockIdx.y: slab.  to_pack: slab -> record.
__global__ void __launch_bounds__(256) pool_io(void** slabs, const long long* sbytes, const long long* soffs,
                                               const int32_t* blocks, int n_blocks, long long record, uint8_t* packed,
                                               int capacity, bool to_pack, uint32_t* status) {
  const int i = blockIdx.x;
  const int ph = blocks[i];
  if (ph < 0 || ph >= capacity) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_err(status, KVS_DEVERR_BLOCK_ID);
    return;
  }
  const long long nb = sbytes[blockIdx.y];
  uint4* slab = reinterpret_cast<uint4*>(static_cast<uint8_t*>(slabs[blockIdx.y]) + (long long)ph * nb);
  uint4* rec = reinterpret_cast<uint4*>(packed + (long long)i * record + soffs[blockIdx.y]);
  if (to_pack)
    for (long long v = threadIdx.x; v < nb / 16; v += blockDim.x) rec[v] = __ldg(slab + v);
  else
    for (long long v = threadIdx.x; v < nb / 16; v += blockDim.x) slab[v] = __ldg(rec + v);
}

}  // namespace kvs

using namespace kvs;

static kvs_status pool_io_call(kvs_pool* pool, const int32_t* blocks, int32_t n_blocks, void* buf, size_t bytes,
                               bool to_pack, cudaStream_t stream, const char* what) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": null pool");
  if (n_blocks < 0) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": bad n_blocks");
  if (n_blocks == 0) return KVS_OK;
  if (!blocks || !buf) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": null pointer");
  if (!aligned16(buf)) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": buffer must be 16-byte aligned");
  if (bytes < (size_t)n_blocks * (size_t)pool->blk_record) return fail(KVS_ERR_CAPACITY, std::string(what) + ": buffer too small");
  if (pool->n_blk_slabs > 65535) return fail(KVS_ERR_UNSUPPORTED, std::string(what) + ": too many layers");
  pool_io<<<dim3(n_blocks, pool->n_blk_slabs), 256, 0, stream>>>(pool->blk_slabs, pool->blk_bytes, pool->blk_offs,
                                                                 blocks, n_blocks, pool->blk_record,
                                                                 static_cast<uint8_t*>(buf), pool->desc.capacity_blocks,
                                                                 to_pack, pool->status);
  count_launch();
  return check_launch(what);
}

extern "C" kvs_status kvs_pool_block_bytes(const kvs_pool* pool, size_t* bytes) {
  if (!pool || !bytes) return fail(KVS_ERR_INVALID_ARG, "pool_block_bytes: null argument");
  *bytes = (size_t)pool->blk_record;
  return KVS_OK;
}

extern "C" kvs_status kvs_pool_export(kvs_pool* pool, const int32_t* blocks_dev, int32_t n_blocks, void* dst_dev,
                                      size_t dst_bytes, cudaStream_t stream) {
  return pool_io_call(pool, blocks_dev, n_blocks, dst_dev, dst_bytes, true, stream, "pool_export");
}

extern "C" kvs_status kvs_pool_import(kvs_pool* pool, const int32_t* blocks_dev, int32_t n_blocks, const void* src_dev,
                                      size_t src_bytes, cudaStream_t stream) {
  return pool_io_call(pool, blocks_dev, n_blocks, const_cast<void*>(src_dev), src_bytes, false, stream, "pool_import");
}

static kvs_status blk_common(const kvs_pool* pool, const int32_t* refcount, const int32_t* free_ids,
                             const int32_t* n_free, const void* ws, const char* what) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": null pool");
  if (!refcount || !free_ids || !n_free || !ws) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": null pointer");
  if (!aligned16(ws)) return fail(KVS_ERR_INVALID_ARG, std::string(what) + ": ws must be 16-byte aligned");
  return KVS_OK;
}

extern "C" kvs_status kvs_blocks_init_free(kvs_pool* pool, const int32_t* refcount_dev, int32_t* free_ids_dev,
                                           int32_t* n_free_dev, void* ws, size_t ws_bytes, cudaStream_t stream) {
  kvs_status st = blk_common(pool, refcount_dev, free_ids_dev, n_free_dev, ws, "blocks_init_free");
  if (st != KVS_OK) return st;
  const int cap = pool->desc.capacity_blocks;
  const BlkLayout L = blk_layout(cap, 1);
  if (ws_bytes < L.total) return fail(KVS_ERR_CAPACITY, "blocks_init_free: workspace too small");
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint8_t* flags = w + L.off_flags;
  blk_zero_flags<<<(cap + 255) / 256, 256, 0, stream>>>(refcount_dev, flags, n_free_dev, cap);
  count_launch();
  if ((st = check_launch("blocks_init_free")) != KVS_OK) return st;
  return push_flagged(pool, flags, reinterpret_cast<int32_t*>(w + L.off_counts), free_ids_dev, n_free_dev,
                      L.n_chunks, stream);
}

extern "C" kvs_status kvs_block_write(kvs_pool* pool, int32_t* block_table_dev, int32_t max_blocks, int32_t n_seq,
                                      const int32_t* write_seq_dev, const int32_t* write_block_dev,
                                      int32_t n_writes, int32_t* refcount_dev, int32_t* free_ids_dev,
                                      int32_t* n_free_dev, void* ws, size_t ws_bytes, cudaStream_t stream) {
  kvs_status st = blk_common(pool, refcount_dev, free_ids_dev, n_free_dev, ws, "block_write");
  if (st != KVS_OK) return st;
  if (n_writes < 0 || n_seq < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "block_write: bad sizes");
  if (n_writes == 0) return KVS_OK;
  if (!block_table_dev || !write_seq_dev || !write_block_dev) return fail(KVS_ERR_INVALID_ARG, "block_write: null pointer");
  const BlkLayout L = blk_layout(pool->desc.capacity_blocks, n_writes);
  if (ws_bytes < L.total) return fail(KVS_ERR_CAPACITY, "block_write: workspace too small");
  if (pool->n_blk_slabs > 65535) return fail(KVS_ERR_UNSUPPORTED, "block_write: too many layers");
  uint8_t* w = static_cast<uint8_t*>(ws);
  WriteParams p{};
  p.table = block_table_dev;
  p.wseq = write_seq_dev;
  p.wblk = write_block_dev;
  p.refcount = refcount_dev;
  p.free_ids = free_ids_dev;
  p.n_free = n_free_dev;
  p.w_old = reinterpret_cast<int32_t*>(w + L.off_wold);
  p.w_dup = reinterpret_cast<int32_t*>(w + L.off_wdup);
  p.w_cow = reinterpret_cast<int32_t*>(w + L.off_wcow);
  p.w_new = reinterpret_cast<int32_t*>(w + L.off_wnew);
  p.slabs = pool->blk_slabs;
  p.sbytes = pool->blk_bytes;
  p.status = pool->status;
  p.n_seq = n_seq;
  p.max_blocks = max_blocks;
  p.n_writes = n_writes;
  p.capacity = pool->desc.capacity_blocks;
  p.n_slabs = pool->n_blk_slabs;
  const int g = (n_writes + kBlkTile - 1) / kBlkTile;
  bw_dups<<<g, kBlkTile, 0, stream>>>(p);
  bw_rank<<<g, kBlkTile, 0, stream>>>(p);
  bw_alloc<<<1, 1024, 0, stream>>>(p);
  bw_apply<<<g, kBlkTile, 0, stream>>>(p);
  bw_copy<<<dim3(n_writes, pool->n_blk_slabs), 256, 0, stream>>>(p);
  count_launch(5);
  return check_launch("block_write");
}

extern "C" kvs_status kvs_seq_release(kvs_pool* pool, int32_t* block_table_dev, int32_t max_blocks,
                                      int32_t* seq_len_dev, int32_t n_seq, const int32_t* release_seq_dev,
                                      int32_t n_release, int32_t* refcount_dev, int32_t* free_ids_dev,
                                      int32_t* n_free_dev, void* ws, size_t ws_bytes, cudaStream_t stream) {
  kvs_status st = blk_common(pool, refcount_dev, free_ids_dev, n_free_dev, ws, "seq_release");
  if (st != KVS_OK) return st;
  if (n_release < 0 || n_seq < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "seq_release: bad sizes");
  if (n_release == 0 || n_seq == 0) return KVS_OK;
  if (!block_table_dev || !seq_len_dev || !release_seq_dev) return fail(KVS_ERR_INVALID_ARG, "seq_release: null pointer");
  const int cap = pool->desc.capacity_blocks;
  const BlkLayout L = blk_layout(cap, n_seq);
  if (ws_bytes < L.total) return fail(KVS_ERR_CAPACITY, "seq_release: workspace too small");
  uint8_t* w = static_cast<uint8_t*>(ws);
  RelParams p{};
  p.table = block_table_dev;
  p.seq_len = seq_len_dev;
  p.rel = release_seq_dev;
  p.refcount = refcount_dev;
  p.seqf = w + L.off_seqf;
  p.freed = w + L.off_flags;
  p.status = pool->status;
  p.n_seq = n_seq;
  p.max_blocks = max_blocks;
  p.n_release = n_release;
  p.capacity = cap;
  p.block_tokens = pool->desc.block_tokens;
  if (cudaMemsetAsync(p.seqf, 0, n_seq, stream) != cudaSuccess || cudaMemsetAsync(p.freed, 0, cap, stream) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "seq_release: memset failed");
  rel_mark<<<(n_release + 255) / 256, 256, 0, stream>>>(p);
  rel_dec<<<std::min(n_seq, pool->num_sms * 8), 256, 0, stream>>>(p);
  count_launch(2);
  if ((st = check_launch("seq_release")) != KVS_OK) return st;
  return push_flagged(pool, p.freed, reinterpret_cast<int32_t*>(w + L.off_counts), free_ids_dev, n_free_dev,
                      L.n_chunks, stream);
}
