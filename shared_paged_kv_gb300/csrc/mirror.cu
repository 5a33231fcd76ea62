// Mirror construction from refreshed critical positions (TokenDance summary,
// section 2: only the critical positions of each request's cached K/V are
// refreshed; section 3, Fig. 7: one master cache, the other caches of the
// family kept as block-sparse K/V differences from it; Fig. 8: the diff is
// applied before the RoPE positions are restored, so it lives in the
// master's frame).
//
// Steps, all on the device:
//  1. mir_agent   one CTA per agent: clear the agent's dirty flags, validate
//                 the refreshed positions and flag the logical blocks holding
//                 one; then count the agent's dirty blocks;
//  2. mir_apply   one CTA per agent: its first diff id (the dirty blocks of
//                 the agents before it: diff ids are consecutive in agent
//                 order, then block order), the diff table, the list of dirty slots,
//                 each dirty block's refreshed rows (the first one's index
//                 and a 16-bit mask: positions are sorted, so the k-th set
//                 bit is refreshed row first + k) and, for rotation calls,
//                 its shift (the last covering segment entry);
//  3. mir_write   one warp per (dirty block, kv head): 16 rows, a refreshed
//                 row becoming bf16(R(-delta) k_new - K_master) and
//                 bf16(v_new - V_master), every other row zero.  Lane (row,
//                 v) holds head dims [8v, 8v+8) and [d/2+8v, d/2+8v+8), so the
//                 rotate-half partners sit in the same lane.
// The three kernels are programmatic dependent launches: each waits for the
// one before it at its first statement and lets the next be scheduled.
#include "common.cuh"
#include "internal.h"

namespace kvs {

constexpr int kMirB = 16;         // block tokens this path supports
constexpr int kMirUnroll = 4;     // refreshed positions a thread takes at once

static size_t mir_align(size_t x) { return (x + 255) & ~size_t(255); }

struct MirLayout {
  size_t off_flags, off_rows, off_counts, off_list, off_delta, total;
};

static MirLayout mir_layout(int n_seq, int max_blocks) {
  const size_t slots = (size_t)n_seq * max_blocks;
  MirLayout L{};
  size_t o = 0;
  L.off_flags = o; o = mir_align(o + slots);
  L.off_rows = o; o = mir_align(o + slots * sizeof(int2));
  L.off_counts = o; o = mir_align(o + (size_t)(n_seq + 1) * sizeof(int32_t));
  L.off_list = o; o = mir_align(o + slots * sizeof(int32_t));
  L.off_delta = o; o = mir_align(o + slots * sizeof(int32_t));
  L.total = o;
  return L;
}

size_t mirror_workspace_bytes(int n_seq, int max_blocks) { return mir_layout(n_seq, max_blocks).total + 256; }

struct MirParams {
  const int32_t* table;
  const int32_t* seq_len;
  const int32_t* idx;
  const int64_t* idx_off;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* rope_off;
  const int4* rope_segs;
  const uint16_t* kslab;
  const uint16_t* vslab;
  uint16_t* dk;
  uint16_t* dv;
  int32_t* diff_table;
  int32_t* n_diff;
  uint8_t* flags;     // [n_seq][max_blocks] 1 = dirty
  int2* rows;         // [n_diff] {first refreshed row, mask of refreshed tokens} per diff id
  int32_t* counts;    // [n_seq] dirty blocks per agent
  int32_t* list;      // [n_diff] dirty slot (a * max_blocks + b) of each diff id
  int32_t* dlt;       // [n_diff] RoPE shift of each dirty block (rotation calls)
  uint32_t* status;
  int n_seq, max_blocks, hkv, capacity, diff_capacity;
  RopeSplit rs;
};

// 1. positions -> dirty flags and row map; dirty blocks per agent
__global__ void __launch_bounds__(256) mir_agent(const __grid_constant__ MirParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  for (int a = blockIdx.x; a < p.n_seq; a += gridDim.x) {
    const long long r0 = p.idx_off[a], r1 = p.idx_off[a + 1];
    int L = p.seq_len[a];
    if (L < 0 || L > p.max_blocks * kMirB) {
      if (threadIdx.x == 0) set_err(p.status, KVS_DEVERR_SEQ_LEN);
      L = L < 0 ? 0 : p.max_blocks * kMirB;
    }
    uint8_t* fl = p.flags + (size_t)a * p.max_blocks;
    for (int b = threadIdx.x; b < p.max_blocks; b += blockDim.x) fl[b] = 0;
    __syncthreads();
    if (r0 < 0 || r1 < r0) {
      if (threadIdx.x == 0) set_err(p.status, KVS_DEVERR_JOB);
    } else {
      // kMirUnroll positions per thread at a time, their loads in flight together
      for (long long base = r0 + threadIdx.x; base < r1; base += (long long)kMirUnroll * blockDim.x) {
        int t[kMirUnroll], tp[kMirUnroll];
#pragma unroll
        for (int k = 0; k < kMirUnroll; ++k) {
          const long long r = base + (long long)k * blockDim.x;
          t[k] = r < r1 ? p.idx[r] : 0;
          tp[k] = (r < r1 && r > r0) ? p.idx[r - 1] : -1;
        }
#pragma unroll
        for (int k = 0; k < kMirUnroll; ++k) {
          if (base + (long long)k * blockDim.x >= r1) continue;
          if (t[k] < 0 || t[k] >= L || tp[k] >= t[k]) {
            set_err(p.status, KVS_DEVERR_JOB);
            continue;
          }
          fl[t[k] / kMirB] = 1;   // equal-value writes
        }
      }
    }
    __syncthreads();
    int cnt = 0;
    for (int b = threadIdx.x; b < p.max_blocks; b += blockDim.x) cnt += fl[b];
    int total;
    block_exclusive_scan(cnt, warp_sums, total);
    if (threadIdx.x == 0) p.counts[a] = total;
  }
}

// 2. diff table, dirty list and shifts, one CTA per agent
constexpr int kMirSegChunk = 256;   // segment entries staged in shared memory at a time

__global__ void __launch_bounds__(256) mir_apply(const __grid_constant__ MirParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  __shared__ int4 segs[kMirSegChunk];
  // the total number of dirty blocks (CTA 0)
  if (blockIdx.x == 0) {
    int x = 0;
    for (int i = threadIdx.x; i < p.n_seq; i += blockDim.x) x += p.counts[i];
    int total;
    block_exclusive_scan(x, warp_sums, total);
    if (threadIdx.x == 0) {
      *p.n_diff = total;
      if (total > p.diff_capacity) set_err(p.status, KVS_DEVERR_DIFF_ID);
    }
  }
  // first diff id of agent a: the dirty blocks of agents 0 .. a-1, summed
  // from the last agent this CTA handled
  int pre = 0, pre_a = 0;
  for (int a = blockIdx.x; a < p.n_seq; a += gridDim.x) {
    {
      int x = 0;
      for (int i = pre_a + threadIdx.x; i < a; i += blockDim.x) x += p.counts[i];
      int total;
      __syncthreads();   // warp_sums is reused
      block_exclusive_scan(x, warp_sums, total);
      pre += total;
      pre_a = a;
    }
    const uint8_t* fl = p.flags + (size_t)a * p.max_blocks;
    const int first = pre;
    int carry = first;
    for (int base = 0; base < p.max_blocks; base += blockDim.x) {
      const int b = base + threadIdx.x;
      const int f = b < p.max_blocks ? fl[b] : 0;
      int total;
      const int ex = block_exclusive_scan(f, warp_sums, total);
      if (b < p.max_blocks) {
        const size_t slot = (size_t)a * p.max_blocks + b;
        const int id = carry + ex;
        p.diff_table[slot] = f ? id : -1;
        if (f && id < p.diff_capacity) {
          p.list[id] = (int)slot;
          p.rows[id] = make_int2(-1, 0);
          if (!p.rope_off) p.dlt[id] = 0;
        }
      }
      carry += total;
    }
    // each dirty block's refreshed rows: the thread holding the first valid
    // position of a block records it, every valid position sets its bit (the
    // validity test is mir_agent's, so an invalid position counts nowhere)
    __syncthreads();   // the diff table entries above are read by other threads
    {
      const long long r0 = p.idx_off[a], r1 = p.idx_off[a + 1];
      int L = p.seq_len[a];
      L = L < 0 ? 0 : min(L, p.max_blocks * kMirB);
      if (r0 >= 0 && r1 >= r0) {
        // kMirUnroll positions per thread at a time: their position loads,
        // then their diff-table loads, each group in flight together
        for (long long base = r0 + threadIdx.x; base < r1; base += (long long)kMirUnroll * blockDim.x) {
          int t[kMirUnroll], tp[kMirUnroll], id[kMirUnroll];
#pragma unroll
          for (int k = 0; k < kMirUnroll; ++k) {
            const long long r = base + (long long)k * blockDim.x;
            t[k] = r < r1 ? p.idx[r] : -1;
            tp[k] = (r < r1 && r > r0) ? p.idx[r - 1] : -1;
          }
#pragma unroll
          for (int k = 0; k < kMirUnroll; ++k) {
            const bool ok = t[k] >= 0 && t[k] < L && tp[k] < t[k];
            id[k] = ok ? p.diff_table[(size_t)a * p.max_blocks + t[k] / kMirB] : -1;
          }
#pragma unroll
          for (int k = 0; k < kMirUnroll; ++k) {
            if (id[k] < 0 || id[k] >= p.diff_capacity) continue;
            const long long r = base + (long long)k * blockDim.x;
            if (r == r0 || tp[k] / kMirB != t[k] / kMirB) p.rows[id[k]].x = (int)r;
            atomicOr(reinterpret_cast<unsigned int*>(&p.rows[id[k]].y), 1u << (t[k] % kMirB));
          }
        }
      }
    }
    if (!p.rope_off) continue;
    // shifts of this agent's dirty blocks: the last covering entry, the
    // segment list streamed through shared memory
    __syncthreads();   // the list entries above are read by other threads
    const int n_dirty = min(carry, p.diff_capacity) - min(first, p.diff_capacity);
    const int e0 = p.rope_off[a], e1 = p.rope_off[a + 1];
    for (int i0 = 0; i0 < n_dirty; i0 += blockDim.x) {
      const int i = i0 + threadIdx.x;
      const int b = i < n_dirty ? p.list[first + i] - a * p.max_blocks : -1;
      int dl = 0;
      for (int c0 = e0; c0 < e1; c0 += kMirSegChunk) {
        __syncthreads();
        for (int e = c0 + threadIdx.x; e < min(e1, c0 + kMirSegChunk); e += blockDim.x) segs[e - c0] = __ldg(p.rope_segs + e);
        __syncthreads();
        const int ne = min(e1, c0 + kMirSegChunk) - c0;
        if (b >= 0)
          for (int e = 0; e < ne; ++e)
            if (b >= segs[e].x && b - segs[e].x < segs[e].y) dl = segs[e].z;
      }
      if (b >= 0) {
        if (dl <= -(1 << 18) || dl >= (1 << 18)) {
          set_err(p.status, KVS_DEVERR_ROPE_RANGE);
          dl = 0;
        }
        p.dlt[first + i] = dl;
      }
    }
    __syncthreads();
  }
}

// 4. diff tiles of every dirty (block, kv head)
template <int D>
__global__ void __launch_bounds__(256) mir_write(const __grid_constant__ MirParams p) {
  pdl_enter();
  constexpr int VEC = 8;              // bf16 per 16-byte vector
  constexpr int NV = D / 2 / VEC;     // lanes per row
  constexpr int RPS = 32 / NV;        // rows per warp step
  __shared__ float rsc[4 * 64];       // RoPE frequency pieces (rotation calls)
  if (p.rope_off) {
    for (int i = threadIdx.x; i < 4 * 64; i += blockDim.x) rsc[i] = p.rs.c[i >> 6][i & 63];
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int v = lane % NV, rl = lane / NV;
  const int n_diff = min(*p.n_diff, p.diff_capacity);
  const long long units = (long long)n_diff * p.hkv;
  const int wpb = blockDim.x >> 5;
  for (long long u = (long long)blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += (long long)gridDim.x * wpb) {
    const int id = (int)(u / p.hkv), h = (int)(u - (long long)id * p.hkv);
    const int slot = p.list[id];
    const int phys = p.table[slot];
    const bool valid = phys >= 0 && phys < p.capacity;
    if (!valid && lane == 0 && h == 0) set_err(p.status, KVS_DEVERR_BLOCK_ID);
    // lane j < 16: the refreshed row of token j of the block (or -1): the
    // k-th refreshed token of the block is row first + k (positions are
    // sorted); a row outside the agent's list (only after invalid input,
    // which mir_agent flags) is treated as not refreshed
    const int2 ri = p.rows[id];
    const int a = slot / p.max_blocks;
    const long long ra = p.idx_off[a], rb = p.idx_off[a + 1];
    long long rr = -1;
    if (lane < kMirB && ri.x >= 0 && ((ri.y >> lane) & 1))
      rr = (long long)ri.x + __popc((unsigned)ri.y & ((1u << lane) - 1u));
    const int myrow = (rr >= ra && rr < rb && rr >= 0) ? (int)rr : -1;
    float cs[VEC], sn[VEC];
    const int delta = p.rope_off ? p.dlt[id] : 0;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      cs[e] = 1.f;
      sn[e] = 0.f;
    }
    if (delta != 0) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) rope_cos_sin(rsc, v * VEC + e, delta, cs[e], sn[e]);
    }
    const size_t tile = ((size_t)id * p.hkv + h) * kMirB;
    const size_t mtile = ((size_t)(valid ? phys : 0) * p.hkv + h) * kMirB;
#pragma unroll
    for (int st = 0; st < kMirB / RPS; ++st) {
      const int row = st * RPS + rl;
      const int r = __shfl_sync(0xffffffffu, myrow, row);
      uint4 dkl = make_uint4(0, 0, 0, 0), dkh = dkl, dvl = dkl, dvh = dkl;
      if (r >= 0 && valid) {
        const size_t mo = (mtile + row) * D + v * VEC;
        const size_t no = ((size_t)r * p.hkv + h) * D + v * VEC;
        const uint4 kml = __ldg(reinterpret_cast<const uint4*>(p.kslab + mo));
        const uint4 kmh = __ldg(reinterpret_cast<const uint4*>(p.kslab + mo + D / 2));
        const uint4 vml = __ldg(reinterpret_cast<const uint4*>(p.vslab + mo));
        const uint4 vmh = __ldg(reinterpret_cast<const uint4*>(p.vslab + mo + D / 2));
        const uint4 knl = __ldg(reinterpret_cast<const uint4*>(p.k_new + no));
        const uint4 knh = __ldg(reinterpret_cast<const uint4*>(p.k_new + no + D / 2));
        const uint4 vnl = __ldg(reinterpret_cast<const uint4*>(p.v_new + no));
        const uint4 vnh = __ldg(reinterpret_cast<const uint4*>(p.v_new + no + D / 2));
        const uint32_t a_kml[4] = {kml.x, kml.y, kml.z, kml.w}, a_kmh[4] = {kmh.x, kmh.y, kmh.z, kmh.w};
        const uint32_t a_vml[4] = {vml.x, vml.y, vml.z, vml.w}, a_vmh[4] = {vmh.x, vmh.y, vmh.z, vmh.w};
        const uint32_t a_knl[4] = {knl.x, knl.y, knl.z, knl.w}, a_knh[4] = {knh.x, knh.y, knh.z, knh.w};
        const uint32_t a_vnl[4] = {vnl.x, vnl.y, vnl.z, vnl.w}, a_vnh[4] = {vnh.x, vnh.y, vnh.z, vnh.w};
        uint32_t o_kl[4], o_kh[4], o_vl[4], o_vh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // R(-delta): lo' = lo cos + hi sin, hi' = hi cos - lo sin
          const float x0 = bf16_lo(a_knl[e]), x1 = bf16_hi(a_knl[e]);
          const float y0 = bf16_lo(a_knh[e]), y1 = bf16_hi(a_knh[e]);
          const float l0 = x0 * cs[2 * e] + y0 * sn[2 * e], l1 = x1 * cs[2 * e + 1] + y1 * sn[2 * e + 1];
          const float h0 = y0 * cs[2 * e] - x0 * sn[2 * e], h1 = y1 * cs[2 * e + 1] - x1 * sn[2 * e + 1];
          o_kl[e] = pack_bf16(l0 - bf16_lo(a_kml[e]), l1 - bf16_hi(a_kml[e]));
          o_kh[e] = pack_bf16(h0 - bf16_lo(a_kmh[e]), h1 - bf16_hi(a_kmh[e]));
          o_vl[e] = pack_bf16(bf16_lo(a_vnl[e]) - bf16_lo(a_vml[e]), bf16_hi(a_vnl[e]) - bf16_hi(a_vml[e]));
          o_vh[e] = pack_bf16(bf16_lo(a_vnh[e]) - bf16_lo(a_vmh[e]), bf16_hi(a_vnh[e]) - bf16_hi(a_vmh[e]));
        }
        dkl = make_uint4(o_kl[0], o_kl[1], o_kl[2], o_kl[3]);
        dkh = make_uint4(o_kh[0], o_kh[1], o_kh[2], o_kh[3]);
        dvl = make_uint4(o_vl[0], o_vl[1], o_vl[2], o_vl[3]);
        dvh = make_uint4(o_vh[0], o_vh[1], o_vh[2], o_vh[3]);
      }
      const size_t dofs = (tile + row) * D + v * VEC;
      *reinterpret_cast<uint4*>(p.dk + dofs) = dkl;
      *reinterpret_cast<uint4*>(p.dk + dofs + D / 2) = dkh;
      *reinterpret_cast<uint4*>(p.dv + dofs) = dvl;
      *reinterpret_cast<uint4*>(p.dv + dofs + D / 2) = dvh;
    }
  }
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_mirror_build(kvs_pool* pool, int32_t layer, const int32_t* block_table_dev,
                                       int32_t max_blocks, const int32_t* seq_len_dev, int32_t n_seq,
                                       const int32_t* idx_dev, const int64_t* idx_off_dev, const void* k_new_dev,
                                       const void* v_new_dev, const int32_t* rope_off_dev,
                                       const kvs_seg_rope* rope_segs_dev, float theta, int32_t* diff_table_dev,
                                       int32_t* n_diff_dev, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "mirror_build: null pool");
  const kvs_pool_desc& d = pool->desc;
  if (d.dtype != KVS_DTYPE_BF16) return fail(KVS_ERR_INVALID_ARG, "mirror_build: bf16 pools only");
  if (d.diff_capacity_blocks <= 0) return fail(KVS_ERR_INVALID_ARG, "mirror_build: the pool has no diff slabs");
  if (d.block_tokens != kMirB) return fail(KVS_ERR_UNSUPPORTED, "mirror_build: block_tokens must be 16");
  if (layer < 0 || layer >= d.num_layers) return fail(KVS_ERR_INVALID_ARG, "mirror_build: layer out of range");
  if (n_seq < 0 || max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "mirror_build: bad sizes");
  if ((rope_off_dev == nullptr) != (rope_segs_dev == nullptr))
    return fail(KVS_ERR_INVALID_ARG, "mirror_build: rope_off and rope_segs go together");
  if (rope_off_dev && !(theta > 0.f)) return fail(KVS_ERR_INVALID_ARG, "mirror_build: theta must be positive");
  if (!n_diff_dev) return fail(KVS_ERR_INVALID_ARG, "mirror_build: null n_diff");
  if (n_seq == 0) return cudaMemsetAsync(n_diff_dev, 0, 4, stream) == cudaSuccess ? KVS_OK : fail(KVS_ERR_CUDA, "mirror_build: memset failed");
  if (!block_table_dev || !seq_len_dev || !idx_dev || !idx_off_dev || !k_new_dev || !v_new_dev || !diff_table_dev ||
      !ws)
    return fail(KVS_ERR_INVALID_ARG, "mirror_build: null pointer");
  if (!aligned16(k_new_dev) || !aligned16(v_new_dev) || !aligned16(ws))
    return fail(KVS_ERR_INVALID_ARG, "mirror_build: k_new, v_new and ws must be 16-byte aligned");
  const MirLayout L = mir_layout(n_seq, max_blocks);
  if (ws_bytes < L.total) return fail(KVS_ERR_CAPACITY, "mirror_build: workspace too small");
  uint8_t* w = static_cast<uint8_t*>(ws);
  MirParams p{};
  p.table = block_table_dev;
  p.seq_len = seq_len_dev;
  p.idx = idx_dev;
  p.idx_off = idx_off_dev;
  p.k_new = static_cast<const uint16_t*>(k_new_dev);
  p.v_new = static_cast<const uint16_t*>(v_new_dev);
  p.rope_off = rope_off_dev;
  p.rope_segs = reinterpret_cast<const int4*>(rope_segs_dev);
  p.kslab = static_cast<const uint16_t*>(pool->k[layer]);
  p.vslab = static_cast<const uint16_t*>(pool->v[layer]);
  p.dk = static_cast<uint16_t*>(pool->dk[layer]);
  p.dv = static_cast<uint16_t*>(pool->dv[layer]);
  p.diff_table = diff_table_dev;
  p.n_diff = n_diff_dev;
  p.flags = w + L.off_flags;
  p.rows = reinterpret_cast<int2*>(w + L.off_rows);
  p.counts = reinterpret_cast<int32_t*>(w + L.off_counts);
  p.list = reinterpret_cast<int32_t*>(w + L.off_list);
  p.dlt = reinterpret_cast<int32_t*>(w + L.off_delta);
  p.status = pool->status;
  p.n_seq = n_seq;
  p.max_blocks = max_blocks;
  p.hkv = d.num_kv_heads;
  p.capacity = d.capacity_blocks;
  p.diff_capacity = d.diff_capacity_blocks;
  if (rope_off_dev) rope_split_host(theta, d.head_dim, p.rs.c);
  const int sms = pool->num_sms;
  const int agent_grid = std::min(n_seq, sms * 8);
  cudaError_t e = launch_pdl(mir_agent, dim3(agent_grid), dim3(256), stream, p);
  if (e == cudaSuccess) e = launch_pdl(mir_apply, dim3(agent_grid), dim3(256), stream, p);
  // the dirty count is only known on the device: a persistent grid of warps
  // walks the (dirty block, kv head) units
  if (e == cudaSuccess)
    e = d.head_dim == 128 ? launch_pdl(mir_write<128>, dim3(sms * 8), dim3(256), stream, p)
                          : launch_pdl(mir_write<64>, dim3(sms * 8), dim3(256), stream, p);
  if (e != cudaSuccess) return fail(KVS_ERR_CUDA, "mirror_build: launch failed");
  count_launch(3);
  return check_launch("mirror_build");
}
