// 4-bit group-quantised (Q4G64) KV: quantiser and decode attention that reads
// the codes directly (Q4 edge paper summary §2.1: 256-token blocks stored
// 4-bit, ratio 0.281 => group 64 with fp16 scale and bias; §2.2: attention on
// the Q4 tensors without a dequantise-to-FP16 pass).
//
// Attention design (GB300): the codes are the *A* operand of mma.sync
// m16n8k16 with tokens (QK^T) or head dims (PV) as the 16-row M dimension and
// the <= 8 query heads of a KV head as the 8-column N dimension, so a GQA
// group of 4 fills half of every MMA instead of a quarter.  Codes are turned
// into fp16 in registers as exact subnormals (a nibble masked in place is
// c * 2^-24 in the low position, c * 2^-20 in the high one; one LOP3 per
// pair), and the affine dequantisation is applied around the MMAs:
//   q.k_hat   = sum_groups  s_g * (q_g . c_g) + b_g * sum(q_g)
//   p.v_hat   = sum_t (p_t s_g[t]) c_t + sum_t p_t b_g[t]
// The head-dim order inside each 16-wide k-step is permuted identically for q
// and the codes (a dot product does not depend on the order), which lets a
// thread fetch its codes with one 8-byte shared load per row and group.  The
// P tile is transposed into the PV B operand with movmatrix.  The powers of
// two of the subnormal codes are folded into the score scale (QK^T) and into
// the final accumulator scaling (PV, 2^24 / 2^20 once).  K/V code tiles
// arrive by 2-D TMA (64-byte swizzle); scale/bias rows by 1-D bulk copies; a
// 2-stage ring shared by the CTA's 4 warps (each warp takes 64 of the 256
// tokens of every block) with full/empty mbarriers.
#include "common.cuh"
#include "internal.h"
#include "merge.cuh"

namespace kvs {

// ------------------------------------------------------------- quantiser ---
__global__ void q4_quantize_kernel(const uint16_t* __restrict__ src_k, const uint16_t* __restrict__ src_v,
                                   const int32_t* __restrict__ dst_blocks, int n_blocks, int hkv, int B, int capacity,
                                   uint8_t* __restrict__ codes_k, uint8_t* __restrict__ codes_v,
                                   __half* __restrict__ sb_k, __half* __restrict__ sb_v, uint32_t* status) {
  constexpr int D = 128, G = 64;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long per_tensor = (long long)n_blocks * hkv * B * (D / G);
  if (gid >= 2 * per_tensor) return;
  const bool is_v = gid >= per_tensor;
  long long r = is_v ? gid - per_tensor : gid;
  const int grp = static_cast<int>(r % (D / G));
  r /= (D / G);
  const long long row = r;                   // (block i, head, token) row in src
  const int i = static_cast<int>(row / ((long long)hkv * B));
  const long long rin = row - (long long)i * hkv * B;
  const int phys = dst_blocks[i];
  if (phys < 0 || phys >= capacity) {
    set_err(status, KVS_DEVERR_BLOCK_ID);
    return;
  }
  const uint16_t* x = (is_v ? src_v : src_k) + row * D + grp * G;
  float v[G];
#pragma unroll
  for (int j = 0; j < G / 8; ++j) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(x) + j);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[j * 8 + 2 * e] = bf16_lo(ws[e]);
      v[j * 8 + 2 * e + 1] = bf16_hi(ws[e]);
    }
  }
  float mn = v[0], mx = v[0];
#pragma unroll
  for (int j = 1; j < G; ++j) {
    mn = fminf(mn, v[j]);
    mx = fmaxf(mx, v[j]);
  }
  const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
  const __half b16 = __float2half_rn(mn);
  const float s = __half2float(s16), b = __half2float(b16);
  uint32_t packed[G / 8];
#pragma unroll
  for (int j = 0; j < G / 8; ++j) {
    uint32_t wv = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float cq = 0.f;
      if (s != 0.f) cq = rintf(__fdiv_rn(__fsub_rn(v[j * 8 + e], b), s));
      cq = fminf(fmaxf(cq, 0.f), 15.f);
      wv |= (static_cast<uint32_t>(cq) & 15u) << (4 * e);
    }
    packed[j] = wv;
  }
  const long long drow = (long long)phys * hkv * B + rin;
  uint8_t* cd = (is_v ? codes_v : codes_k) + drow * (D / 2) + grp * (G / 2);
  reinterpret_cast<uint4*>(cd)[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  reinterpret_cast<uint4*>(cd)[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  __half2 sbv = __halves2half2(s16, b16);
  reinterpret_cast<__half2*>((is_v ? sb_v : sb_k) + (drow * (D / G) + grp) * 2)[0] = sbv;
}

// ------------------------------------------------------------- attention ---
struct Q4Params {
  const uint16_t* q;          // bf16 [n_seq][hq][128]
  const int32_t* block_table; // [n_seq][max_blocks]
  const int32_t* seq_len;
  const uint8_t* ksb;         // fp16 scale/bias slab of this layer, 8 bytes per token-head
  const uint8_t* vsb;
  float* out;
  float* part;
  float* part_ml;
  int32_t* tickets;
  uint32_t* status;
  // mirror diffs per 16-token sub-block (nullptr: none): diff_table [n_seq]
  // [max_blocks * 16] ids into dk / dv bf16 [diff_capacity][hkv][16][128]
  const int32_t* diff_table;
  const uint16_t* dk;
  const uint16_t* dv;
  int diff_capacity;
  int max_blocks, n_seq, hkv, g, hq, bpc, n_chunks, capacity;
  float scale_log2;
};

constexpr int kQ4Sub = 16;   // tokens per mirror-diff sub-block (one warp m-tile)

constexpr int kQ4B = 256, kQ4D = 128, kQ4Stages = 2;
constexpr int kQ4Codes = kQ4B * kQ4D / 2;       // 16 KB per K or V tile
constexpr int kQ4Sb = kQ4B * 8;                 // 2 KB scale/bias per tile
constexpr int kQ4Stage = 2 * kQ4Codes + 2 * kQ4Sb;
constexpr int kQ4Smem = 1024 + kQ4Stages * kQ4Stage;

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// fp16x2 subnormals: bits [0,4) and [16,20) of w as c * 2^-24, bits [4,8)
// and [20,24) as c * 2^-20 (exact)
__device__ __forceinline__ uint32_t nib_lo_sub(uint32_t w) { return w & 0x000F000Fu; }
__device__ __forceinline__ uint32_t nib_hi_sub(uint32_t w) { return w & 0x00F000F0u; }

// The 4 diff entries of warp w's sub-blocks of block b (-1 where none; an
// id beyond the diff capacity is reported and ignored).
template <bool DIFF>
__device__ __forceinline__ int4 q4_diff_entries(const Q4Params& p, int a, int b, int warp) {
  if (!DIFF) return make_int4(-1, -1, -1, -1);
  int4 e = __ldg(reinterpret_cast<const int4*>(p.diff_table + ((size_t)a * p.max_blocks + b) * (kQ4B / kQ4Sub) + warp * 4));
  int* v = reinterpret_cast<int*>(&e);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (v[k] >= p.diff_capacity) {
      set_err(p.status, KVS_DEVERR_DIFF_ID);
      v[k] = -1;
    }
  return e;
}

__device__ __forceinline__ int int4_at(const int4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// L2 prefetch of the diff rows (DK and DV, 4 KB each) of the dirty
// sub-blocks in e, one lane per sub-block, so that the direct loads below
// find them in L2.
__device__ __forceinline__ void q4_prefetch_diffs(const Q4Params& p, const int4& e, int h, int lane) {
  if (lane >= 4) return;
  const int did = int4_at(e, lane);
  if (did < 0) return;
  const size_t off = ((size_t)did * p.hkv + h) * kQ4Sub * kQ4D;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.dk + off), "r"(kQ4Sub * kQ4D * 2) : "memory");
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.dv + off), "r"(kQ4Sub * kQ4D * 2) : "memory");
}

// q . DK for the 16 tokens of one dirty sub-block (rows g and g + 8, the
// m-tile's score rows) and query columns (2c, 2c + 1), in bf16 MMAs from the
// exact bf16 query.  Each 32-dim slice of the head dims feeds two k-steps;
// the dims are permuted identically for DK and q (thread c takes dims
// 8c .. 8c + 7 of the slice), so one 16-byte load serves both k-steps.
__device__ __forceinline__ void q4_diff_scores(const Q4Params& p, int did, int h, int g, int c, int G_,
                                               const uint16_t* qbase, float* dks) {
  const uint4* r0 = reinterpret_cast<const uint4*>(p.dk + (((size_t)did * p.hkv + h) * kQ4Sub + g) * kQ4D);
  const uint4* r1 = r0 + 8 * kQ4D / 8;
  const uint4* qr = reinterpret_cast<const uint4*>(qbase + (size_t)g * kQ4D);
#pragma unroll
  for (int j = 0; j < kQ4D / 32; ++j) {
    const uint4 x0 = __ldg(r0 + 4 * j + c), x1 = __ldg(r1 + 4 * j + c);
    const uint4 qq = g < G_ ? __ldg(qr + 4 * j + c) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t a0[4] = {x0.x, x1.x, x0.y, x1.y};
    const uint32_t a1[4] = {x0.z, x1.z, x0.w, x1.w};
    mma_bf16(dks, a0, qq.x, qq.y);
    mma_bf16(dks, a1, qq.z, qq.w);
  }
}

// P . DV of one dirty sub-block into the O^T accumulators: A = DV^T with the
// accumulators' row order (row g: head dim 8g + 2lm of the group, row g + 8:
// the next one; tokens 2c, 2c+1, 2c+8, 2c+9 as k), B = P^T (bf16) through
// movmatrix.  The accumulator rows carry 2^-24 (even dims) and 2^-20 (odd
// dims) from the subnormal V codes, so the products are scaled to match.
__device__ __forceinline__ void q4_diff_values(const Q4Params& p, int did, int h, int g, int c, const float* pv,
                                               float (*acc)[4]) {
  const uint32_t pb0 = movmatrix_t(pack_bf16(pv[0], pv[1]));
  const uint32_t pb1 = movmatrix_t(pack_bf16(pv[2], pv[3]));
  const uint16_t* vb = p.dv + ((size_t)did * p.hkv + h) * kQ4Sub * kQ4D;
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
    const int col = grp * 64 + 8 * g;
    const uint4 w0 = __ldg(reinterpret_cast<const uint4*>(vb + (2 * c) * kQ4D + col));
    const uint4 w1 = __ldg(reinterpret_cast<const uint4*>(vb + (2 * c + 1) * kQ4D + col));
    const uint4 w8 = __ldg(reinterpret_cast<const uint4*>(vb + (2 * c + 8) * kQ4D + col));
    const uint4 w9 = __ldg(reinterpret_cast<const uint4*>(vb + (2 * c + 9) * kQ4D + col));
    const uint32_t e0[4] = {w0.x, w0.y, w0.z, w0.w}, e1[4] = {w1.x, w1.y, w1.z, w1.w};
    const uint32_t e8[4] = {w8.x, w8.y, w8.z, w8.w}, e9[4] = {w9.x, w9.y, w9.z, w9.w};
#pragma unroll
    for (int lm = 0; lm < 4; ++lm) {
      const uint32_t a[4] = {__byte_perm(e0[lm], e1[lm], 0x5410), __byte_perm(e0[lm], e1[lm], 0x7632),
                             __byte_perm(e8[lm], e9[lm], 0x5410), __byte_perm(e8[lm], e9[lm], 0x7632)};
      float t[4] = {0.f, 0.f, 0.f, 0.f};
      mma_bf16(t, a, pb0, pb1);
      float* ac = acc[grp * 4 + lm];
      ac[0] = fmaf(t[0], 5.9604644775390625e-8f, ac[0]);   // 2^-24
      ac[1] = fmaf(t[1], 5.9604644775390625e-8f, ac[1]);
      ac[2] = fmaf(t[2], 9.5367431640625e-7f, ac[2]);      // 2^-20
      ac[3] = fmaf(t[3], 9.5367431640625e-7f, ac[3]);
    }
  }
}

template <bool DIFF>
__global__ void __launch_bounds__(128, 2)
q4_attn_kernel(const __grid_constant__ Q4Params p, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kQ4Stages], empty[kQ4Stages];
  __shared__ int s_last;
  __shared__ float sM[16], sL[16];
  __shared__ __align__(16) float s_acc[kAttnWarps][8][kQ4D];   // the warps' states at the end
  __shared__ float2 s_wml[kAttnWarps][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  int bid = blockIdx.x;
  const int a = bid % p.n_seq;
  bid /= p.n_seq;
  const int h = bid % p.hkv;
  const int chunk = bid / p.hkv;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  // launched as a programmatic dependent of the kernel before it on the
  // stream: nothing is read before that kernel has completed; the kernel
  // queued behind this one may then be scheduled as this grid drains (it
  // waits the same way before it reads anything)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  int L = p.seq_len[a];
  if (L < 0 || L > p.max_blocks * kQ4B) {
    if (threadIdx.x == 0 && chunk == 0) set_err(p.status, KVS_DEVERR_SEQ_LEN);
    L = L < 0 ? 0 : p.max_blocks * kQ4B;
  }
  const int nblk = (L + kQ4B - 1) / kQ4B;
  const int nch = (nblk + p.bpc - 1) / p.bpc;
  if (nblk == 0) {
    if (chunk == 0)
      for (int i = threadIdx.x; i < p.g * kQ4D; i += blockDim.x) p.out[((size_t)a * p.hq + h * p.g) * kQ4D + i] = 0.f;
    return;
  }
  if (chunk >= nch) return;
  const int b0 = chunk * p.bpc;
  const int n_mine = min(p.bpc, nblk - b0);
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int32_t* trow = p.block_table + (size_t)a * p.max_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQ4Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAttnWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int i, int s) {
    uint64_t* bar = &full[s];
    const int phys = __ldg(trow + b0 + i);
    if (phys < 0 || phys >= p.capacity) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, kQ4Stage);
    uint8_t* st = base + s * kQ4Stage;
    const int row = (phys * p.hkv + h) * kQ4B;
    tma_load_2d(st, &tk, 0, row, bar);
    tma_load_2d(st + kQ4Codes, &tv, 0, row, bar);
    bulk_load(st + 2 * kQ4Codes, p.ksb + (size_t)row * 8, kQ4Sb, bar);
    bulk_load(st + 2 * kQ4Codes + kQ4Sb, p.vsb + (size_t)row * 8, kQ4Sb, bar);
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < kQ4Stages && i < n_mine; ++i) issue(i, i);

  // ---- query as the B operand (k = head dim, n = query head), fp16.  Each
  // 32-bit code word w (elements 8w..8w+7 of this thread's 16 head dims of a
  // group) feeds two MMAs: "lo" takes the low nibbles (elements 0,4 and 2,6)
  // and "hi" the high nibbles (elements 1,5 and 3,7); the query is laid out
  // in the same k order.  The codes enter as exact fp16 subnormals (a low
  // nibble masked in place is c * 2^-24, a high nibble c * 2^-20), so
  //   (q . c) * 2^-24 = acc_lo + acc_hi / 16   (no offset, no cancellation).
  // Each query row is first scaled by a power of two 2^-e that puts its
  // largest |q| in [2^14, 2^15): every finite bf16 query then converts to
  // fp16 without overflow or loss of its leading bits, and 2^e is folded
  // back into the row's score scale (exact).
  const int G_ = p.g;
  const uint16_t* qbase = p.q + ((size_t)a * p.hq + h * G_) * kQ4D;
  uint32_t qlo[2][2][2], qhi[2][2][2];   // [group][word][k half]
  float qs[2][2];                        // [group][column 2c / 2c+1]: 2^-24 * sum of the group's q
  float colscale[2];                     // [column]: scale * log2(e) * 2^24 * 2^e(row)
  {
    const bool ok = g < G_;
    float qf[2][2][8];
    float qmax = 0.f;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
      for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int d = grp * 64 + 16 * c + 8 * w + j;
          qf[grp][w][j] = ok ? __uint_as_float((uint32_t)qbase[g * kQ4D + d] << 16) : 0.f;
          qmax = fmaxf(qmax, fabsf(qf[grp][w][j]));
        }
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
    // qmax = f * 2^x with f in [0.5, 1) and x = biased exponent - 126 (normal
    // qmax); e = x - 15; zero, subnormal and non-finite rows keep e = 0 or
    // the clamp, so both 2^-e and 2^e stay normal floats
    const int bexp = (int)((__float_as_uint(qmax) >> 23) & 255u);
    int e = (bexp > 0 && bexp < 255) ? bexp - 126 - 15 : 0;
    e = min(max(e, -100), 113);
    const float down = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
    const float up = __uint_as_float((uint32_t)(127 + e) << 23);     // 2^e
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const float* v = qf[grp][w];
        qlo[grp][w][0] = pack_f16(v[0] * down, v[4] * down);
        qlo[grp][w][1] = pack_f16(v[2] * down, v[6] * down);
        qhi[grp][w][0] = pack_f16(v[1] * down, v[5] * down);
        qhi[grp][w][1] = pack_f16(v[3] * down, v[7] * down);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float2 l2 = __half22float2(*reinterpret_cast<const __half2*>(&qlo[grp][w][k]));
          const float2 h2 = __half22float2(*reinterpret_cast<const __half2*>(&qhi[grp][w][k]));
          sum += (l2.x + l2.y) + (h2.x + h2.y);
        }
      }
      // sums over the 4 lanes of row g, then fetched for columns 2c and 2c+1
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum *= 5.9604644775390625e-8f;   // 2^-24
      qs[grp][0] = __shfl_sync(0xffffffffu, sum, (2 * c) * 4);
      qs[grp][1] = __shfl_sync(0xffffffffu, sum, (2 * c + 1) * 4);
    }
    const float rs = p.scale_log2 * 16777216.f;   // 2^24
    colscale[0] = rs * __shfl_sync(0xffffffffu, up, (2 * c) * 4);
    colscale[1] = rs * __shfl_sync(0xffffffffu, up, (2 * c + 1) * 4);
  }

  // the same per-column constants as packed pairs (columns 2c, 2c+1)
  const float2 qs2[2] = {make_float2(qs[0][0], qs[0][1]), make_float2(qs[1][0], qs[1][1])};
  const float2 cs2 = make_float2(colscale[0], colscale[1]);
  const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float acc[8][4];
  float corr[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  // mirror diffs: this warp's sub-block entries of the current block and of
  // the next two; the rows of block i + 2's dirty sub-blocks are prefetched
  // into L2 at the end of block i
  int4 d_cur = make_int4(-1, -1, -1, -1), d_n1 = d_cur, d_n2 = d_cur;
  if (DIFF) {
    if (n_mine > 0) d_cur = q4_diff_entries<DIFF>(p, a, b0, warp);
    if (n_mine > 1) d_n1 = q4_diff_entries<DIFF>(p, a, b0 + 1, warp);
    q4_prefetch_diffs(p, d_cur, h, lane);
    q4_prefetch_diffs(p, d_n1, h, lane);
  }

  bool timed_out = false;
  for (int i = 0; i < n_mine; ++i) {
    const int s = i % kQ4Stages;
    if (DIFF) d_n2 = i + 2 < n_mine ? q4_diff_entries<DIFF>(p, a, b0 + i + 2, warp) : make_int4(-1, -1, -1, -1);
    if (!mbar_wait_bounded(&full[s], (i / kQ4Stages) & 1, p.status)) {
      timed_out = true;
      break;
    }
    const int b = b0 + i;
    const int phys = __ldg(trow + b);
    const int nv = min(kQ4B, L - b * kQ4B);
    const int tw = warp * 64;   // this warp's first token in the block
    if (phys >= 0 && phys < p.capacity && tw < nv) {
      const uint8_t* kc = base + s * kQ4Stage;
      const uint8_t* vc = kc + kQ4Codes;
      const uint8_t* ksb = kc + 2 * kQ4Codes;
      const uint8_t* vsb = ksb + kQ4Sb;
      float sc[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int t0 = tw + 16 * mt + g, t1 = t0 + 8;
        // 2^-24 q . c per group: [group][row t0 / t1], columns (2c, 2c+1) as a pair
        float2 cg[2][2];
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
          float al_[4] = {0.f, 0.f, 0.f, 0.f}, ah_[4] = {0.f, 0.f, 0.f, 0.f};
          const uint2 w0 = *reinterpret_cast<const uint2*>(kc + swz64(t0 * 64 + 32 * grp + 8 * c));
          const uint2 w1 = *reinterpret_cast<const uint2*>(kc + swz64(t1 * 64 + 32 * grp + 8 * c));
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const uint32_t r0 = w ? w0.y : w0.x, r1 = w ? w1.y : w1.x;
            const uint32_t s0 = r0 >> 8, s1 = r1 >> 8;
            mma_f16(al_, nib_lo_sub(r0), nib_lo_sub(r1), nib_lo_sub(s0), nib_lo_sub(s1), qlo[grp][w][0], qlo[grp][w][1]);
            mma_f16(ah_, nib_hi_sub(r0), nib_hi_sub(r1), nib_hi_sub(s0), nib_hi_sub(s1), qhi[grp][w][0], qhi[grp][w][1]);
          }
          const float2 s16 = make_float2(0.0625f, 0.0625f);
          cg[grp][0] = __ffma2_rn(make_float2(ah_[0], ah_[1]), s16, make_float2(al_[0], al_[1]));
          cg[grp][1] = __ffma2_rn(make_float2(ah_[2], ah_[3]), s16, make_float2(al_[2], al_[3]));
        }
        float dks[4] = {0.f, 0.f, 0.f, 0.f};   // q . DK of a dirty sub-block (true units)
        if (DIFF && int4_at(d_cur, mt) >= 0) q4_diff_scores(p, int4_at(d_cur, mt), h, g, c, G_, qbase, dks);
        const uint2 sb0 = *reinterpret_cast<const uint2*>(ksb + t0 * 8);
        const uint2 sb1 = *reinterpret_cast<const uint2*>(ksb + t1 * 8);
        const float2 g00 = __half22float2(*reinterpret_cast<const __half2*>(&sb0.x));   // (s, b) group 0, t0
        const float2 g01 = __half22float2(*reinterpret_cast<const __half2*>(&sb0.y));   // group 1, t0
        const float2 g10 = __half22float2(*reinterpret_cast<const __half2*>(&sb1.x));
        const float2 g11 = __half22float2(*reinterpret_cast<const __half2*>(&sb1.y));
        // per row (t0, t1), both columns at once (packed fp32 pairs):
        // x = s0 cg0 + b0 qs0 + s1 cg1 + b1 qs1, score = dks scale + x colscale
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const float2 s0 = hr ? g10 : g00;
          const float2 s1 = hr ? g11 : g01;
          float2 x = __fmul2_rn(make_float2(s0.x, s0.x), cg[0][hr]);
          x = __ffma2_rn(make_float2(s0.y, s0.y), qs2[0], x);
          x = __ffma2_rn(make_float2(s1.x, s1.x), cg[1][hr], x);
          x = __ffma2_rn(make_float2(s1.y, s1.y), qs2[1], x);
          const float2 y = __ffma2_rn(make_float2(dks[2 * hr], dks[2 * hr + 1]), sl2, __fmul2_rn(x, cs2));
          const bool live = (hr ? t1 : t0) < nv;
          sc[mt][2 * hr] = live ? y.x : -INFINITY;
          sc[mt][2 * hr + 1] = live ? y.y : -INFINITY;
        }
      }
      // online softmax over this warp's 64 tokens, per query column
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        mx[0] = fmaxf(mx[0], fmaxf(sc[mt][0], sc[mt][2]));
        mx[1] = fmaxf(mx[1], fmaxf(sc[mt][1], sc[mt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
      }
      float al[2];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const float mn = fmaxf(m[cc], mx[cc]);
        al[cc] = fast_exp2(m[cc] - mn);
        m[cc] = mn;
      }
      // rescale the state only when some column's maximum moved
      if (__any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f)) {
        const float2 al2 = make_float2(al[0], al[1]);
        float2 t = __fmul2_rn(make_float2(l[0], l[1]), al2);
        l[0] = t.x; l[1] = t.y;
        t = __fmul2_rn(make_float2(corr[0][0], corr[0][1]), al2);
        corr[0][0] = t.x; corr[0][1] = t.y;
        t = __fmul2_rn(make_float2(corr[1][0], corr[1][1]), al2);
        corr[1][0] = t.x; corr[1][1] = t.y;
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {
          const float2 a01 = __fmul2_rn(make_float2(acc[i2][0], acc[i2][1]), al2);
          const float2 a23 = __fmul2_rn(make_float2(acc[i2][2], acc[i2][3]), al2);
          acc[i2][0] = a01.x; acc[i2][1] = a01.y;
          acc[i2][2] = a23.x; acc[i2][3] = a23.y;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const int t0 = tw + 16 * mt + g, t1 = t0 + 8;
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = fast_exp2(sc[mt][e] - m[e & 1]);
        l[0] += pv[0] + pv[2];
        l[1] += pv[1] + pv[3];
        const uint2 sb0 = *reinterpret_cast<const uint2*>(vsb + t0 * 8);
        const uint2 sb1 = *reinterpret_cast<const uint2*>(vsb + t1 * 8);
        const float2 v00 = __half22float2(*reinterpret_cast<const __half2*>(&sb0.x));
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&sb0.y));
        const float2 v10 = __half22float2(*reinterpret_cast<const __half2*>(&sb1.x));
        const float2 v11 = __half22float2(*reinterpret_cast<const __half2*>(&sb1.y));
        // B operands (k = token, n = query head) per group, via transposition
        uint32_t bb[2][2];
        // (P of rows t0 and t1, both columns as packed pairs)
        const float2 p0 = make_float2(pv[0], pv[1]), p1 = make_float2(pv[2], pv[3]);
        float2 t = __fmul2_rn(p0, make_float2(v00.x, v00.x));
        bb[0][0] = movmatrix_t(pack_f16(t.x, t.y));
        t = __fmul2_rn(p1, make_float2(v10.x, v10.x));
        bb[0][1] = movmatrix_t(pack_f16(t.x, t.y));
        t = __fmul2_rn(p0, make_float2(v01.x, v01.x));
        bb[1][0] = movmatrix_t(pack_f16(t.x, t.y));
        t = __fmul2_rn(p1, make_float2(v11.x, v11.x));
        bb[1][1] = movmatrix_t(pack_f16(t.x, t.y));
        t = __ffma2_rn(p1, make_float2(v10.y, v10.y), __fmul2_rn(p0, make_float2(v00.y, v00.y)));
        t = __fadd2_rn(make_float2(corr[0][0], corr[0][1]), t);
        corr[0][0] = t.x; corr[0][1] = t.y;
        t = __ffma2_rn(p1, make_float2(v11.y, v11.y), __fmul2_rn(p0, make_float2(v01.y, v01.y)));
        t = __fadd2_rn(make_float2(corr[1][0], corr[1][1]), t);
        corr[1][0] = t.x; corr[1][1] = t.y;
        // A operand: V codes, m = head dim (row g: the even dim 8g + 2lm of
        // the group's 64, as c * 2^-24; row g + 8: the odd one, as c * 2^-20),
        // k = token
        const int tb = tw + 16 * mt;
        const int tr[4] = {tb + 2 * c, tb + 2 * c + 1, tb + 2 * c + 8, tb + 2 * c + 9};
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
          uint32_t wv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) wv[u] = *reinterpret_cast<const uint32_t*>(vc + swz64(tr[u] * 64 + 32 * grp + 4 * g));
#pragma unroll
          for (int lm = 0; lm < 4; ++lm) {
            const uint32_t sel = (uint32_t)lm | ((uint32_t)(4 + lm) << 8);
            const uint32_t x01 = __byte_perm(wv[0], wv[1], sel);
            const uint32_t x89 = __byte_perm(wv[2], wv[3], sel);
            mma_f16(acc[grp * 4 + lm], nib_lo_sub(x01), nib_hi_sub(x01), nib_lo_sub(x89), nib_hi_sub(x89),
                    bb[grp][0], bb[grp][1]);
          }
        }
        if (DIFF && int4_at(d_cur, mt) >= 0) q4_diff_values(p, int4_at(d_cur, mt), h, g, c, pv, acc);
      }
    }
    if (DIFF) {
      q4_prefetch_diffs(p, d_n2, h, lane);
      d_cur = d_n1;
      d_n1 = d_n2;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (threadIdx.x == 0 && i + kQ4Stages < n_mine) {
      if (!mbar_wait_bounded(&empty[s], (i / kQ4Stages) & 1, p.status)) {
        timed_out = true;
      } else {
        // every warp has arrived after its last read of the stage (plain
        // reads that have completed): the copy may overwrite it with no
        // proxy fence
        issue(i + kQ4Stages, s);
      }
    }
    if (__shfl_sync(0xffffffffu, timed_out ? 1 : 0, 0)) break;
  }
  if (timed_out) {
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }
  // reduce l and the bias corrections over the 8 token lanes of each column
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      l[cc] += __shfl_xor_sync(0xffffffffu, l[cc], o);
      corr[0][cc] += __shfl_xor_sync(0xffffffffu, corr[0][cc], o);
      corr[1][cc] += __shfl_xor_sync(0xffffffffu, corr[1][cc], o);
    }
  }
  // The four warps' states (64 tokens of every block each) combine in
  // shared memory into one split per CTA, so the merge behind the last CTA
  // of the (sequence, KV head) reads one split per chunk.
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int r = 2 * c + cc;
    if (r >= G_) continue;
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
      for (int lm = 0; lm < 4; ++lm) {
        const int d0 = grp * 64 + 8 * g + 2 * lm;
        *reinterpret_cast<float2*>(&s_acc[warp][r][d0]) =
            make_float2(fmaf(acc[grp * 4 + lm][cc], 16777216.f, corr[grp][cc]),
                        fmaf(acc[grp * 4 + lm][2 + cc], 1048576.f, corr[grp][cc]));
      }
    }
    if (g == 0) s_wml[warp][r] = make_float2(m[cc], l[cc]);
  }
  __syncthreads();
  const size_t sidx = ((size_t)a * p.hkv + h) * p.n_chunks + chunk;
  {
    const int r = threadIdx.x >> 4, c0 = (threadIdx.x & 15) * 8;   // 8 rows x 16 threads of 8 columns
    if (r < G_) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w)
        if (s_wml[w][r].y > 0.f) M = fmaxf(M, s_wml[w][r].x);
      float Lc = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float2 ml = s_wml[w][r];
        const float wt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
        Lc += wt * ml.y;
        const float4 x0 = *reinterpret_cast<const float4*>(&s_acc[w][r][c0]);
        const float4 x1 = *reinterpret_cast<const float4*>(&s_acc[w][r][c0 + 4]);
        o[0] += wt * x0.x; o[1] += wt * x0.y; o[2] += wt * x0.z; o[3] += wt * x0.w;
        o[4] += wt * x1.x; o[5] += wt * x1.y; o[6] += wt * x1.z; o[7] += wt * x1.w;
      }
      float* pr = p.part + (sidx * G_ + r) * kQ4D + c0;
      __stcg(reinterpret_cast<float4*>(pr), make_float4(o[0], o[1], o[2], o[3]));
      __stcg(reinterpret_cast<float4*>(pr + 4), make_float4(o[4], o[5], o[6], o[7]));
      if ((threadIdx.x & 15) == 0) __stcg(reinterpret_cast<float2*>(p.part_ml + (sidx * G_ + r) * 2), make_float2(M, Lc));
    }
  }
  if (!arrive_last(p.tickets + a * p.hkv + h, nch, &s_last)) return;
  const size_t s0 = ((size_t)a * p.hkv + h) * p.n_chunks;
  merge_splits<kQ4D>(p.part, p.part_ml, s0, nch, G_, p.out + ((size_t)a * p.hq + h * G_) * kQ4D, sM, sL);
}

AttnPlan q4_plan(const kvs_pool* pool, int n_seq, int max_blocks) {
  // about one wave of CTAs (two resident per SM): each CTA streams several
  // 256-token blocks so its pipeline start-up is amortised
  const long long work = (long long)n_seq * pool->desc.num_kv_heads * max_blocks;
  const long long target = (long long)pool->num_sms * 2;
  long long bpc = (work + target - 1) / target;
  if (bpc < 1) bpc = 1;
  if (bpc > 64) bpc = 64;
  AttnPlan pl;
  pl.bpc = static_cast<int>(bpc);
  pl.n_chunks = (max_blocks + pl.bpc - 1) / pl.bpc;
  if (pl.n_chunks < 1) pl.n_chunks = 1;
  return pl;
}

}  // namespace kvs

using namespace kvs;

extern "C" kvs_status kvs_quantize_q4(kvs_pool* pool, int32_t layer, const void* k_src_dev, const void* v_src_dev,
                                      const int32_t* dst_blocks_dev, int32_t n_blocks, cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: null pool");
  const kvs_pool_desc& d = pool->desc;
  if (d.dtype != KVS_DTYPE_Q4G64) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: pool is not Q4G64");
  if (layer < 0 || layer >= d.num_layers) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: layer out of range");
  if (n_blocks < 0) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: n_blocks < 0");
  if (n_blocks == 0) return KVS_OK;
  if (!k_src_dev || !v_src_dev || !dst_blocks_dev) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: null pointer");
  if (!aligned16(k_src_dev) || !aligned16(v_src_dev)) return fail(KVS_ERR_INVALID_ARG, "quantize_q4: sources must be 16-byte aligned");
  const long long threads = 2ll * n_blocks * d.num_kv_heads * d.block_tokens * (d.head_dim / 64);
  const int tb = 128;
  q4_quantize_kernel<<<(unsigned)((threads + tb - 1) / tb), tb, 0, stream>>>(
      static_cast<const uint16_t*>(k_src_dev), static_cast<const uint16_t*>(v_src_dev), dst_blocks_dev, n_blocks,
      d.num_kv_heads, d.block_tokens, d.capacity_blocks, static_cast<uint8_t*>(pool->k[layer]),
      static_cast<uint8_t*>(pool->v[layer]), static_cast<__half*>(pool->ksb[layer]), static_cast<__half*>(pool->vsb[layer]),
      pool->status);
  count_launch();
  return check_launch("quantize_q4");
}

extern "C" kvs_status kvs_decode_attn_q4(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                                         const int32_t* block_table_dev, int32_t max_blocks, const int32_t* seq_len_dev,
                                         int32_t n_seq, const int32_t* diff_table_dev, float scale, float* out_dev,
                                         void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: null pool");
  const kvs_pool_desc& d = pool->desc;
  if (d.dtype != KVS_DTYPE_Q4G64) return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: pool is not Q4G64");
  if (layer < 0 || layer >= d.num_layers) return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: layer out of range");
  if (n_seq < 0 || n_seq > d.max_seqs) return fail(KVS_ERR_CAPACITY, "decode_attn_q4: n_seq exceeds the pool's max_seqs");
  if (n_seq == 0) return KVS_OK;
  if (!q_dev || !block_table_dev || !seq_len_dev || !out_dev || !ws)
    return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: null pointer");
  if (!aligned16(q_dev) || !aligned16(out_dev) || !aligned16(ws))
    return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: q, out and ws must be 16-byte aligned");
  if (diff_table_dev && (d.diff_capacity_blocks < 1 || !aligned16(diff_table_dev)))
    return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: a diff table needs a pool with diff slabs and 16-byte alignment");
  if (max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: max_blocks must be >= 1");
  if (n_q_heads < 1 || n_q_heads % d.num_kv_heads) return fail(KVS_ERR_INVALID_ARG, "decode_attn_q4: n_q_heads must be a multiple of num_kv_heads");
  const int g = n_q_heads / d.num_kv_heads;
  if (g > 8) return fail(KVS_ERR_UNSUPPORTED, "decode_attn_q4: more than 8 query heads per KV head");
  const AttnPlan plan = q4_plan(pool, n_seq, max_blocks);
  size_t need = 0;
  kvs_workspace_size(pool, KVS_OP_DECODE_ATTN_Q4, n_seq, max_blocks, n_q_heads, &need);
  if (ws_bytes < need) return fail(KVS_ERR_CAPACITY, "decode_attn_q4: workspace too small");
  const long long grid = (long long)n_seq * d.num_kv_heads * plan.n_chunks;
  if (grid > 0x7fffffffll) return fail(KVS_ERR_CAPACITY, "decode_attn_q4: grid too large");
  Q4Params prm{};
  prm.q = static_cast<const uint16_t*>(q_dev);
  prm.block_table = block_table_dev;
  prm.seq_len = seq_len_dev;
  prm.ksb = static_cast<const uint8_t*>(pool->ksb[layer]);
  prm.vsb = static_cast<const uint8_t*>(pool->vsb[layer]);
  prm.out = out_dev;
  const size_t splits = (size_t)n_seq * d.num_kv_heads * plan.n_chunks * kAttnWarps;
  prm.part = static_cast<float*>(ws);
  prm.part_ml = prm.part + splits * g * kQ4D;
  prm.tickets = pool->tickets;
  prm.status = pool->status;
  prm.diff_table = diff_table_dev;
  if (diff_table_dev) {
    prm.dk = static_cast<const uint16_t*>(pool->dk[layer]);
    prm.dv = static_cast<const uint16_t*>(pool->dv[layer]);
    prm.diff_capacity = d.diff_capacity_blocks;
  }
  prm.max_blocks = max_blocks;
  prm.n_seq = n_seq;
  prm.hkv = d.num_kv_heads;
  prm.g = g;
  prm.hq = n_q_heads;
  prm.bpc = plan.bpc;
  prm.n_chunks = plan.n_chunks;
  prm.capacity = d.capacity_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  auto kern = diff_table_dev ? q4_attn_kernel<true> : q4_attn_kernel<false>;
  if (!(diff_table_dev ? smem_limit_once<q4_attn_kernel<true>>(kQ4Smem, pool->device)
                       : smem_limit_once<q4_attn_kernel<false>>(kQ4Smem, pool->device)))
    return fail(KVS_ERR_CUDA, "decode_attn_q4: cannot raise the shared-memory limit");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kQ4Smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm, pool->tk[layer], pool->tv[layer]) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_attn_q4: launch failed");
  count_launch();
  return check_launch("decode_attn_q4");
}
