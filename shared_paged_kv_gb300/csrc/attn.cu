// Paged decode attention over a shared bf16 KV block pool, with the mirror
// diff overlay and the segment RoPE restore fused into the read.
//
// What is computed (TokenDance summary, section 3 / Fig. 8: blocks carrying a
// diff are corrected on chip before attention, no dense mirror is built; INMS
// walkthrough §3.2: reused K is rotated by the position shift, V is not;
// MemDecay post §4.2: softmax(q.k / sqrt(d)) V):
//   out[a][h] = sum_t softmax_t(scale * <q, R(delta)(K + DK)>) (V + DV)
//
// How (GB300): one CTA = 4 warps = one (sequence, kv head, chunk of logical
// blocks).  Each warp owns a contiguous quarter of the chunk and a private
// ring of S shared-memory stages; lane 0 gathers each 16-token block of K and
// V (and, when the block carries a diff, the diff tiles) through the block
// table with 3-D TMA tensor loads (128-byte swizzle) completing on an
// mbarrier.  The G query heads of the KV head form a 16-row tile (rows >= G
// are zero) so QK^T and PV run on mma.sync m16n8k16 with fp32 accumulation.
// The diff overlay uses linearity: q.(K+DK) = q.K + q.DK and p.(V+DV) =
// p.V + p.DV accumulate into the same fragments.  Rotation is moved to the
// query: <q, R(d)k> = <R(-d)q, k>, so K bytes are read as stored and only the
// query fragments are re-rotated when the segment changes.  Each warp keeps an
// online-softmax state and writes an (m, l, acc) split; the last CTA of the
// (sequence, kv head) to arrive merges all splits (an arrival counter, no
// spinning) and writes fp32 output.
#include <cfloat>

#include "common.cuh"
#include "internal.h"
#include "merge.cuh"

namespace kvs {

struct AttnParams {
  const uint16_t* q;          // bf16 bits [n_seq][hq][D]
  const int32_t* block_table; // [n_seq][max_blocks]
  const int32_t* seq_len;     // [n_seq]
  const int32_t* diff_table;  // [n_seq][max_blocks] or null
  const int32_t* rope_off;    // [n_seq+1] or null
  const int4* rope_segs;      // {first_block, n_blocks, delta, -}
  float* out;                 // [n_seq][hq][D]
  float* part;                // [splits][g][D]
  float* part_ml;             // [splits][g][2]
  int32_t* tickets;           // [n_seq * hkv]
  uint32_t* status;
  int max_blocks, n_seq, hkv, g, hq, bpc, n_chunks, capacity, diff_capacity;
  float scale_log2;
  RopeSplit rs;
};

template <int D>
struct AttnCfg {
  static constexpr int B = 16;
  static constexpr int TILE = B * D * 2;
  static constexpr int KS = D / 16;
};

template <int D, bool DIFF>
__host__ __device__ constexpr int attn_stages() {
  return (D == 128) ? 3 : (DIFF ? 3 : 4);
}

template <int D, bool DIFF, int W = kAttnWarps>
__host__ __device__ constexpr int attn_smem_bytes() {
  return 1024 + W * attn_stages<D, DIFF>() * (DIFF ? 4 : 2) * AttnCfg<D>::TILE;
}

// Warps per CTA: four, or eight for calls that take a whole (sequence, KV
// head) in one CTA (twice the warps on its blocks, half the chain per warp)
// where eight warps' rings fit in shared memory.
template <int D, bool DIFF>
__host__ __device__ constexpr bool attn_wide_cta_ok() {
  return attn_smem_bytes<D, DIFF, 8>() <= 227 * 1024;
}


template <int D, bool DIFF, bool ROPE, int W>
__global__ void __launch_bounds__(32 * W, W == 4 ? 2 : 1)
attn_bf16_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdk,
                 const __grid_constant__ CUtensorMap tdv) {
  using C = AttnCfg<D>;
  constexpr int B = C::B, TILE = C::TILE, KS = C::KS;
  constexpr int S = attn_stages<D, DIFF>();
  constexpr int NT = DIFF ? 4 : 2;
  constexpr int STAGE = NT * TILE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[W][S];
  __shared__ int s_last;
  __shared__ float sM[16], sL[16];
  __shared__ float rsc[ROPE ? 4 * 64 : 1];   // RoPE frequency pieces (rotation calls)
  __shared__ float2 s_wml[W][16];    // the warps' (m, l) at the end
  if (threadIdx.x == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    if (DIFF) {
      prefetch_tmap(&tdk);
      prefetch_tmap(&tdv);
    }
  }
  if (ROPE) {
    for (int i = threadIdx.x; i < 4 * 64; i += blockDim.x) rsc[i] = p.rs.c[i >> 6][i & 63];
    __syncthreads();
  }
  // launched as a programmatic dependent of the kernel before it on the
  // stream: nothing is read before that kernel has completed; the kernel
  // queued behind this one may be scheduled as this grid drains
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  int bid = blockIdx.x;
  const int a = bid % p.n_seq;
  bid /= p.n_seq;
  const int h = bid % p.hkv;
  const int chunk = bid / p.hkv;

  int L = p.seq_len[a];
  if (L < 0 || L > p.max_blocks * B) {
    if (threadIdx.x == 0 && chunk == 0) set_err(p.status, KVS_DEVERR_SEQ_LEN);
    L = L < 0 ? 0 : p.max_blocks * B;
  }
  const int nblk = (L + B - 1) / B;
  const int nch = (nblk + p.bpc - 1) / p.bpc;
  if (nblk == 0) {
    if (chunk == 0)
      for (int i = threadIdx.x; i < p.g * D; i += blockDim.x) p.out[((size_t)a * p.hq + h * p.g) * D + i] = 0.f;
    return;
  }
  if (chunk >= nch) return;

  // ---- shared memory carve-up (1024-byte aligned tiles for the swizzle)
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* wbase = base + warp * S * STAGE;
  const uint32_t wbase_u32 = smem_u32(wbase);

  // ---- this warp's contiguous block range
  const int quarter = p.bpc / W;
  const int b_first = chunk * p.bpc + warp * quarter;
  int n_mine = min(quarter, nblk - b_first);
  if (n_mine < 0) n_mine = 0;
  const int32_t* trow = p.block_table + (size_t)a * p.max_blocks;
  const int32_t* drow = DIFF ? p.diff_table + (size_t)a * p.max_blocks : nullptr;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[warp][s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto issue = [&](int i, int s) {
    const int b = b_first + i;
    uint64_t* bar = &bars[warp][s];
    const int phys = __ldg(trow + b);
    if (phys < 0 || phys >= p.capacity) {
      set_err(p.status, KVS_DEVERR_BLOCK_ID);
      mbar_arrive(bar);
      return;
    }
    int did = -1;
    if (DIFF) {
      did = __ldg(drow + b);
      if (did >= p.diff_capacity) {
        set_err(p.status, KVS_DEVERR_DIFF_ID);
        did = -1;
      }
    }
    mbar_arrive_expect_tx(bar, (did >= 0 ? 4 : 2) * TILE);
    uint8_t* st = wbase + s * STAGE;
    const int row = (phys * p.hkv + h) * B;
    tma_load_kv_tile<D>(st, &tk, row, bar);
    tma_load_kv_tile<D>(st + TILE, &tv, row, bar);
    if (DIFF && did >= 0) {
      const int drow_ = (did * p.hkv + h) * B;
      tma_load_kv_tile<D>(st + 2 * TILE, &tdk, drow_, bar);
      tma_load_kv_tile<D>(st + 3 * TILE, &tdv, drow_, bar);
    }
  };

  if (lane == 0)
    for (int i = 0; i < S && i < n_mine; ++i) issue(i, i);

  // ---- query fragments (A operand, 16 rows x D, rows >= g are zero)
  const bool r0ok = g < p.g, r1ok = g + 8 < p.g;
  const uint16_t* q0 = p.q + ((size_t)a * p.hq + h * p.g + g) * D;
  const uint16_t* q1 = q0 + 8 * D;
  uint32_t qa[KS][4];
  // low part of a rotated query (q' - bf16(q')), so q' enters the MMA to
  // ~16 significant bits; zero while the query is unrotated (exact bf16)
  uint32_t qa_lo[ROPE ? KS : 1][4];
  bool q_has_lo = false;
  auto load_q = [&]() {
    q_has_lo = false;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int col = kk * 16 + 2 * c;
      qa[kk][0] = r0ok ? __ldg(reinterpret_cast<const uint32_t*>(q0 + col)) : 0u;
      qa[kk][1] = r1ok ? __ldg(reinterpret_cast<const uint32_t*>(q1 + col)) : 0u;
      qa[kk][2] = r0ok ? __ldg(reinterpret_cast<const uint32_t*>(q0 + col + 8)) : 0u;
      qa[kk][3] = r1ok ? __ldg(reinterpret_cast<const uint32_t*>(q1 + col + 8)) : 0u;
    }
  };
  // query rotated by -delta: q'_lo = lo*cos + hi*sin, q'_hi = hi*cos - lo*sin
  auto rotate_q = [&](int delta) {
    q_has_lo = true;
#pragma unroll
    for (int kk = 0; kk < KS / 2; ++kk) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {   // columns +0/+1 and +8/+9
        const int col = kk * 16 + 2 * c + half * 8;
        float cs0, sn0, cs1, sn1;
        rope_cos_sin(rsc, col, delta, cs0, sn0);
        rope_cos_sin(rsc, col + 1, delta, cs1, sn1);
#pragma unroll
        for (int row = 0; row < 2; ++row) {
          const bool ok = row ? r1ok : r0ok;
          const uint16_t* qr = row ? q1 : q0;
          uint32_t lo = ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + col)) : 0u;
          uint32_t hi = ok ? __ldg(reinterpret_cast<const uint32_t*>(qr + col + D / 2)) : 0u;
          const float l0 = bf16_lo(lo), l1 = bf16_hi(lo), h0 = bf16_lo(hi), h1 = bf16_hi(hi);
          split_bf16(l0 * cs0 + h0 * sn0, l1 * cs1 + h1 * sn1, qa[kk][half * 2 + row],
                     qa_lo[ROPE ? kk : 0][half * 2 + row]);
          split_bf16(h0 * cs0 - l0 * sn0, h1 * cs1 - l1 * sn1, qa[kk + KS / 2][half * 2 + row],
                     qa_lo[ROPE ? kk + KS / 2 : 0][half * 2 + row]);
        }
      }
    }
  };
  load_q();
  int cur_delta = 0, seg_lo = 0, seg_hi = 0;   // cached segment [lo, hi)
  const int seg_beg = ROPE ? p.rope_off[a] : 0;
  const int seg_end = ROPE ? p.rope_off[a + 1] : 0;

  // ---- per-lane ldmatrix offsets
  uint32_t koff[KS], voff[KS];
  {
    const int mi = lane >> 3, r = lane & 7;
    const int tk_ = ((mi >> 1) << 3) + r, ck = (mi & 1) << 3;
    const int tv_ = ((mi & 1) << 3) + r, cv = (mi >> 1) << 3;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      koff[kk] = kv_tile_off<D>(tk_, kk * 16 + ck);
      voff[kk] = kv_tile_off<D>(tv_, kk * 16 + cv);
    }
  }

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  bool timed_out = false;
  int i = 0;
  for (; i < n_mine; ++i) {
    const int s = i % S;
    const uint32_t par = (i / S) & 1;
    if (!mbar_wait_bounded(&bars[warp][s], par, p.status)) {
      timed_out = true;
      break;
    }
    const int b = b_first + i;
    const int phys = __ldg(trow + b);
    if (phys >= 0 && phys < p.capacity) {
      int did = -1;
      if (DIFF) {
        did = __ldg(drow + b);
        if (did >= p.diff_capacity) did = -1;
      }
      if (ROPE) {
        if (b < seg_lo || b >= seg_hi) {
          int found = 0x7fffffff, fd = 0, flo = 0, fhi = 0;
          for (int e = seg_beg + lane; e < seg_end; e += 32) {
            const int4 sg = __ldg(p.rope_segs + e);
            if (b >= sg.x && b < sg.x + sg.y && e < found) {
              found = e; fd = sg.z; flo = sg.x; fhi = sg.x + sg.y;
            }
          }
#pragma unroll
          for (int o = 16; o; o >>= 1) {
            const int f2 = __shfl_xor_sync(0xffffffffu, found, o);
            const int d2 = __shfl_xor_sync(0xffffffffu, fd, o);
            const int lo2 = __shfl_xor_sync(0xffffffffu, flo, o);
            const int hi2 = __shfl_xor_sync(0xffffffffu, fhi, o);
            if (f2 < found) { found = f2; fd = d2; flo = lo2; fhi = hi2; }
          }
          int nd = 0;
          if (found != 0x7fffffff) {
            nd = fd; seg_lo = flo; seg_hi = fhi;
          } else {
            seg_lo = seg_hi = 0;
          }
          if (nd <= -(1 << 18) || nd >= (1 << 18)) {
            if (lane == 0) set_err(p.status, KVS_DEVERR_ROPE_RANGE);
            nd = 0;
          }
          if (nd != cur_delta) {
            if (nd == 0) load_q(); else rotate_q(nd);
            cur_delta = nd;
          }
        }
      }
      const uint32_t tkb = wbase_u32 + s * STAGE;
      const uint32_t tvb = tkb + TILE;
      // S = Q K^T over 16 tokens (two n-tiles of 8)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tkb + koff[kk], b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk], b0, b1);
        mma_bf16(sc[1], qa[kk], b2, b3);
        if (ROPE && q_has_lo) {
          mma_bf16(sc[0], qa_lo[ROPE ? kk : 0], b0, b1);
          mma_bf16(sc[1], qa_lo[ROPE ? kk : 0], b2, b3);
        }
      }
      if (DIFF && did >= 0) {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(tkb + 2 * TILE + koff[kk], b0, b1, b2, b3);
          mma_bf16(sc[0], qa[kk], b0, b1);
          mma_bf16(sc[1], qa[kk], b2, b3);
          if (ROPE && q_has_lo) {
            mma_bf16(sc[0], qa_lo[ROPE ? kk : 0], b0, b1);
            mma_bf16(sc[1], qa_lo[ROPE ? kk : 0], b2, b3);
          }
        }
      }
      const int nv = min(B, L - b * B);
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int tok = n * 8 + 2 * c + (j & 1);
          float x = sc[n][j] * p.scale_log2;
          if (tok >= nv) x = -INFINITY;
          sc[n][j] = x;
        }
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      // Lazy rescale: a row keeps its reference point while none of its
      // scores exceeds it by more than 2^8 in P (the bf16 hi + lo split and
      // the fp32 sums carry such P at full relative precision); only then are
      // the row maxima reduced and l and the accumulators rescaled.
      if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // (a row whose state is still empty has l = 0 and acc = 0)
        const float al0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mn0);
        const float al1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          acc[n][0] *= al0; acc[n][1] *= al0;
          acc[n][2] *= al1; acc[n][3] *= al1;
        }
      }
      // nothing live yet: reference point 0, so that 2^(-inf - 0) = 0
      const float r0 = m0 == -INFINITY ? 0.f : m0, r1 = m1 == -INFINITY ? 0.f : m1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        sc[n][0] = fast_exp2(sc[n][0] - r0);
        sc[n][1] = fast_exp2(sc[n][1] - r0);
        sc[n][2] = fast_exp2(sc[n][2] - r1);
        sc[n][3] = fast_exp2(sc[n][3] - r1);
        ps0 += sc[n][0] + sc[n][1];
        ps1 += sc[n][2] + sc[n][3];
      }
      l0 += ps0;
      l1 += ps1;
      // P = P_hi + P_lo, both bf16, so the probabilities enter the PV MMA to
      // ~16 significant bits (V is exact bf16)
      uint32_t pa[4], pl[4];
      split_bf16(sc[0][0], sc[0][1], pa[0], pl[0]);
      split_bf16(sc[0][2], sc[0][3], pa[1], pl[1]);
      split_bf16(sc[1][0], sc[1][1], pa[2], pl[2]);
      split_bf16(sc[1][2], sc[1][3], pa[3], pl[3]);
#pragma unroll
      for (int jj = 0; jj < KS; ++jj) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tvb + voff[jj], b0, b1, b2, b3);
        mma_bf16(acc[2 * jj], pa, b0, b1);
        mma_bf16(acc[2 * jj + 1], pa, b2, b3);
        mma_bf16(acc[2 * jj], pl, b0, b1);
        mma_bf16(acc[2 * jj + 1], pl, b2, b3);
      }
      if (DIFF && did >= 0) {
#pragma unroll
        for (int jj = 0; jj < KS; ++jj) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(tvb + 2 * TILE + voff[jj], b0, b1, b2, b3);
          mma_bf16(acc[2 * jj], pa, b0, b1);
          mma_bf16(acc[2 * jj + 1], pa, b2, b3);
          mma_bf16(acc[2 * jj], pl, b0, b1);
          mma_bf16(acc[2 * jj + 1], pl, b2, b3);
        }
      }
    }
    // the copy overwrites tiles this warp has only read, and those reads have
    // completed (their registers fed the MMAs above): no proxy fence needed
    __syncwarp();
    if (lane == 0 && i + S < n_mine) issue(i + S, s);
  }
  if (timed_out) {
    // drain the copies this warp still has in flight (each wait bounded)
    for (int j = i + 1; j < n_mine && j < i + S; ++j) mbar_wait_bounded(&bars[warp][j % S], (j / S) & 1, p.status);
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- the W warps' states combine into one split per CTA.  The stage
  // buffers are free once every warp is past its last block (a warp that
  // timed out has drained its copies, each wait bounded), so they hold the
  // warps' accumulators: [warp][row][D] fp32.
  __syncthreads();
  float* s_acc = reinterpret_cast<float*>(base);
  static_assert(W * 16 * D * 4 <= W * S * STAGE, "combine buffer fits the stages");
  if (r0ok) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2*>(s_acc + ((size_t)warp * 16 + g) * D + n * 8 + 2 * c) = make_float2(acc[n][0], acc[n][1]);
    if (c == 0) s_wml[warp][g] = make_float2(m0, l0);
  }
  if (r1ok) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2*>(s_acc + ((size_t)warp * 16 + g + 8) * D + n * 8 + 2 * c) = make_float2(acc[n][2], acc[n][3]);
    if (c == 0) s_wml[warp][g + 8] = make_float2(m1, l1);
  }
  __syncthreads();
  const size_t sidx = ((size_t)a * p.hkv + h) * p.n_chunks + chunk;
  {
    constexpr int CPT = D / 8;   // columns per thread: 16 rows x 8 threads (g <= 16 rows used)
    const int r = threadIdx.x >> 3, c0 = (threadIdx.x & 7) * CPT;
    if (nch == 1) {
      // the whole context in this CTA: its combined state is the output (an
      // empty context gives zeros)
      if (r < p.g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w)
          if (s_wml[w][r].y > 0.f) M = fmaxf(M, s_wml[w][r].x);
        float Lc = 0.f, o[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) o[j] = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 ml = s_wml[w][r];
          const float wt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
          Lc += wt * ml.y;
          const float* src = s_acc + ((size_t)w * 16 + r) * D + c0;
#pragma unroll
          for (int j = 0; j < CPT; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            o[j] += wt * x.x; o[j + 1] += wt * x.y; o[j + 2] += wt * x.z; o[j + 3] += wt * x.w;
          }
        }
        const float inv = Lc > 0.f ? 1.f / Lc : 0.f;
        float* dst = p.out + ((size_t)a * p.hq + h * p.g + r) * D + c0;
#pragma unroll
        for (int j = 0; j < CPT; j += 4)
          *reinterpret_cast<float4*>(dst + j) = make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
      }
      return;
    }
    if (r < p.g) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w)
        if (s_wml[w][r].y > 0.f) M = fmaxf(M, s_wml[w][r].x);
      float Lc = 0.f, o[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) o[j] = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float2 ml = s_wml[w][r];
        const float wt = ml.y > 0.f ? fast_exp2(ml.x - M) : 0.f;
        Lc += wt * ml.y;
        const float* src = s_acc + ((size_t)w * 16 + r) * D + c0;
#pragma unroll
        for (int j = 0; j < CPT; j += 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + j);
          o[j] += wt * x.x; o[j + 1] += wt * x.y; o[j + 2] += wt * x.z; o[j + 3] += wt * x.w;
        }
      }
      float* pr = p.part + (sidx * p.g + r) * D + c0;
#pragma unroll
      for (int j = 0; j < CPT; j += 4) __stcg(reinterpret_cast<float4*>(pr + j), make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]));
      if ((threadIdx.x & 7) == 0) __stcg(reinterpret_cast<float2*>(p.part_ml + (sidx * p.g + r) * 2), make_float2(M, Lc));
    }
  }
  if (!arrive_last(p.tickets + a * p.hkv + h, nch, &s_last)) return;
  const size_t s0 = ((size_t)a * p.hkv + h) * p.n_chunks;
  merge_splits<D>(p.part, p.part_ml, s0, nch, p.g, p.out + ((size_t)a * p.hq + h * p.g) * D, sM, sL);
}

template <int D, bool DIFF, bool ROPE, int W>
static kvs_status launch_attn_w(const AttnParams& prm, const kvs_pool* pool, int layer, int grid, cudaStream_t st) {
  auto kern = attn_bf16_kernel<D, DIFF, ROPE, W>;
  constexpr int smem = attn_smem_bytes<D, DIFF, W>();
  if (!smem_limit_once<attn_bf16_kernel<D, DIFF, ROPE, W>>(smem, pool->device))
    return fail(KVS_ERR_CUDA, "decode_attn: cannot raise the shared-memory limit");
  const CUtensorMap& dk = DIFF ? pool->tdk[layer] : pool->tk[layer];
  const CUtensorMap& dv = DIFF ? pool->tdv[layer] : pool->tv[layer];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * W);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm, pool->tk[layer], pool->tv[layer], dk, dv) != cudaSuccess)
    return fail(KVS_ERR_CUDA, "decode_attn: launch failed");
  count_launch();
  return check_launch("decode_attn");
}

template <int D, bool DIFF, bool ROPE>
static kvs_status launch_attn(const AttnParams& prm, const kvs_pool* pool, int layer, int grid, bool wide_cta,
                              cudaStream_t st) {
  if constexpr (attn_wide_cta_ok<D, DIFF>()) {
    if (wide_cta) return launch_attn_w<D, DIFF, ROPE, 8>(prm, pool, layer, grid, st);
  }
  return launch_attn_w<D, DIFF, ROPE, kAttnWarps>(prm, pool, layer, grid, st);
}

}  // namespace kvs

using namespace kvs;

// Small calls with a query group <= 8 run on the 16-row kernel alone, unless
// a test asks for the planned path.
static bool use_small_path(const kvs_pool* pool, int n_seq, int max_blocks, int g) {
  return small_call(n_seq, pool->desc.num_kv_heads, max_blocks, g) && !(pool->test_flags & KVS_TEST_TOKEN_MAJOR);
}

// Host checks shared by the decode-attention entry points.
static kvs_status attn_check(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                             const int32_t* block_table_dev, int32_t max_blocks, const int32_t* seq_len_dev,
                             int32_t n_seq, const int32_t* diff_table_dev, const int32_t* rope_off_dev,
                             const kvs_seg_rope* rope_segs_dev, float theta, const float* out_dev, const void* ws,
                             size_t ws_bytes, bool need_q) {
  if (!pool) return fail(KVS_ERR_INVALID_ARG, "decode_attn: null pool");
  const kvs_pool_desc& d = pool->desc;
  if (d.dtype != KVS_DTYPE_BF16) return fail(KVS_ERR_INVALID_ARG, "decode_attn: pool is not bf16 (use kvs_decode_attn_q4)");
  if (need_q && (layer < 0 || layer >= d.num_layers)) return fail(KVS_ERR_INVALID_ARG, "decode_attn: layer out of range");
  if (n_seq < 0 || n_seq > d.max_seqs) return fail(KVS_ERR_CAPACITY, "decode_attn: n_seq exceeds the pool's max_seqs");
  if (n_seq == 0) return KVS_OK;
  if (!block_table_dev || !seq_len_dev || !ws || (need_q && (!q_dev || !out_dev)))
    return fail(KVS_ERR_INVALID_ARG, "decode_attn: null pointer");
  if ((need_q && (!aligned16(q_dev) || !aligned16(out_dev))) || !aligned16(ws))
    return fail(KVS_ERR_INVALID_ARG, "decode_attn: q, out and ws must be 16-byte aligned");
  if (max_blocks < 1) return fail(KVS_ERR_INVALID_ARG, "decode_attn: max_blocks must be >= 1");
  if (n_q_heads < 1 || n_q_heads % d.num_kv_heads) return fail(KVS_ERR_INVALID_ARG, "decode_attn: n_q_heads must be a multiple of num_kv_heads");
  if (n_q_heads / d.num_kv_heads > 16) return fail(KVS_ERR_UNSUPPORTED, "decode_attn: more than 16 query heads per KV head");
  if (diff_table_dev && d.diff_capacity_blocks == 0) return fail(KVS_ERR_INVALID_ARG, "decode_attn: diff table given but the pool has no diff slabs");
  if ((rope_off_dev == nullptr) != (rope_segs_dev == nullptr)) return fail(KVS_ERR_INVALID_ARG, "decode_attn: rope_off and rope_segs go together");
  if (need_q && rope_off_dev && !(theta > 0.f)) return fail(KVS_ERR_INVALID_ARG, "decode_attn: theta must be positive");
  size_t need = 0;
  kvs_workspace_size(pool, KVS_OP_DECODE_ATTN, n_seq, max_blocks, n_q_heads, &need);
  if (ws_bytes < need) return fail(KVS_ERR_CAPACITY, "decode_attn: workspace too small");
  return KVS_OK;
}

extern "C" kvs_status kvs_decode_plan(kvs_pool* pool, int32_t n_q_heads, const int32_t* block_table_dev,
                                      int32_t max_blocks, const int32_t* seq_len_dev, int32_t n_seq,
                                      const int32_t* diff_table_dev, const int32_t* rope_off_dev,
                                      const kvs_seg_rope* rope_segs_dev, void* ws, size_t ws_bytes,
                                      cudaStream_t stream) {
  kvs_status st = attn_check(pool, 0, nullptr, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq,
                             diff_table_dev, rope_off_dev, rope_segs_dev, 1.f, nullptr, ws, ws_bytes, false);
  if (st != KVS_OK || n_seq == 0) return st;
  // the 16-row kernel (groups of 9-16, and small calls) needs no plan
  if (n_q_heads / pool->desc.num_kv_heads > kTmMaxGroup ||
      use_small_path(pool, n_seq, max_blocks, n_q_heads / pool->desc.num_kv_heads))
    return KVS_OK;
  return decode_plan_token_major(pool, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq, diff_table_dev,
                                 rope_off_dev, rope_segs_dev, ws, stream);
}

static kvs_status attn_launch(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                              const int32_t* block_table_dev, int32_t max_blocks, const int32_t* seq_len_dev,
                              int32_t n_seq, const int32_t* diff_table_dev, const int32_t* rope_off_dev,
                              const kvs_seg_rope* rope_segs_dev, float theta, float scale, float* out_dev, void* ws,
                              cudaStream_t stream) {
  const kvs_pool_desc& d = pool->desc;
  const int g = n_q_heads / d.num_kv_heads;
  if (g <= kTmMaxGroup && !use_small_path(pool, n_seq, max_blocks, g))
    return decode_attn_token_major(pool, layer, q_dev, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq,
                                   diff_table_dev, rope_off_dev, rope_segs_dev, theta, scale, out_dev, ws, stream);
  AttnPlan plan = attn_plan(pool, n_seq, max_blocks);
  const bool diff = diff_table_dev != nullptr;
  bool wide_cta = false;
  if (g <= kTmMaxGroup && max_blocks <= kSmallOneChunk) {
    // a small call with short contexts: one CTA per (sequence, KV head)
    // writes its output directly, with no split and no merge (the 4-agent,
    // 24-block layer: 11.7-12.1 us against 12.9 us in three chunks), on
    // eight warps where their rings fit (all but head_dim 128 with diffs)
    wide_cta = !(d.head_dim == 128 && diff);
    const int w = wide_cta ? 8 : kAttnWarps;
    plan.bpc = (max_blocks + w - 1) / w * w;
    plan.n_chunks = 1;
  }
  const long long grid = (long long)n_seq * d.num_kv_heads * plan.n_chunks;
  if (grid > 0x7fffffffll) return fail(KVS_ERR_CAPACITY, "decode_attn: grid too large");
  AttnParams prm{};
  prm.q = static_cast<const uint16_t*>(q_dev);
  prm.block_table = block_table_dev;
  prm.seq_len = seq_len_dev;
  prm.diff_table = diff_table_dev;
  prm.rope_off = rope_off_dev;
  prm.rope_segs = reinterpret_cast<const int4*>(rope_segs_dev);
  prm.out = out_dev;
  const size_t splits = (size_t)n_seq * d.num_kv_heads * plan.n_chunks * kAttnWarps;
  prm.part = static_cast<float*>(ws);
  prm.part_ml = prm.part + splits * g * d.head_dim;
  prm.tickets = pool->tickets;
  prm.status = pool->status;
  prm.max_blocks = max_blocks;
  prm.n_seq = n_seq;
  prm.hkv = d.num_kv_heads;
  prm.g = g;
  prm.hq = n_q_heads;
  prm.bpc = plan.bpc;
  prm.n_chunks = plan.n_chunks;
  prm.capacity = d.capacity_blocks;
  prm.diff_capacity = d.diff_capacity_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  const bool rope = rope_off_dev != nullptr;
  if (rope) rope_split_host(theta, d.head_dim, prm.rs.c);
  const int gr = static_cast<int>(grid);
  if (d.head_dim == 128) {
    if (diff) return rope ? launch_attn<128, true, true>(prm, pool, layer, gr, wide_cta, stream)
                          : launch_attn<128, true, false>(prm, pool, layer, gr, wide_cta, stream);
    return rope ? launch_attn<128, false, true>(prm, pool, layer, gr, wide_cta, stream)
                : launch_attn<128, false, false>(prm, pool, layer, gr, wide_cta, stream);
  }
  if (diff) return rope ? launch_attn<64, true, true>(prm, pool, layer, gr, wide_cta, stream)
                        : launch_attn<64, true, false>(prm, pool, layer, gr, wide_cta, stream);
  return rope ? launch_attn<64, false, true>(prm, pool, layer, gr, wide_cta, stream)
              : launch_attn<64, false, false>(prm, pool, layer, gr, wide_cta, stream);
}

extern "C" kvs_status kvs_decode_attn_planned(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                                              const int32_t* block_table_dev, int32_t max_blocks,
                                              const int32_t* seq_len_dev, int32_t n_seq,
                                              const int32_t* diff_table_dev, const int32_t* rope_off_dev,
                                              const kvs_seg_rope* rope_segs_dev, float theta, float scale,
                                              float* out_dev, void* ws, size_t ws_bytes, cudaStream_t stream) {
  kvs_status st = attn_check(pool, layer, q_dev, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq,
                             diff_table_dev, rope_off_dev, rope_segs_dev, theta, out_dev, ws, ws_bytes, true);
  if (st != KVS_OK || n_seq == 0) return st;
  return attn_launch(pool, layer, q_dev, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq, diff_table_dev,
                     rope_off_dev, rope_segs_dev, theta, scale, out_dev, ws, stream);
}

extern "C" kvs_status kvs_decode_attn(kvs_pool* pool, int32_t layer, const void* q_dev, int32_t n_q_heads,
                                      const int32_t* block_table_dev, int32_t max_blocks,
                                      const int32_t* seq_len_dev, int32_t n_seq, const int32_t* diff_table_dev,
                                      const int32_t* rope_off_dev, const kvs_seg_rope* rope_segs_dev,
                                      float theta, float scale, float* out_dev, void* ws, size_t ws_bytes,
                                      cudaStream_t stream) {
  kvs_status st = attn_check(pool, layer, q_dev, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq,
                             diff_table_dev, rope_off_dev, rope_segs_dev, theta, out_dev, ws, ws_bytes, true);
  if (st != KVS_OK || n_seq == 0) return st;
  st = kvs_decode_plan(pool, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq, diff_table_dev,
                       rope_off_dev, rope_segs_dev, ws, ws_bytes, stream);
  if (st != KVS_OK) return st;
  return attn_launch(pool, layer, q_dev, n_q_heads, block_table_dev, max_blocks, seq_len_dev, n_seq, diff_table_dev,
                     rope_off_dev, rope_segs_dev, theta, scale, out_dev, ws, stream);
}
