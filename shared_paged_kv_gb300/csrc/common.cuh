// Device helpers shared by the libkvs kernels (sm_103a): status reporting,
// mbarrier + TMA (cp.async.bulk[.tensor]) wrappers, ldmatrix / mma.sync
// wrappers, fast exp2, and the RoPE angle evaluation.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>

#include "kvs.h"

namespace kvs {

// ---------------------------------------------------------------- status ---
__device__ __forceinline__ void set_err(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// -------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after ~2^31 cycles (about a second at GB300 clocks),
// records KVS_DEVERR_WAIT_TIMEOUT and returns false.  Never spins forever.
// Wait for a phase with a short limit and no error report: used after a
// timed-out wait to let the copies still in flight land before the CTA's
// shared memory is released.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < (1ll << 24)) {
  }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > (1ll << 31)) {
      set_err(status, KVS_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------- TMA ---
// Fetch a tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache, so that the first copy through it does not wait for it.
// It reads only the kernel's own parameters, so it may run before
// griddepcontrol.wait.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// The same copy with an L2 cache policy (createpolicy), e.g. evict-first for
// data that is read once, so that it does not push out data read again.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// A store with an L2 cache policy (e.g. evict-last for data that another
// kernel reads soon, so that streaming reads do not push it out first).
__device__ __forceinline__ void st_hint_f32(float* p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint_v2f32(float* p, float2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(p), "f"(v.x), "f"(v.y), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint_v4u32(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of a 16-byte-chunked tile under the TMA swizzle modes (tile base
// aligned to 1024 bytes).  128B: bits [4,7) ^= bits [7,10).  64B: bits [4,6)
// ^= bits [7,9).
__device__ __forceinline__ uint32_t swz128(uint32_t o) { return o ^ (((o >> 7) & 7u) << 4); }
__device__ __forceinline__ uint32_t swz64(uint32_t o) { return o ^ (((o >> 7) & 3u) << 4); }

// A bf16 KV tile of one 16-token block and one KV head, head_dim D, is loaded
// by one 3-D TMA box as D/64 panels of 16 rows x 64 elements (128-byte rows,
// 128-byte swizzle) stacked as [D/64][16][64].  Consecutive tokens are
// consecutive 128-byte rows, so the swizzle spreads any 8 consecutive tokens
// over all eight 16-byte bank groups (ldmatrix without conflicts).
template <int D>
__device__ __forceinline__ void tma_load_kv_tile(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  tma_load_3d(dst, map, 0, row, 0, bar);   // all D/64 halves of the tile in one copy
}

template <int D>
__device__ __forceinline__ void tma_load_kv_tile_hint(void* dst, const CUtensorMap* map, int row, uint64_t* bar,
                                                      uint64_t policy) {
  tma_load_3d_hint(dst, map, 0, row, 0, bar, policy);
}

template <int D>
__device__ __forceinline__ uint32_t kv_tile_off(int t, int col) {
  return swz128(((uint32_t)((col >> 6) * 16 + t) << 7) + ((uint32_t)(col & 63) << 1));
}

// ------------------------------------------------------- tensor-core mma ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (x, y) -> hi = bf16x2(x, y) and lo = bf16x2 of the rounding remainders, so
// hi + lo carries x and y to ~16 significant bits through a bf16 MMA.
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x, y);
  lo = pack_bf16(x - bf16_lo(hi), y - bf16_hi(hi));
}

// ------------------------------------------------------------ RoPE angle ---
// cos / sin of (delta * w_i) for an integer position shift |delta| < 2^18.
// Argument reduction follows Cody and Waite: the host splits f_i = w_i/(2*pi)
// into c0 + c1 + c2 + c3 where c0, c1, c2 hold 6 fraction bits each at fixed
// positions (2^-1..2^-6, 2^-7..2^-12, 2^-13..2^-18), so delta*c0..c2 are exact
// in float32 and their fractional parts are exact; delta*c3 < 1 carries only
// float32 rounding.  The reduced angle lies in [-pi, pi], where the hardware
// __sincosf is accurate to about 4e-7 absolute.
// Kernels of a chain on one stream (the dedup steps, the plan steps) are
// programmatic dependent launches: each is scheduled while the one before it
// runs, and its first statement (pdl_enter) waits for that kernel to complete
// with its writes visible, then lets the next kernel of the chain be
// scheduled.  A kernel launched without the attribute passes the wait at once.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct RopeSplit {
  float c[4][64];   // [piece][frequency index], up to head_dim 128
};

// c points at a copy of RopeSplit::c in shared memory (lanes index it with
// different i; indexed loads from the kernel-parameter bank would serialise).
__device__ __forceinline__ void rope_cos_sin(const float* c, int i, int delta, float& cs, float& sn) {
  const float d = static_cast<float>(delta);
  float t0 = d * c[i];
  float t1 = d * c[64 + i];
  float t2 = d * c[128 + i];
  float turns = (t0 - floorf(t0)) + (t1 - floorf(t1)) + (t2 - floorf(t2)) + d * c[192 + i];
  turns -= rintf(turns);
  __sincosf(6.28318530717958647692f * turns, &sn, &cs);
}


// Exclusive prefix sum of x over the CTA (blockDim.x a multiple of 32, at
// most 1024 threads); total receives the CTA-wide sum.  warp_sums needs one
// int per warp.  Every thread of the CTA must call it.
__device__ __forceinline__ int block_exclusive_scan(int x, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int res = incl - x + (warp ? warp_sums[warp - 1] : 0);
  total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return res;
}

}  // namespace kvs
