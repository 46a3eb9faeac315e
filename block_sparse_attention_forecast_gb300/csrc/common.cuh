// Device-side helpers shared by the kernels of libsparda: fixed sizes, inline-PTX wrappers
// for mbarriers, bulk and tiled TMA copies, ldmatrix and warp-level bf16 MMA, and the
// bounded wait every kernel uses on a copy's completion.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sparda.h"

namespace sparda {

constexpr int kHeadDim = 128;        // d
constexpr int kHeads = 16;           // query heads per KV group
constexpr int kBlock = 64;           // tokens per KV block
constexpr int kWinKernel = 32;       // tokens per compression window
constexpr int kWinStride = 16;       // stride of compression windows
constexpr int kWinPerBlock = kBlock / kWinStride;   // 4
constexpr int kMaxTopk = 62;
constexpr int kMaxCtx = 262144;
constexpr int kRowBytes = kHeadDim * 2;             // one bf16 key/value row: 256 B
constexpr int kBlockBytes = kBlock * kRowBytes;     // one 64-token K (or V) block: 16 KiB
constexpr int kHotSlots = 3;

// Every wait on an mbarrier polls with try_wait and a suspend-time hint: a waiting thread
// sleeps (issuing nothing) until the phase completes or the hint elapses. At most kWaitPolls
// polls of at most kWaitHintNs each bound a wait to about 2.6 s.
constexpr uint32_t kWaitHintNs = 10000;
constexpr uint32_t kWaitPolls = 1u << 18;

__host__ __device__ constexpr int num_windows(int n_tokens) {
  return n_tokens < kWinKernel ? 0 : (n_tokens - kWinKernel) / kWinStride + 1;
}

// ------------------------------------------------------------------ shared-memory PTX
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes initialised mbarriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete, at most kWaitPolls polls. On
// timeout ORs SPARDA_DEV_WAIT_TIMEOUT into *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(err, SPARDA_DEV_WAIT_TIMEOUT);
  return false;
}

// ------------------------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster; release / acquire at cluster scope, so that the
// shared- and global-memory writes before it are visible to the cluster's reads after it. The
// barrier instructions are warp-aligned: the warp reconverges first.
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory data of CTA `rank` of the cluster at the same offset as the local `p`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
  return remote;
}
__device__ __forceinline__ float ld_cluster_f(const void* p, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_f2(const void* p, uint32_t rank) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_f(void* p, uint32_t rank, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr(p, rank)), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f4(void* p, uint32_t rank, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr(p, rank)), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(const void* p, uint32_t rank) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr(p, rank))
               : "memory");
  return v;
}

// Untiled bulk copy global -> this CTA's shared memory; completes `bytes` on the mbarrier.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Tiled 2-D TMA load of the box at (x = column, y = row) of `map` into shared memory.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ warp MMA (bf16)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, float32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ bf16 helpers
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two floats -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// float64 -> bf16 rounded to nearest even, without double rounding: first round to float32
// with round-to-odd (truncate, then set the last bit when inexact), then round to bf16
// (Boldo & Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms using
// rounding to odd", IEEE TC 2008: rounding to odd with at least two extra bits makes the
// second rounding correct).
__device__ __forceinline__ __nv_bfloat16 f64_to_bf16_rn(double x) {
  float t = __double2float_rz(x);
  if (static_cast<double>(t) != x) t = __uint_as_float(__float_as_uint(t) | 1u);
  return __float2bfloat16_rn(t);
}

// Float -> unsigned key whose unsigned order is the float order (NaN-free inputs).
__device__ __forceinline__ uint32_t ordered_key(float x) {
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start while the previous kernel in its stream still runs; grid_dep_wait() blocks
// until that kernel has completed and its writes are visible. grid_dep_launch() lets the
// next such kernel start launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Hot slot of block j (>= 0) of an offloaded layer.
__device__ __forceinline__ int hot_slot(int j) { return j == 0 ? 0 : 1 + (j & 1); }

}  // namespace sparda
