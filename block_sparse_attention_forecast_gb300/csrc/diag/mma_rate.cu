// Diagnostic (not part of libsparda): the throughput of back-to-back tcgen05.mma of
// kind::f16 (bf16 x bf16 -> fp32) issued by one thread, one CTA per SM, for the operand
// shapes and sources the prefill attention uses. Operands sit in shared memory (zeros) or, for
// A, in tensor memory. Each case runs alone or beside eight other warps of the CTA (two per SM
// sub-partition, as the prefill attention's softmax warps) that, until the MMAs are done, run
// one of: chains of ex2.approx (MUFU-bound), independent float32 FMA chains (issue-bound), a
// softmax-like mix per pair of values (two FMAs, two ex2.approx, two adds, one bf16 pack), or
// tensor-memory loads. Prints SM clocks per MMA and flop per clock per SM.
//
//   python -m block_sparse_attention_forecast_gb300.mma_rate
#include <cstdint>
#include <cstdio>

#include "../tc05.cuh"

using namespace sparda;

namespace {

__device__ unsigned long long g_clk[1024][2];

constexpr int kReps = 64;                    // 8 MMAs (K = 128) per repetition
constexpr int kSmem = 1024 + 1024 + 32768 + 65536;

// A: 128 rows x 128 dims, K-major with the 128-byte swizzle (two 64-dim halves of 16 KiB).
// B K-major: up to 256 rows x 128 dims (two halves of 32 KiB); B M/N-major: 64-column chunks
// of 128 K rows (16 KiB each, 16 KiB apart).
// The side warps' work (warps 2-9 of the CTA).
enum Side { kAlone = 0, kExp2 = 1, kFma = 2, kSoftmaxMix = 3, kTmemLoad = 4 };

template <int kSide>
__device__ __forceinline__ void side_work(uint32_t tmem, int warp, int tid, volatile uint32_t* stop, float* sink) {
  float x0 = tid * 1e-3f, x1 = x0 + 0.1f, x2 = x0 + 0.2f, x3 = x0 + 0.3f;
  uint32_t pk = 0;
  for (int it = 0; it < (1 << 20); ++it) {            // bounded; the issuer sets *stop when done
    if ((it & 63) == 0 && __shfl_sync(0xffffffffu, (int)*stop, 0)) break;
    if (kSide == kExp2) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x0));
        asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x1));
        asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x2));
        asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(x3));
        x0 = fmaf(x0, -0.5f, 0.1f);
        x1 = fmaf(x1, -0.5f, 0.1f);
        x2 = fmaf(x2, -0.5f, 0.1f);
        x3 = fmaf(x3, -0.5f, 0.1f);
      }
    } else if (kSide == kFma) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x0 = fmaf(x0, 0.999f, 0.1f);
        x1 = fmaf(x1, 0.999f, 0.1f);
        x2 = fmaf(x2, 0.999f, 0.1f);
        x3 = fmaf(x3, 0.999f, 0.1f);
      }
    } else if (kSide == kSoftmaxMix) {
      float p[16];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float a0 = fmaf(x0 + u, 0.07f, -x1), a1 = fmaf(x0 + u, 0.05f, -x2);
        asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(p[2 * u]) : "f"(a0));
        asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(p[2 * u + 1]) : "f"(a1));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        x3 += p[2 * u] + p[2 * u + 1];
        uint32_t w;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p[2 * u + 1]), "f"(p[2 * u]));
        pk ^= w;
      }
      x1 = x1 * 0.5f + (float)(pk & 1u);
    } else if (kSide == kTmemLoad) {
      float v[32];
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;   // this warp's lane quarter
      tc05::ld32(tmem + lane_off + 384, v);                          // columns the MMAs do not use
      tc05::wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) x0 += v[e];
    }
  }
  if (x0 + x1 + x2 + x3 == 12345.f) sink[tid] = x0;   // keeps the work
}

template <int N, bool kATmem, bool kBMnMajor, int kSide>
__global__ void __launch_bounds__(320, 1) mma_rate_kernel(float* sink) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tbase = reinterpret_cast<uint32_t*>(smem + 64);
  uint8_t* A = smem + 1024;
  uint8_t* B = A + 32768;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < (32768 + 65536) / 16; i += blockDim.x) reinterpret_cast<uint4*>(A)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc05::alloc(tbase, 512);
    tc05::relinquish();
  }
  fence_proxy_async_shared();
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = *tbase;
  volatile uint32_t* stop = reinterpret_cast<volatile uint32_t*>(smem + 128);
  if (tid == 0) *stop = 0;
  __syncthreads();
  if (warp >= 2 && kSide != kAlone) side_work<kSide>(tmem, warp, tid, stop, sink);
  if (tid == 0) {
    const uint32_t id = tc05::idesc_bf16(128, N, 0, kBMnMajor ? 1 : 0);
    const uint32_t aa = smem_addr(A), bb = smem_addr(B);
    const unsigned long long t0 = clock64();
    for (int r = 0; r < kReps; ++r) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t db = kBMnMajor ? tc05::smem_desc(bb + kk * 2048, 16384, 1024)
                                      : tc05::smem_desc(bb + (kk >> 2) * 32768 + (kk & 3) * 32, 16, 1024);
        if (kATmem) {
          tc05::mma_bf16_ts(tmem + 256, tmem + 8 * kk, db, id, 1u);
        } else {
          const uint64_t da = tc05::smem_desc(aa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          tc05::mma_bf16_ss(tmem + 256, da, db, id, 1u);
        }
      }
    }
    tc05::commit(bar);
    uint32_t done = 0;
    for (int i = 0; i < (1 << 24) && !done; ++i)     // bounded wait for the last MMA
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(done)
                   : "r"(smem_addr(bar))
                   : "memory");
    *stop = 1;
    if (blockIdx.x < 1024) {
      g_clk[blockIdx.x][0] = clock64() - t0;
      g_clk[blockIdx.x][1] = done;
    }
  }
  tc05::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc05::fence_after();
    tc05::dealloc(tmem, 512);
  }
}

template <int N, bool kATmem, bool kBMnMajor, int kSide = kAlone>
void run(const char* name, int ctas) {
  auto k = mma_rate_kernel<N, kATmem, kBMnMajor, kSide>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  static float* sink = nullptr;
  if (!sink && cudaMalloc(&sink, 320 * sizeof(float)) != cudaSuccess) return;
  k<<<ctas, 320, kSmem>>>(sink);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    std::printf("%s: %s\n", name, cudaGetErrorString(e));
    return;
  }
  static unsigned long long h[1024][2];
  cudaMemcpyFromSymbol(h, g_clk, sizeof(h));
  double clk = 0.0;
  int done = 0;
  for (int i = 0; i < ctas; ++i) {
    clk += (double)h[i][0];
    done += h[i][1] ? 1 : 0;
  }
  const double per = clk / ctas / (kReps * 8.0);
  std::printf("%-34s CTAs %3d  %6.1f clk/MMA  %6.0f flop/clk/SM%s\n", name, ctas, per, 2.0 * 128 * N * 16 / per,
              done == ctas ? "" : "  (a wait ran out)");
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  if (sms <= 0 || sms > 1024) sms = 1;
  for (int ctas : {1, sms}) {
    run<64, false, false>("M128 N64  K16, A smem, B K-major", ctas);
    run<128, false, false>("M128 N128 K16, A smem, B K-major", ctas);
    run<256, false, false>("M128 N256 K16, A smem, B K-major", ctas);
    run<128, false, true>("M128 N128 K16, A smem, B MN-major", ctas);
    run<128, true, true>("M128 N128 K16, A tmem, B MN-major", ctas);
    run<128, false, false, kExp2>("  N128 A smem, beside ex2 warps", ctas);
    run<128, false, false, kFma>("  N128 A smem, beside FMA warps", ctas);
    run<128, false, false, kSoftmaxMix>("  N128 A smem, beside softmax mix", ctas);
    run<128, false, false, kTmemLoad>("  N128 A smem, beside TMEM loads", ctas);
    run<128, true, true, kSoftmaxMix>("  N128 A tmem, beside softmax mix", ctas);
  }
  return 0;
}
