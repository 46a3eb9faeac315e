// Diagnostic (not part of libsparda): the throughput of back-to-back tcgen05.mma of
// kind::f16 (bf16 x bf16 -> fp32) issued by one thread, one CTA per SM, for the operand
// shapes and sources the prefill attention uses. Operands sit in shared memory (zeros) or, for
// A, in tensor memory. Prints SM clocks per MMA and flop per clock per SM.
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
template <int N, bool kATmem, bool kBMnMajor>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel() {
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

template <int N, bool kATmem, bool kBMnMajor>
void run(const char* name, int ctas) {
  auto k = mma_rate_kernel<N, kATmem, kBMnMajor>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  k<<<ctas, 128, kSmem>>>();
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
  }
  return 0;
}
