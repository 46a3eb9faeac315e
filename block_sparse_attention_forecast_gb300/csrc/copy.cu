// A device-side copy between two buffers the device can address: device memory, or pinned
// host memory mapped into the device's address space (unified virtual addressing). It moves
// a step's first inputs in from the host and its last outputs out to it on the compute
// stream itself: a DMA copy costs tens of microseconds from submission to completion on this
// path, a few CTAs of 16-byte loads and stores only the link's round trip.
//
// Every thread keeps kCopyInFlight 16-byte loads in flight (non-caching: the source is read
// once) before it stores them; the CTAs walk the buffer with a grid stride.
#include "common.cuh"
#include "kernels.h"

namespace sparda {

constexpr int kCopyThreads = 256;
constexpr int kCopyInFlight = 4;

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(uint4* dst, const uint4* src, size_t n16) {
  const size_t step = (size_t)gridDim.x * kCopyThreads * kCopyInFlight;
  for (size_t base = (size_t)blockIdx.x * kCopyThreads * kCopyInFlight + threadIdx.x; base < n16; base += step) {
    uint4 r[kCopyInFlight];
#pragma unroll
    for (int u = 0; u < kCopyInFlight; ++u) {
      const size_t i = base + (size_t)u * kCopyThreads;
      if (i < n16) r[u] = ld_stream16(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyInFlight; ++u) {
      const size_t i = base + (size_t)u * kCopyThreads;
      if (i < n16) dst[i] = r[u];
    }
  }
}

int sm_count();

// The stream-ordered read of the device error word: one thread copies it out and, when asked,
// resets it in the same atomic step, so that a bit set by a kernel running elsewhere on the
// device is either reported now or kept for the next read.
__global__ void device_status_kernel(int* err, int32_t* out, int clear) {
  *out = clear ? atomicExch(err, 0) : atomicOr(err, 0);
}

void launch_device_status(int* err, int32_t* out, bool clear, cudaStream_t s) {
  device_status_kernel<<<1, 1, 0, s>>>(err, out, clear ? 1 : 0);
}

void launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  const size_t per_cta = (size_t)kCopyThreads * kCopyInFlight;
  size_t grid = (n16 + per_cta - 1) / per_cta;
  const size_t cap = (size_t)sm_count();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  copy16_kernel<<<(unsigned)grid, kCopyThreads, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
}

}  // namespace sparda
