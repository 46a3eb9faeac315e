// sparda_forecast_select_static: the Forecast selector without a caller-provided workspace.
//
// Some callers cannot allocate device memory at all: a plugin inside a host engine that hands
// it only the input and output tensors and keeps every allocation to itself, or a serving
// loop that forbids any allocation once it has started. For them the selector's scratch (the
// per-group arrival counters and the block scores) lives in a fixed array in this library's
// own device memory, reserved once when the library is loaded on a device and kept until the
// process exits. Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace sparda;

namespace {

constexpr size_t kCounterBytes = (size_t)SPARDA_STATIC_MAX_GROUPS * sizeof(unsigned);

// Counters first (SPARDA_STATIC_MAX_GROUPS of them), then block scores. Every call shares
// this array; it keeps the contents of the last call.
static __device__ __align__(256) unsigned char g_select_scratch[SPARDA_STATIC_SCRATCH_BYTES];

// Device address of g_select_scratch on each device, looked up on the first call made with
// that device current. In host code the array's name is only a host-side stand-in.
void* scratch_ptr() {
  static void* ptrs[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int32_t sparda_forecast_select_static(const sparda_shape* s, const void* ck,
                                                 const void* forecast, const int32_t* seq_len,
                                                 int32_t batch, int32_t* idx, int32_t* cnt,
                                                 void* stream) {
  const int32_t shape_ok = sparda_check_shape(s);
  if (shape_ok != SPARDA_OK) return shape_ok;
  if (batch < 1 || batch > s->max_batch) return SPARDA_ERR_INVALID_ARG;
  if (!ck || !forecast || !seq_len || !idx || !cnt) return SPARDA_ERR_INVALID_ARG;
  const uintptr_t m16 = 15, m4 = 3;
  if ((reinterpret_cast<uintptr_t>(ck) & m16) || (reinterpret_cast<uintptr_t>(forecast) & m16) ||
      (reinterpret_cast<uintptr_t>(idx) & m4) || (reinterpret_cast<uintptr_t>(cnt) & m4) ||
      (reinterpret_cast<uintptr_t>(seq_len) & m4))
    return SPARDA_ERR_MISALIGNED;
  const size_t groups = (size_t)batch * s->n_groups;
  const int nb_cap = s->max_ctx / kBlock;
  if (groups > (size_t)SPARDA_STATIC_MAX_GROUPS ||
      kCounterBytes + groups * nb_cap * sizeof(float) > (size_t)SPARDA_STATIC_SCRATCH_BYTES)
    return SPARDA_ERR_STATIC_SCRATCH_LIMIT;

  unsigned char* scratch = static_cast<unsigned char*>(scratch_ptr());
  if (!scratch) return SPARDA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The counters must start at zero; the kernel leaves them at zero, but a fresh clear keeps
  // this call independent of whatever an earlier call left behind.
  if (cudaMemsetAsync(scratch, 0, groups * sizeof(unsigned), st) != cudaSuccess) return SPARDA_ERR_CUDA;
  int* err = dev_error_word();          // the library's device error word
  if (!err) return SPARDA_ERR_CUDA;
  SelectArgs a{static_cast<const __nv_bfloat16*>(ck), static_cast<const __nv_bfloat16*>(forecast),
               seq_len, idx, cnt, reinterpret_cast<float*>(scratch + kCounterBytes),
               reinterpret_cast<unsigned*>(scratch), err, s->n_groups, num_windows(s->max_ctx),
               s->max_ctx, nb_cap, s->topk, select_chunk_blocks(nb_cap, (int)groups), 0};
  launch_forecast_select(a, (int)groups, st);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SPARDA_OK : SPARDA_ERR_CUDA;
}
