// Per-CTA timeline records for the decode step's two per-layer launches, compiled in only with
// -DSPARDA_TIMELINE (block_sparse_attention_forecast_gb300/timeline.py builds that variant as a
// separate library). Each record holds the launch it belongs to (a host-side count of the
// instrumented launches, fixed at capture time inside a CUDA graph), the CTA's role and block
// index, and %globaltimer (ns) at its entry, after its wait for the previous launch (0 when it
// does not wait) and at its exit. The product build compiles every macro below to nothing.
#pragma once

#include <stdint.h>

namespace sparda {

enum TimelineRole : uint32_t {
  kTlAttention = 1, kTlSelection = 2, kTlProjection = 3, kTlTopk = 4, kTlAppend = 5,
};

struct TimelineRec {
  unsigned long long t_entry, t_release, t_exit;
  uint32_t launch, role_cta;            // role << 24 | block index
};
constexpr int kTimelineMax = 1 << 16;
// The record store: a count, then the records (the library's one instance lives in api.cu; its
// device address reaches the kernels through their launch arguments).
struct TimelineBuf {
  unsigned int n;
  unsigned int pad[3];
  TimelineRec rec[kTimelineMax];
};

#ifdef SPARDA_TIMELINE
__device__ __forceinline__ unsigned long long tl_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tl_record(void* buf, uint32_t launch, uint32_t role, unsigned long long t0,
                                          unsigned long long t_rel) {
  __syncthreads();
  TimelineBuf* b = static_cast<TimelineBuf*>(buf);
  if (threadIdx.x == 0 && b) {
    const unsigned int i = atomicAdd(&b->n, 1u);
    if (i < kTimelineMax) b->rec[i] = TimelineRec{t0, t_rel, tl_now(), launch, (role << 24) | blockIdx.x};
  }
}
#define SPARDA_TL_ENTRY() const unsigned long long tl_t0_ = tl_now()
#define SPARDA_TL_RELEASE(var) var = tl_now()
#define SPARDA_TL_EXIT(buf, launch, role, t_rel) tl_record((buf), (launch), (role), tl_t0_, (t_rel))
#else
#define SPARDA_TL_ENTRY() \
  do {                    \
  } while (0)
#define SPARDA_TL_RELEASE(var) \
  do {                         \
  } while (0)
#define SPARDA_TL_EXIT(buf, launch, role, t_rel) \
  do {                                           \
  } while (0)
#endif

// Host side: the next launch's number (counts instrumented launches) and the device address of
// the record store; 0 and nullptr in the product build.
uint32_t timeline_next_launch();
void* timeline_buffer();

}  // namespace sparda
