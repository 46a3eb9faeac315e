// Launches of the standalone Forecast selector: the selector kernel, whose per-CTA work is
// sel_cta (select_body.cuh, shared with the fused attend-and-select kernel, fused.cu); the
// scores-only kernel (queue-fed when it can be); and the top-k behind it.
#include "select_body.cuh"

namespace sparda {

size_t smem_select_bytes(int) { return kSelSmem; }
int select_chunk_blocks(int, int) { return kSubBlocks; }

__global__ void __launch_bounds__(kSelThreads, 1) forecast_select_kernel(const SelectArgs a) {
  sel_cta(a, blockIdx.x, gridDim.x);
}

// The selection's block scores without the top-k, on every SM: sub-chunks handed out from the
// workspace's queue when the forecasts of all (sequence, group)s fit beside the ring, fixed
// ranges otherwise.
constexpr int kScoreSmem = 256 + kSelStages * kSelStageBytes + kSelDynMaxGroups * kHeadDim * 2;
static_assert(kScoreSmem <= 227 * 1024, "the queue-fed selection's ring and forecast table fit");

__global__ void __launch_bounds__(kSelThreads, 1) forecast_score_kernel(const SelectArgs a) {
  if (a.queue)
    sel_cta_dyn(a, blockIdx.x, gridDim.x);
  else
    sel_cta(a, blockIdx.x, gridDim.x);
}

static int sel_sm_count() {
  static int n[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!n[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 152;
  }
  return n[dev];
}

void launch_forecast_select(const SelectArgs& a, int bg_count, cudaStream_t s) {
  cudaFuncSetAttribute(forecast_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmem);
  SelectArgs b = a;
  b.n_units = bg_count * a.nb_cap;
  const int by_work = (b.n_units + kSubBlocks - 1) / kSubBlocks;   // >= one sub-chunk each
  const int grid = by_work < sel_sm_count() ? by_work : sel_sm_count();
  // Programmatic serialization: the producer starts streaming compressed keys while the
  // projection that writes the forecast still runs; consumers wait for it (grid_dep_wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = kSelSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, forecast_select_kernel, b);
}

// The top-k of block scores a scoring launch left in the workspace: one CTA per (sequence,
// group), launched behind that scoring launch (programmatic dependent launch).
__global__ void __launch_bounds__(kTopkThreads) select_topk_kernel(const SelectArgs a) {
  __shared__ TopkShared sh;
  const int bg = blockIdx.x;
  grid_dep_wait();
  const int T = a.seq_len[bg / a.G];
  topk_select(a.block_scores + (size_t)bg * a.nb_cap, a.idx + (size_t)bg * (a.topk + 2), a.cnt + bg, a.topk,
              a.max_ctx, T, sh);
}

void launch_select_topk(const SelectArgs& a, int bg_count, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(bg_count);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, select_topk_kernel, a);
}

void launch_forecast_score(const SelectArgs& a, int bg_count, cudaStream_t s) {
  cudaFuncSetAttribute(forecast_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem);
  SelectArgs b = a;
  b.n_units = bg_count * a.nb_cap;
  const int by_work = (b.n_units + kSubBlocks - 1) / kSubBlocks;
  const int grid = by_work < sel_sm_count() ? by_work : sel_sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = kScoreSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, forecast_score_kernel, b);
}

}  // namespace sparda
