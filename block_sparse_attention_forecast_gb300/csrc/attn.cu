// Launch of the standalone block-sparse decode attention kernel; its per-CTA work is
// attn_cta (attn_body.cuh), which the fused attend-and-select kernel (fused.cu) shares.
#include "attn_body.cuh"

namespace sparda {

int attn_blocks_per_cta() { return 1; }   // workspace holds up to topk+2 partials per group

__global__ void __launch_bounds__(kAttnThreads, 1) sparse_attn_kernel(
    const AttnArgs a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
    const __grid_constant__ CUtensorMap hk, const __grid_constant__ CUtensorMap hv) {
  attn_cta(a, &mk, &mv, &hk, &hv, blockIdx.x, gridDim.x);
}

int sm_count() {
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

void launch_sparse_attn(const AttnArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& hk, const CUtensorMap& hv, int bg_count,
                        cudaStream_t s) {
  cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  AttnArgs b = a;
  b.n_units = bg_count * a.kslots;
  int grid = b.n_units < sm_count() ? b.n_units : sm_count();
  // a whole number of CTAs per (sequence, group) when the groups fit the SMs: no CTA spans
  // two groups
  if (bg_count <= sm_count()) {
    int sg = sm_count() / bg_count;
    if (sg > a.kslots) sg = a.kslots;
    b.seg_per_group = sg;
    grid = sg * bg_count;
  }
  // Programmatic serialization: barrier set-up and the unit metadata overlap the append
  // before it in the stream; the producer waits for it before the first TMA load.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kAttnSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, sparse_attn_kernel, b, mk, mv, hk, hv);
}

}  // namespace sparda
