// Launch of the standalone block-sparse decode attention kernel; its per-CTA work is
// attn_cta (attn_body.cuh), which the fused attend-and-select kernel (fused.cu) shares. When
// every (sequence, group) gets the same number (2 to 8) of CTAs, that number is the cluster
// size and a group's partial results meet in distributed shared memory, not in the workspace.
//
// Every CTA lets the next launch in the stream begin as soon as it starts (programmatic
// dependent launch): that launch's CTAs take the SMs this one leaves free and set up there
// (barriers, tensor-map prefetch), and each of the library's kernels that may begin early
// waits for this one to complete before it reads or writes anything this one touches (the
// output, the workspace, the error word). Back to back, one launch's start-up then overlaps
// the previous one's merge.
#include "attn_body.cuh"

namespace sparda {

int attn_blocks_per_cta() { return 1; }   // workspace holds up to topk+2 partials per group

__global__ void __launch_bounds__(kAttnThreads, 1) sparse_attn_kernel(
    const AttnArgs a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
    const __grid_constant__ CUtensorMap hk, const __grid_constant__ CUtensorMap hv) {
  SPARDA_TL_ENTRY();
  grid_dep_launch();
  unsigned long long tl_first = 0;
  attn_cta(a, &mk, &mv, &hk, &hv, blockIdx.x, gridDim.x, &tl_first);
  SPARDA_TL_EXIT(a.tl_buf, a.tl_launch, kTlAttention, tl_first);
}

__global__ void __launch_bounds__(kAttnThreads, 1) sparse_attn_cluster_kernel(
    const AttnArgs a, const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
    const __grid_constant__ CUtensorMap hk, const __grid_constant__ CUtensorMap hv) {
  SPARDA_TL_ENTRY();
  grid_dep_launch();
  unsigned long long tl_first = 0;
  attn_cta<true>(a, &mk, &mv, &hk, &hv, blockIdx.x, gridDim.x, &tl_first);
  SPARDA_TL_EXIT(a.tl_buf, a.tl_launch, kTlAttention, tl_first);
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
  AttnArgs b = a;
  b.n_units = bg_count * a.kslots;
  const int sms = sm_count();
  int grid = b.n_units < sms ? b.n_units : sms;
  int cluster = 0;
  // a whole number of CTAs per (sequence, group) when the groups fit the SMs: no CTA spans
  // two groups. Up to 8 of them form one cluster, when the clusters still cover three
  // quarters of the SMs (otherwise more CTAs per group, merged through the workspace).
  if (bg_count <= sms) {
    int sg = sms / bg_count;
    if (sg > a.kslots) sg = a.kslots;   // every CTA has a unit (the cluster form relies on it)
    const int sg_cl = sg < kMaxClusterCtas ? sg : kMaxClusterCtas;
    if (sg_cl >= 2 && 4 * sg_cl * bg_count >= 3 * sms) {
      sg = sg_cl;
      cluster = sg;
    }
    b.seg_per_group = sg;
    grid = sg * bg_count;
  }
  b.tl_launch = timeline_next_launch();
  b.tl_buf = timeline_buffer();
  auto kern = cluster ? sparse_attn_cluster_kernel : sparse_attn_kernel;
  const int smem = cluster ? kAttnClusterSmem : kAttnSmem;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // Programmatic serialization: the barrier set-up overlaps the kernel before it in the
  // stream; the producer waits for it before it reads the unit metadata, the consumers before
  // they write anything.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster ? 2 : 1;
  cudaLaunchKernelEx(&cfg, kern, b, mk, mv, hk, hv);
}

}  // namespace sparda
