// A layer's decode prologue: three small, independent jobs of one layer in one launch.
//
//   * the top-k of the layer's block scores, which the previous layer's launch computed
//     while it attended (bittide thread: layer L's forecast selects layer L+1's blocks
//     while layer L still computes), giving the blocks this layer attends;
//   * the append of this layer's token key/value and the compressed key of a window that
//     the token completes (techwalker section 四);
//   * the forecast projection of this layer's hidden state for the next layer (techwalker
//     section 二).
//
// Each alone is a launch of a few microseconds that leaves most of the GPU idle; together they
// cost one launch. The grid is cut into role ranges: projection tiles (8 rows x kProjSeqs
// sequences each), then one top-k CTA per (sequence, group), then append CTAs of four (sequence, group)
// pairs each. Only the top-k reads what the previous launch (attention beside the selection)
// writes: the layer's block scores. The projection reads the layer's hidden state and
// weights, and the append writes the token's key/value and the window it completes, which
// that launch does not read (it scores windows [0, num_windows(T-1)) of this layer, and the
// token completes window num_windows(T-1)). So only the top-k CTAs wait for the previous
// launch to complete; the others start as soon as SMs free up -- the previous launch lets
// this one begin while it runs, and the projection tiles, first in the grid, take the SMs its
// attention CTAs release while its selection CTAs still stream. The top-k CTAs let the next
// launch begin only after their wait (programmatic dependent launch: its selection producers
// start streaming compressed keys during the top-k), so the next launch never begins before
// the previous one has completed. A launch without a top-k has its append CTAs wait instead,
// so that it still completes after the previous launch.
#include "append_body.cuh"
#include "project_body.cuh"
#include "timeline.cuh"
#include "topk.cuh"

namespace sparda {

static_assert(kTopkThreads == kProjThreads, "the roles share one CTA shape");
constexpr int kPrologueThreads = kProjThreads;     // 256
constexpr int kAppendPerCta = kPrologueThreads / 64;

union PrologueShared {
  ProjShared pj;
  TopkShared tk;
};

__global__ void __launch_bounds__(kPrologueThreads) decode_prologue_kernel(const PrologueArgs a) {
  __shared__ PrologueShared sh;
  SPARDA_TL_ENTRY();
  unsigned long long t_rel = 0;
  int c = blockIdx.x;
  if (c < a.n_proj) {                  // reads only the layer's inputs and weights: no wait
    grid_dep_launch();
    const int n_tiles = a.pj.rows / 8;
    project_rows(a.pj, c % n_tiles, c / n_tiles, sh.pj, 1);
    SPARDA_TL_EXIT(a.tl_buf, a.tl_launch, kTlProjection, t_rel);
    return;
  }
  c -= a.n_proj;
  if (c < a.n_topk) {                  // the scores are the previous launch's output
    grid_dep_wait();
    SPARDA_TL_RELEASE(t_rel);
    grid_dep_launch();                 // only once the previous launch has completed
    if (c < a.bg_count) {
      const int T = a.ap.seq_len[c / a.ap.G];
      topk_select(a.block_scores + (size_t)c * a.nb_cap, a.idx + (size_t)c * (a.topk + 2), a.cnt + c,
                  a.topk, a.ap.max_ctx, T, sh.tk);
    }
    SPARDA_TL_EXIT(a.tl_buf, a.tl_launch, kTlTopk, t_rel);
    return;
  }
  if (a.n_topk == 0) grid_dep_wait();
  grid_dep_launch();
  c -= a.n_topk;
  const int bg = c * kAppendPerCta + (int)threadIdx.x / 64;
  if (bg < a.bg_count) append_token(a.ap, bg, threadIdx.x % 64);
  SPARDA_TL_EXIT(a.tl_buf, a.tl_launch, kTlAppend, t_rel);
}

void launch_decode_prologue(const PrologueArgs& args, cudaStream_t s) {
  PrologueArgs a = args;
  a.n_proj = a.pj.W ? proj_ctas(a.pj.rows, a.pj.batch) : 0;
  a.n_topk = a.block_scores ? a.bg_count : 0;
  const int n_append = (a.bg_count + kAppendPerCta - 1) / kAppendPerCta;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_proj + a.n_topk + n_append);
  cfg.blockDim = dim3(kPrologueThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  a.tl_launch = timeline_next_launch();
  a.tl_buf = timeline_buffer();
  cudaLaunchKernelEx(&cfg, decode_prologue_kernel, a);
}

}  // namespace sparda
