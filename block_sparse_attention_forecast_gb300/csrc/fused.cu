// Layer L's block-sparse attention and layer L+1's Forecast selection in one persistent
// launch. Under lookahead the two are independent (layer L's forecast already exists when
// layer L attends), and each alone is a persistent kernel that wants every SM, so launched
// side by side they would only run one after the other. Here the grid is one CTA per SM,
// split between the two jobs in proportion to the bytes each must stream: the first CTAs run
// the selection work (sel_cta) over the selection units, the last n_attn the attention work
// (attn_cta) over the attention units, so both jobs stream concurrently from HBM and finish
// together, with one launch and one start-up per layer. The selection CTAs come first because
// the launch begins while the next layer's top-k CTAs of the launch before still hold SMs:
// the selection, which does not depend on them, streams on the SMs free at the start, and
// the attention CTAs, which need that top-k's blocks, take the SMs its CTAs release.
#include "attn_body.cuh"
#include "select_body.cuh"
#include "timeline.cuh"

namespace sparda {

static_assert(kAttnThreads == kSelThreads, "both jobs run with the same CTA shape");
// streamed-byte weight of an attention unit against a selection unit when splitting the SMs
constexpr double kAttnWeightWithTopk = 1.1;
constexpr double kAttnWeightScoresOnly = 1.9;
constexpr int kFusedSmem = kAttnSmem > kSelSmem ? kAttnSmem : kSelSmem;
static_assert(kFusedSmem >= 256 + kSelStages * kSelStageBytes + kSelDynMaxGroups * kHeadDim * 2,
              "the dynamic selection's forecast table fits beside its ring");

__global__ void __launch_bounds__(kAttnThreads, 1) attend_and_select_kernel(
    const AttnArgs aa, const SelectArgs sa, int n_attn, const __grid_constant__ CUtensorMap mk,
    const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap hk,
    const __grid_constant__ CUtensorMap hv) {
  SPARDA_TL_ENTRY();
  grid_dep_launch();                   // the next prologue's projection may take freed SMs
  const int n_sel = (int)gridDim.x - n_attn;
  const bool attn = (int)blockIdx.x >= n_sel;
  unsigned long long tl_first = 0;         // an attention CTA's first block (timeline build)
  if (attn)
    attn_cta(aa, &mk, &mv, &hk, &hv, blockIdx.x - n_sel, n_attn, &tl_first);
  else if (sa.queue)
    sel_cta_dyn(sa, blockIdx.x, n_sel);
  else
    sel_cta(sa, blockIdx.x, n_sel);
  SPARDA_TL_EXIT(aa.tl_buf, aa.tl_launch, attn ? kTlAttention : kTlSelection, tl_first);
}

int sm_count();

void launch_attend_and_select(const AttnArgs& a, const SelectArgs& s, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& hk, const CUtensorMap& hv,
                              int bg_count, cudaStream_t st) {
  cudaFuncSetAttribute(attend_and_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem);
  AttnArgs aa = a;
  SelectArgs sa = s;
  aa.n_units = bg_count * a.kslots;
  sa.n_units = bg_count * s.nb_cap;
  // split the SMs by streamed bytes: an attention unit is one K+V block (32 KiB), a selection
  // unit one block's four windows of compressed keys (1 KiB). An attention CTA streams fewer
  // bytes per microsecond than a selection CTA (it merges split groups and computes more per
  // byte); a selection CTA that also runs top-k tails streams fewer. The weights are measured
  // at 128K context, batch 16.
  const double w_attn = sa.do_topk ? kAttnWeightWithTopk : kAttnWeightScoresOnly;
  const double wa = w_attn * (double)aa.n_units * (2.0 * kBlockBytes);
  const double ws = (double)sa.n_units * (kWinPerBlock * kRowBytes);
  const int sms = sm_count();
  int n_attn = (int)(sms * wa / (wa + ws) + 0.5);
  n_attn = n_attn < 1 ? 1 : (n_attn > sms - 1 ? sms - 1 : n_attn);
  if (n_attn > aa.n_units) n_attn = aa.n_units;
  // Prefer a whole number of attention CTAs per (sequence, group), so that no CTA spans two
  // groups (a group boundary costs a CTA a merge and a fresh start of its pipeline), when
  // that lands within about a third of the byte-proportional count.
  const int per = aa.kslots;
  int sg = (n_attn + bg_count / 2) / bg_count;
  if (sg < 1) sg = 1;
  if (sg > per) sg = per;
  const int aligned = sg * bg_count;
  if (aligned <= sms - 1 && 3 * abs(aligned - n_attn) <= n_attn) {
    n_attn = aligned;
    aa.seg_per_group = sg;
  }
  int n_sel = sms - n_attn;
  const int sel_work = (sa.n_units + kSubBlocks - 1) / kSubBlocks;
  if (n_sel > sel_work) n_sel = sel_work;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_attn + n_sel);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  aa.tl_launch = timeline_next_launch();
  aa.tl_buf = timeline_buffer();
  cudaLaunchKernelEx(&cfg, attend_and_select_kernel, aa, sa, n_attn, mk, mv, hk, hv);
}

}  // namespace sparda
