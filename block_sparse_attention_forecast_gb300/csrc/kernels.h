// Internal launch interface between the C ABI (api.cu) and the kernel translation units.
// Every struct is passed to its kernel by value; pointers are device (or UVA) addresses.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sparda {

// The scores-only selection of the fused launch hands out its work dynamically for up to this
// many (sequence, group)s: their forecasts must fit in shared memory beside its ring.
constexpr int kSelDynMaxGroups = 35;

struct AppendArgs {
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  __nv_bfloat16* ck;
  __nv_bfloat16* hot_k;
  __nv_bfloat16* hot_v;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int32_t* seq_len;
  int* err;
  int G, max_ctx, W_cap, on_host;
};

struct CompressArgs {
  const __nv_bfloat16* k;
  const __nv_bfloat16* hot_k;
  __nv_bfloat16* ck;
  const int32_t* seq_len;
  int* err;
  int G, max_ctx, W_cap, on_host;
};

struct ProjectArgs {
  const __nv_bfloat16* W;
  const __nv_bfloat16* h;
  __nv_bfloat16* f;
  int rows, hidden, batch;
};

struct SelectArgs {
  const __nv_bfloat16* ck;
  const __nv_bfloat16* f;        // forecast [B, G, d]
  const int32_t* seq_len;
  int32_t* idx;                  // [B, G, topk+2]
  int32_t* cnt;                  // [B, G]
  float* block_scores;           // workspace [B*G, nb_cap]
  unsigned* counters;            // workspace [B*G], zero between calls
  int* err;
  int G, W_cap, max_ctx, nb_cap, topk, chunk_blocks;
  int n_units;                   // B*G*nb_cap, set by the launcher
  int do_topk = 1;               // 0: leave the block scores for a later top-k (decode prologue)
  // scores-only selection of the fused launch with at most 35 (sequence, group)s: sub-chunks
  // are handed out from queue[0] (queue[1] counts the producers that finished); nullptr:
  // contiguous ranges
  unsigned* queue = nullptr;
  // optional: a buffer the next launches read (the next layer's forecast weights), pulled
  // into L2 by the selection CTAs once they have issued their last load
  const void* l2_prefetch = nullptr;
  size_t l2_prefetch_bytes = 0;
};

struct AttnArgs {
  const __nv_bfloat16* q;        // [B, G*H, d]
  const int32_t* idx;
  const int32_t* cnt;
  const int32_t* seq_len;
  __nv_bfloat16* out;            // [B, G*H, d]
  float* part_o;                 // workspace [B*G, n_split, H, d]
  float* part_ml;                // workspace [B*G, n_split, 2, H]
  unsigned* counters;            // workspace [B*G]
  int* err;
  int G, max_ctx, kslots, n_split, offload;
  int n_units;                   // B*G*kslots, set by the launcher
  // > 0: the grid is seg_per_group CTAs per (sequence, group), each taking an equal share of
  // that group's slots (no CTA spans two groups); 0: contiguous balanced unit ranges
  int seg_per_group = 0;
  // offload with the block cache: idx entry u's staged block is in row block
  // (bg * stage_slots + stage_slot[u]) of the staging map; nullptr: row block u
  const int32_t* stage_slot = nullptr;
  int stage_slots = 0;
  uint32_t tl_launch = 0;        // launch number for the timeline build's records
  void* tl_buf = nullptr;        // the timeline build's record store
};

struct MultiheadArgs {
  const __nv_bfloat16* q;        // [B, G*H, d]
  const int32_t* seq_len;
  int32_t* idx;                  // [B, G, topk+2]
  int32_t* cnt;                  // [B, G]
  float* block_scores;           // workspace [B*G, nb_cap]
  int* err;
  int G, W_cap, max_ctx, nb_cap, topk;
  int cluster;                   // CTAs per (sequence, group): one thread-block cluster
  int tiles_per_cta;             // 64-window tiles a CTA holds at most (shared-memory sizing)
};

struct PrefetchArgs {
  const __nv_bfloat16* hk;       // host cache (UVA) [B, G, max_ctx, d]
  const __nv_bfloat16* hv;
  const int32_t* idx;
  const int32_t* cnt;
  const int32_t* seq_len;
  __nv_bfloat16* sk;             // staging [B, G, kslots, 64, d]
  __nv_bfloat16* sv;
  int* err;
  int B, G, max_ctx, kslots;
};

// The cross-step block cache of an offloaded layer (prefetch.cu).
struct CacheArgs {
  const __nv_bfloat16* hk;       // host cache (UVA) [B, G, max_ctx, d]
  const __nv_bfloat16* hv;
  const int32_t* idx;            // [B, G, kslots]
  const int32_t* cnt;            // [B, G]
  const int32_t* seq_len;
  int32_t* cache_blocks;         // [max_batch*G, n_cache], persistent: block held per slot, -1 none
  int32_t* slot;                 // [B, G, kslots] out: cache slot of each idx entry (-1: hot / none)
  int32_t* fetch;                // [max_batch*G, n_cache] scratch: block to fetch per slot, -1 none
  unsigned long long* stats;     // optional [2]: hits, misses (accumulated)
  __nv_bfloat16* ck_cache;       // [max_batch, G, n_cache, 64, d]
  __nv_bfloat16* cv_cache;
  int* err;
  int B, G, max_ctx, kslots, n_cache;
};
void launch_cache_gather(const CacheArgs& a, cudaStream_t s);   // one CTA per (sequence, group)

void launch_append_kv(const AppendArgs& a, int bg_count, cudaStream_t s);
void launch_compress_keys(const CompressArgs& a, int bg_count, cudaStream_t s);
void launch_forecast_project(const ProjectArgs& a, cudaStream_t s);
void launch_forecast_select(const SelectArgs& a, int bg_count, cudaStream_t s);
// maps: K and V of the resident cache or of the staging buffer, then hot K and V (offload).
void launch_sparse_attn(const AttnArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& hk, const CUtensorMap& hv, int bg_count,
                        cudaStream_t s);
void launch_prefetch(const PrefetchArgs& a, int n_ctas, cudaStream_t s);
void launch_attend_and_select(const AttnArgs& a, const SelectArgs& s, const CUtensorMap& mk,
                              const CUtensorMap& mv, const CUtensorMap& hk, const CUtensorMap& hv,
                              int bg_count, cudaStream_t st);
// One launch of a layer's decode prologue (prologue.cu): the top-k of the layer's block
// scores, the append of its token and the forecast projection for the next layer.
struct PrologueArgs {
  AppendArgs ap;
  ProjectArgs pj;                // pj.W == nullptr: no projection
  const float* block_scores;     // [B*G, nb_cap]; nullptr: no top-k
  int32_t* idx;                  // [B, G, topk+2]
  int32_t* cnt;                  // [B, G]
  int topk, nb_cap, bg_count;
  int n_proj, n_topk;            // CTAs of the projection and top-k roles
  uint32_t tl_launch;            // launch number for the timeline build's records
  void* tl_buf;                  // the timeline build's record store
};
void launch_decode_prologue(const PrologueArgs& a, cudaStream_t s);
void launch_multihead_select(const MultiheadArgs& a, const CUtensorMap& mck, int bg_count, cudaStream_t s);

// Chunked prefill (prefill.cu): 64-token query chunks, chunk c of sequence-group bg at row
// bg * nb_cap + c of idx [.., topk+2], cnt and the block scores [.., nb_cap].
struct PrefillArgs {
  const __nv_bfloat16* ck;       // [max_batch, G, W_cap, d]
  const __nv_bfloat16* f;        // per-token forecasts [max_batch, max_ctx, G, d]
  const __nv_bfloat16* q;        // per-token queries [max_batch, max_ctx, G*H, d]
  __nv_bfloat16* out;            // attention output [max_batch, max_ctx, G*H, d]
  const int32_t* seq_len;        // prompt lengths [B]
  int32_t* idx;                  // [B*G, nb_cap, topk+2]
  int32_t* cnt;                  // [B*G, nb_cap]
  float* block_scores;           // workspace [B*G, nb_cap, nb_cap]
  int* err;
  int G, W_cap, max_ctx, nb_cap, topk;
};
void launch_prefill_forecast_select(const PrefillArgs& a, int batch, cudaStream_t s);
// mq: the queries [B*max_ctx*G*16 rows, 128] in boxes of 16 rows; mck: the compressed keys.
void launch_prefill_multihead_select(const PrefillArgs& a, const CUtensorMap& mq, const CUtensorMap& mck, int batch,
                                     cudaStream_t s);
// the causal block-sparse prefill attention on tcgen05 tensor cores; mq: the queries as
// [rows, 128] in 64 x 16 boxes, mk / mv: the layer's K and V as [rows, 128] in 64 x 64 boxes
void launch_prefill_attn_tc(const PrefillArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, int batch, cudaStream_t s);
int multihead_tiles(int w_cap);
int multihead_cluster_size(int n_tiles_cap, int bg_count);

// Device address of the library's device error word on the current device (api.cu).
int* dev_error_word();

// Sizes the C ABI needs to lay out workspaces.
int select_chunk_blocks(int nb_cap, int bg_count);
int attn_blocks_per_cta();
size_t smem_select_bytes(int chunk_blocks);

}  // namespace sparda
