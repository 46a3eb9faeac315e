// The C ABI of libsparda (declared in include/sparda.h): argument checks, workspace layout,
// TMA tensor-map encoding and kernel launches. Nothing here allocates device or host memory.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace sparda;

namespace sparda {
void launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t s);   // copy.cu
void launch_device_status(int* err, int32_t* out, bool clear, cudaStream_t s);  // copy.cu
void launch_forecast_score(const SelectArgs& a, int bg_count, cudaStream_t s);  // select.cu
void launch_select_topk(const SelectArgs& a, int bg_count, cudaStream_t s);     // select.cu
}

// The device error word (bits SPARDA_DEV_*). Kernels receive its device address.
__device__ int g_sparda_dev_error;

#include "timeline.cuh"
#ifdef SPARDA_TIMELINE
#include <atomic>
static __device__ sparda::TimelineBuf g_sparda_timeline;
namespace sparda {
static std::atomic<uint32_t> g_tl_launch{0};
uint32_t timeline_next_launch() { return g_tl_launch.fetch_add(1) + 1; }
void* timeline_buffer() {
  void* p = nullptr;
  return cudaGetSymbolAddress(&p, g_sparda_timeline) == cudaSuccess ? p : nullptr;
}
}  // namespace sparda
// Timeline build only (not part of the product ABI): copy up to max_records records
// (t_entry, t_release, t_exit as uint64 ns; launch, role << 24 | cta as uint32) to host memory,
// the count to *n, and, if reset != 0, clear the count and restart the launch numbering.
extern "C" int32_t sparda_timeline_read(void* host, int32_t max_records, int32_t* n, int32_t reset) {
  unsigned int cnt = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPARDA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&cnt, g_sparda_timeline, sizeof(cnt)) != cudaSuccess) return SPARDA_ERR_CUDA;
  if (cnt > (unsigned)sparda::kTimelineMax) cnt = sparda::kTimelineMax;
  const unsigned int k = cnt < (unsigned)max_records ? cnt : (unsigned)max_records;
  if (host && k &&
      cudaMemcpyFromSymbol(host, g_sparda_timeline, k * sizeof(sparda::TimelineRec),
                           offsetof(sparda::TimelineBuf, rec)) != cudaSuccess)
    return SPARDA_ERR_CUDA;
  if (n) *n = (int32_t)k;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_sparda_timeline, &zero, sizeof(zero)) != cudaSuccess) return SPARDA_ERR_CUDA;
    sparda::g_tl_launch = 0;
  }
  return SPARDA_OK;
}
#else
namespace sparda {
uint32_t timeline_next_launch() { return 0; }
void* timeline_buffer() { return nullptr; }
}  // namespace sparda
#endif

namespace {

constexpr int kMaxDevices = 64;

int* dev_error_ptr() {
  static int* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sparda_dev_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int32_t shape_status(const sparda_shape* s) {
  if (!s) return SPARDA_ERR_INVALID_ARG;
  if (s->head_dim != kHeadDim || s->heads_per_group != kHeads || s->block != kBlock ||
      s->win_kernel != kWinKernel || s->win_stride != kWinStride)
    return SPARDA_ERR_UNSUPPORTED_SHAPE;
  if (s->n_groups < 1 || s->max_batch < 1 || s->topk < 1 || s->topk > kMaxTopk ||
      s->max_ctx < kBlock || s->max_ctx % kBlock != 0 || s->max_ctx > kMaxCtx)
    return SPARDA_ERR_UNSUPPORTED_SHAPE;
  // every row index of a cache must fit a signed 32-bit TMA coordinate
  if ((int64_t)s->max_batch * s->n_groups * s->max_ctx >= (int64_t)1 << 31)
    return SPARDA_ERR_UNSUPPORTED_SHAPE;
  return SPARDA_OK;
}

int32_t batch_status(const sparda_shape* s, int32_t batch) {
  return (batch < 1 || batch > s->max_batch) ? SPARDA_ERR_INVALID_ARG : SPARDA_OK;
}

int w_cap(const sparda_shape* s) { return num_windows(s->max_ctx); }
int nb_cap(const sparda_shape* s) { return s->max_ctx / kBlock; }
int kslots(const sparda_shape* s) { return s->topk + 2; }
int attn_splits(const sparda_shape* s) {
  return (kslots(s) + attn_blocks_per_cta() - 1) / attn_blocks_per_cta();
}
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspaces are laid out for max_batch sequences so that their counters sit at the same
// place whatever batch a call uses: [counters: max_batch*G u32][data]. The selection
// workspace starts with kQueueBytes for the dynamic selection's work counter.
constexpr size_t kQueueBytes = 256;
size_t counters_bytes(const sparda_shape* s) {
  return round256((size_t)s->max_batch * s->n_groups * sizeof(unsigned));
}
size_t select_data_bytes(const sparda_shape* s) {
  return round256((size_t)s->max_batch * s->n_groups * nb_cap(s) * sizeof(float));
}
size_t attn_o_bytes(const sparda_shape* s) {
  return round256((size_t)s->max_batch * s->n_groups * attn_splits(s) * kHeads * kHeadDim * sizeof(float));
}
size_t attn_ml_bytes(const sparda_shape* s) {
  return round256((size_t)s->max_batch * s->n_groups * attn_splits(s) * 2 * kHeads * sizeof(float));
}


int32_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SPARDA_OK;
  std::fprintf(stderr, "sparda: CUDA error %s\n", cudaGetErrorString(e));
  return SPARDA_ERR_CUDA;
}

// ------------------------------------------------------------------ TMA tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A [rows, 128] bf16 matrix read in boxes of box_rows rows x 64 columns, 128-byte swizzle.
int32_t make_kv_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows = 64) {
  EncodeTiledFn enc = encoder();
  if (!enc) return SPARDA_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPARDA_OK : SPARDA_ERR_CUDA;
}

// Pinned host memory mapped into the device's address space.
int32_t host_mapped_status(const void* p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return SPARDA_ERR_NOT_MAPPED_HOST;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return SPARDA_ERR_NOT_MAPPED_HOST;
  // the kernels dereference the pointer as given: it must be the memory's device address
  if (attr.devicePointer != p) return SPARDA_ERR_NOT_MAPPED_HOST;
  return SPARDA_OK;
}

// Memory the kernels can dereference as given: device memory, or mapped pinned host memory.
int32_t device_addressable_status(const void* p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return SPARDA_ERR_NOT_MAPPED_HOST;
  }
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) return SPARDA_OK;
  return host_mapped_status(p);
}

int32_t layer_status(const sparda_layer_kv* L, bool need_kv) {
  if (!L || !L->ck) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(L->ck, 16)) return SPARDA_ERR_MISALIGNED;
  if (!need_kv) return SPARDA_OK;
  if (!L->k || !L->v) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(L->k, 16) || !aligned(L->v, 16)) return SPARDA_ERR_MISALIGNED;
  if (L->on_host) {
    if (!L->hot_k || !L->hot_v) return SPARDA_ERR_INVALID_ARG;
    if (!aligned(L->hot_k, 16) || !aligned(L->hot_v, 16)) return SPARDA_ERR_MISALIGNED;
    int32_t st = host_mapped_status(L->k);
    if (st == SPARDA_OK) st = host_mapped_status(L->v);
    if (st != SPARDA_OK) return st;
  }
  return SPARDA_OK;
}

#define SPARDA_TRY(x)                     \
  do {                                    \
    const int32_t st_ = (x);              \
    if (st_ != SPARDA_OK) return st_;     \
  } while (0)

}  // namespace

int* sparda::dev_error_word() { return dev_error_ptr(); }

extern "C" {

int32_t sparda_abi_version(void) { return 1; }

const char* sparda_status_string(int32_t status) {
  switch (status) {
    case SPARDA_OK: return "ok";
    case SPARDA_ERR_INVALID_ARG: return "invalid argument";
    case SPARDA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SPARDA_ERR_MISALIGNED: return "misaligned pointer";
    case SPARDA_ERR_NOT_MAPPED_HOST: return "host memory not pinned and mapped for the device";
    case SPARDA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SPARDA_ERR_CUDA: return "CUDA error";
    case SPARDA_ERR_STATIC_SCRATCH_LIMIT:
      return "request exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int32_t sparda_check_shape(const sparda_shape* shape) { return shape_status(shape); }

size_t sparda_workspace_bytes(const sparda_shape* s, int32_t batch, int32_t kind) {
  if (shape_status(s) != SPARDA_OK || batch < 1 || batch > s->max_batch) return 0;
  switch (kind) {
    case SPARDA_WS_SELECT: return kQueueBytes + counters_bytes(s) + select_data_bytes(s);
    case SPARDA_WS_ATTN: return counters_bytes(s) + attn_o_bytes(s) + attn_ml_bytes(s);
    case SPARDA_WS_MULTIHEAD: return select_data_bytes(s);
    case SPARDA_WS_PREFILL: return round256((size_t)s->max_batch * s->n_groups * nb_cap(s) * nb_cap(s) * sizeof(float));
    default: return 0;
  }
}

size_t sparda_block_scores_offset(const sparda_shape* s) {
  return shape_status(s) == SPARDA_OK ? kQueueBytes + counters_bytes(s) : 0;
}

int32_t sparda_device_error(int32_t* flags, int32_t clear) {
  if (!flags) return SPARDA_ERR_INVALID_ARG;
  int* p = dev_error_ptr();
  if (!p) return SPARDA_ERR_CUDA;
  SPARDA_TRY(cuda_status(cudaDeviceSynchronize()));
  SPARDA_TRY(cuda_status(cudaMemcpy(flags, p, sizeof(int), cudaMemcpyDeviceToHost)));
  if (clear) SPARDA_TRY(cuda_status(cudaMemset(p, 0, sizeof(int))));
  return SPARDA_OK;
}

int32_t sparda_get_device_status(int32_t* dev_flag, int32_t clear, void* stream) {
  if (!dev_flag) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(dev_flag, 4)) return SPARDA_ERR_MISALIGNED;
  SPARDA_TRY(device_addressable_status(dev_flag));
  int* p = dev_error_ptr();
  if (!p) return SPARDA_ERR_CUDA;
  launch_device_status(p, dev_flag, clear != 0, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_prefetch_default_ctas(int32_t batch) { return batch < 32 ? 64 : 152; }

int32_t sparda_copy(void* dst, const void* src, size_t bytes, void* stream) {
  if (!dst || !src || bytes == 0 || bytes % 16 != 0) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(dst, 16) || !aligned(src, 16)) return SPARDA_ERR_MISALIGNED;
  SPARDA_TRY(device_addressable_status(dst));
  SPARDA_TRY(device_addressable_status(src));
  launch_copy16(dst, src, bytes, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_append_kv(const sparda_shape* s, const sparda_layer_kv* L, const void* k_new,
                         const void* v_new, const int32_t* seq_len, int32_t batch, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  SPARDA_TRY(layer_status(L, true));
  if (!k_new || !v_new || !seq_len) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(seq_len, 4)) return SPARDA_ERR_MISALIGNED;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  AppendArgs a{static_cast<__nv_bfloat16*>(L->k), static_cast<__nv_bfloat16*>(L->v),
               static_cast<__nv_bfloat16*>(L->ck), static_cast<__nv_bfloat16*>(L->hot_k),
               static_cast<__nv_bfloat16*>(L->hot_v), static_cast<const __nv_bfloat16*>(k_new),
               static_cast<const __nv_bfloat16*>(v_new), seq_len, err, s->n_groups, s->max_ctx,
               w_cap(s), L->on_host ? 1 : 0};
  launch_append_kv(a, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_compress_keys(const sparda_shape* s, const sparda_layer_kv* L, const int32_t* seq_len,
                             int32_t batch, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  SPARDA_TRY(layer_status(L, true));
  if (!seq_len) return SPARDA_ERR_INVALID_ARG;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  CompressArgs a{static_cast<const __nv_bfloat16*>(L->k), static_cast<const __nv_bfloat16*>(L->hot_k),
                 static_cast<__nv_bfloat16*>(L->ck), seq_len, err, s->n_groups, s->max_ctx, w_cap(s),
                 L->on_host ? 1 : 0};
  launch_compress_keys(a, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_forecast_project(const void* W, const void* h, int32_t rows, int32_t hidden,
                                int32_t batch, void* f, void* stream) {
  if (!W || !h || !f) return SPARDA_ERR_INVALID_ARG;
  if (rows < 8 || rows % 8 != 0 || hidden < 32 || hidden % 32 != 0 || batch < 1)
    return SPARDA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W, 16) || !aligned(h, 16) || !aligned(f, 16)) return SPARDA_ERR_MISALIGNED;
  ProjectArgs a{static_cast<const __nv_bfloat16*>(W), static_cast<const __nv_bfloat16*>(h),
                static_cast<__nv_bfloat16*>(f), rows, hidden, batch};
  launch_forecast_project(a, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

}  // extern "C"

namespace {

// Argument checks and kernel arguments of the selection call (shared by the standalone and
// the fused entry points). With idx == cnt == nullptr only the block scores are wanted
// (the top-k runs later, in the decode prologue).
int32_t prepare_select(const sparda_shape* s, const void* ck, const void* forecast, const int32_t* seq_len,
                       int32_t batch, int32_t* idx, int32_t* cnt, void* ws, size_t ws_bytes, SelectArgs* out,
                       bool scores_only = false) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!ck || !forecast || !seq_len || !ws) return SPARDA_ERR_INVALID_ARG;
  if (!scores_only && (!idx || !cnt)) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(ck, 16) || !aligned(forecast, 16) || !aligned(ws, 16) || !aligned(idx, 4) ||
      !aligned(cnt, 4) || !aligned(seq_len, 4))
    return SPARDA_ERR_MISALIGNED;
  if (ws_bytes < sparda_workspace_bytes(s, batch, SPARDA_WS_SELECT)) return SPARDA_ERR_WORKSPACE_TOO_SMALL;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws) + kQueueBytes;
  const int bgc = batch * s->n_groups;
  *out = SelectArgs{static_cast<const __nv_bfloat16*>(ck), static_cast<const __nv_bfloat16*>(forecast),
                    seq_len, idx, cnt, reinterpret_cast<float*>(w + counters_bytes(s)),
                    reinterpret_cast<unsigned*>(w), err, s->n_groups, w_cap(s), s->max_ctx, nb_cap(s),
                    s->topk, select_chunk_blocks(nb_cap(s), bgc), 0, scores_only ? 0 : 1};
  // the scores-only selection hands out its sub-chunks dynamically when the forecasts of all
  // its (sequence, group)s fit in shared memory beside the ring
  if (scores_only && bgc <= kSelDynMaxGroups) out->queue = static_cast<unsigned*>(ws);
  return SPARDA_OK;
}

// Argument checks, tensor maps and kernel arguments of the attention call.
int32_t prepare_attn(const sparda_shape* s, const sparda_layer_kv* L, const void* staging_k,
                     const void* staging_v, const void* q, const int32_t* idx, const int32_t* cnt,
                     const int32_t* seq_len, int32_t batch, void* out, void* ws, size_t ws_bytes,
                     AttnArgs* args, CUtensorMap* mk, CUtensorMap* mv, CUtensorMap* hk, CUtensorMap* hv,
                     int staging_slots = 0) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!L || !q || !idx || !cnt || !seq_len || !out || !ws) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(ws, 16) || !aligned(idx, 4) || !aligned(cnt, 4))
    return SPARDA_ERR_MISALIGNED;
  if (ws_bytes < sparda_workspace_bytes(s, batch, SPARDA_WS_ATTN)) return SPARDA_ERR_WORKSPACE_TOO_SMALL;
  const uint64_t bgcap = (uint64_t)s->max_batch * s->n_groups;
  if (L->on_host) {
    if (!staging_k || !staging_v || !L->hot_k || !L->hot_v) return SPARDA_ERR_INVALID_ARG;
    if (!aligned(staging_k, 16) || !aligned(staging_v, 16) || !aligned(L->hot_k, 16) || !aligned(L->hot_v, 16))
      return SPARDA_ERR_MISALIGNED;
    const uint64_t per_bg = (uint64_t)(staging_slots > 0 ? staging_slots : kslots(s));
    SPARDA_TRY(make_kv_map(mk, staging_k, bgcap * per_bg * kBlock));
    SPARDA_TRY(make_kv_map(mv, staging_v, bgcap * per_bg * kBlock));
    SPARDA_TRY(make_kv_map(hk, L->hot_k, bgcap * kHotSlots * kBlock));
    SPARDA_TRY(make_kv_map(hv, L->hot_v, bgcap * kHotSlots * kBlock));
  } else {
    if (!L->k || !L->v) return SPARDA_ERR_INVALID_ARG;
    if (!aligned(L->k, 16) || !aligned(L->v, 16)) return SPARDA_ERR_MISALIGNED;
    SPARDA_TRY(make_kv_map(mk, L->k, bgcap * s->max_ctx));
    SPARDA_TRY(make_kv_map(mv, L->v, bgcap * s->max_ctx));
    *hk = *mk;
    *hv = *mv;
  }
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  *args = AttnArgs{static_cast<const __nv_bfloat16*>(q), idx, cnt, seq_len, static_cast<__nv_bfloat16*>(out),
                   reinterpret_cast<float*>(w + counters_bytes(s)),
                   reinterpret_cast<float*>(w + counters_bytes(s) + attn_o_bytes(s)),
                   reinterpret_cast<unsigned*>(w), err, s->n_groups, s->max_ctx, kslots(s), attn_splits(s),
                   L->on_host ? 1 : 0, 0};
  return SPARDA_OK;
}

}  // namespace

extern "C" {

int32_t sparda_forecast_select(const sparda_shape* s, const void* ck, const void* forecast,
                               const int32_t* seq_len, int32_t batch, int32_t* idx, int32_t* cnt,
                               void* ws, size_t ws_bytes, void* stream) {
  SelectArgs a;
  SPARDA_TRY(prepare_select(s, ck, forecast, seq_len, batch, idx, cnt, ws, ws_bytes, &a));
  const int bgc = batch * s->n_groups;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (bgc <= kSelDynMaxGroups) {
    // the block scores on every SM, handed out from the workspace's queue, then one top-k CTA
    // per (sequence, group): the queue keeps the SMs busy to the end, which a top-k tail on
    // the last CTA of each group does not
    SelectArgs sc = a;
    sc.queue = static_cast<unsigned*>(ws);
    sc.do_topk = 0;
    launch_forecast_score(sc, bgc, st);
    launch_select_topk(a, bgc, st);
  } else {
    launch_forecast_select(a, bgc, st);
  }
  return cuda_status(cudaGetLastError());
}

int32_t sparda_forecast_score(const sparda_shape* s, const void* ck, const void* forecast,
                              const int32_t* seq_len, int32_t batch, void* ws, size_t ws_bytes,
                              void* stream) {
  SelectArgs a;
  SPARDA_TRY(prepare_select(s, ck, forecast, seq_len, batch, nullptr, nullptr, ws, ws_bytes, &a, true));
  launch_forecast_score(a, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_sparse_decode_attn(const sparda_shape* s, const sparda_layer_kv* L, const void* staging_k,
                                  const void* staging_v, const void* q, const int32_t* idx,
                                  const int32_t* cnt, const int32_t* seq_len, int32_t batch, void* out,
                                  void* ws, size_t ws_bytes, void* stream) {
  AttnArgs a;
  CUtensorMap mk, mv, hk, hv;
  SPARDA_TRY(prepare_attn(s, L, staging_k, staging_v, q, idx, cnt, seq_len, batch, out, ws, ws_bytes, &a, &mk,
                          &mv, &hk, &hv));
  launch_sparse_attn(a, mk, mv, hk, hv, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_attend_and_select(const sparda_shape* s, const sparda_layer_kv* L, const void* staging_k,
                                 const void* staging_v, const void* q, const int32_t* idx, const int32_t* cnt,
                                 void* out, void* ws_attn, size_t ws_attn_bytes, const void* ck_next,
                                 const void* forecast_next, int32_t* idx_next, int32_t* cnt_next, void* ws_sel,
                                 size_t ws_sel_bytes, const int32_t* seq_len, int32_t batch, void* stream) {
  if (idx_next == idx || cnt_next == cnt || ws_sel == ws_attn) return SPARDA_ERR_INVALID_ARG;
  AttnArgs a;
  CUtensorMap mk, mv, hk, hv;
  SPARDA_TRY(prepare_attn(s, L, staging_k, staging_v, q, idx, cnt, seq_len, batch, out, ws_attn, ws_attn_bytes,
                          &a, &mk, &mv, &hk, &hv));
  SelectArgs sa;
  SPARDA_TRY(prepare_select(s, ck_next, forecast_next, seq_len, batch, idx_next, cnt_next, ws_sel, ws_sel_bytes,
                            &sa));
  launch_attend_and_select(a, sa, mk, mv, hk, hv, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_attend_and_score(const sparda_shape* s, const sparda_layer_kv* L, const void* staging_k,
                                const void* staging_v, const void* q, const int32_t* idx, const int32_t* cnt,
                                void* out, void* ws_attn, size_t ws_attn_bytes, const void* ck_next,
                                const void* forecast_next, void* ws_scores, size_t ws_scores_bytes,
                                const void* l2_next, size_t l2_next_bytes, const int32_t* seq_len, int32_t batch,
                                void* stream) {
  if (l2_next && (!aligned(l2_next, 16) || l2_next_bytes % 16 != 0)) return SPARDA_ERR_MISALIGNED;
  if (ws_scores == ws_attn) return SPARDA_ERR_INVALID_ARG;
  AttnArgs a;
  CUtensorMap mk, mv, hk, hv;
  SPARDA_TRY(prepare_attn(s, L, staging_k, staging_v, q, idx, cnt, seq_len, batch, out, ws_attn, ws_attn_bytes,
                          &a, &mk, &mv, &hk, &hv));
  SelectArgs sa;
  SPARDA_TRY(prepare_select(s, ck_next, forecast_next, seq_len, batch, nullptr, nullptr, ws_scores,
                            ws_scores_bytes, &sa, true));
  sa.l2_prefetch = l2_next;
  sa.l2_prefetch_bytes = l2_next ? l2_next_bytes : 0;
  launch_attend_and_select(a, sa, mk, mv, hk, hv, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_decode_prologue(const sparda_shape* s, const sparda_layer_kv* L, const void* k_new,
                               const void* v_new, const void* ws_scores, size_t ws_scores_bytes, int32_t* idx,
                               int32_t* cnt, const void* W_next, const void* h, int32_t hidden,
                               void* forecast_next, const int32_t* seq_len, int32_t batch, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  SPARDA_TRY(layer_status(L, true));
  if (!k_new || !v_new || !seq_len) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(seq_len, 4)) return SPARDA_ERR_MISALIGNED;
  if (ws_scores) {
    if (!idx || !cnt) return SPARDA_ERR_INVALID_ARG;
    if (!aligned(ws_scores, 16) || !aligned(idx, 4) || !aligned(cnt, 4)) return SPARDA_ERR_MISALIGNED;
    if (ws_scores_bytes < sparda_workspace_bytes(s, batch, SPARDA_WS_SELECT))
      return SPARDA_ERR_WORKSPACE_TOO_SMALL;
  }
  if (W_next) {
    if (!h || !forecast_next) return SPARDA_ERR_INVALID_ARG;
    if (hidden < 32 || hidden % 32 != 0) return SPARDA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(W_next, 16) || !aligned(h, 16) || !aligned(forecast_next, 16)) return SPARDA_ERR_MISALIGNED;
  }
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  PrologueArgs a{};
  a.ap = AppendArgs{static_cast<__nv_bfloat16*>(L->k), static_cast<__nv_bfloat16*>(L->v),
                    static_cast<__nv_bfloat16*>(L->ck), static_cast<__nv_bfloat16*>(L->hot_k),
                    static_cast<__nv_bfloat16*>(L->hot_v), static_cast<const __nv_bfloat16*>(k_new),
                    static_cast<const __nv_bfloat16*>(v_new), seq_len, err, s->n_groups, s->max_ctx,
                    w_cap(s), L->on_host ? 1 : 0};
  a.pj = ProjectArgs{static_cast<const __nv_bfloat16*>(W_next), static_cast<const __nv_bfloat16*>(h),
                     static_cast<__nv_bfloat16*>(forecast_next), s->n_groups * kHeadDim, hidden, batch};
  a.block_scores = ws_scores ? reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws_scores) +
                                                              sparda_block_scores_offset(s))
                             : nullptr;
  a.idx = idx;
  a.cnt = cnt;
  a.topk = s->topk;
  a.nb_cap = nb_cap(s);
  a.bg_count = batch * s->n_groups;
  launch_decode_prologue(a, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_prefetch_blocks(const sparda_shape* s, const sparda_layer_kv* L, const int32_t* idx,
                               const int32_t* cnt, const int32_t* seq_len, int32_t batch, void* staging_k,
                               void* staging_v, int32_t n_ctas, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!L || !L->on_host) return SPARDA_ERR_INVALID_ARG;
  SPARDA_TRY(layer_status(L, true));
  if (!idx || !cnt || !seq_len || !staging_k || !staging_v || n_ctas < 0 || n_ctas > 4096)
    return SPARDA_ERR_INVALID_ARG;
  if (!aligned(staging_k, 16) || !aligned(staging_v, 16)) return SPARDA_ERR_MISALIGNED;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  PrefetchArgs a{static_cast<const __nv_bfloat16*>(L->k), static_cast<const __nv_bfloat16*>(L->v), idx, cnt,
                 seq_len, static_cast<__nv_bfloat16*>(staging_k), static_cast<__nv_bfloat16*>(staging_v), err,
                 batch, s->n_groups, s->max_ctx, kslots(s)};
  launch_prefetch(a, n_ctas ? n_ctas : sparda_prefetch_default_ctas(batch), static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_multihead_select(const sparda_shape* s, const void* ck, const void* q, const int32_t* seq_len,
                                int32_t batch, int32_t* idx, int32_t* cnt, void* ws, size_t ws_bytes,
                                void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!ck || !q || !seq_len || !idx || !cnt || !ws) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(ck, 16) || !aligned(q, 16) || !aligned(ws, 16) || !aligned(idx, 4) || !aligned(cnt, 4) ||
      !aligned(seq_len, 4))
    return SPARDA_ERR_MISALIGNED;
  if (ws_bytes < sparda_workspace_bytes(s, batch, SPARDA_WS_MULTIHEAD)) return SPARDA_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap mck;
  SPARDA_TRY(make_kv_map(&mck, ck, (uint64_t)s->max_batch * s->n_groups * w_cap(s)));
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  const int n_tiles = multihead_tiles(w_cap(s));
  const int ncl = multihead_cluster_size(n_tiles, batch * s->n_groups);
  MultiheadArgs a{static_cast<const __nv_bfloat16*>(q), seq_len, idx, cnt, static_cast<float*>(ws), err,
                  s->n_groups, w_cap(s), s->max_ctx, nb_cap(s), s->topk, ncl, (n_tiles + ncl - 1) / ncl};
  launch_multihead_select(a, mck, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}


// ------------------------------------------------------------------ chunked prefill
}  // extern "C"

namespace {

int32_t prepare_prefill(const sparda_shape* s, const void* ck, const void* qf, const int32_t* seq_len, int32_t batch,
                        int32_t* idx, int32_t* cnt, void* ws, size_t ws_bytes, PrefillArgs* a) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!ck || !qf || !seq_len || !idx || !cnt || !ws) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(ck, 16) || !aligned(qf, 16) || !aligned(ws, 16) || !aligned(idx, 4) || !aligned(cnt, 4) ||
      !aligned(seq_len, 4))
    return SPARDA_ERR_MISALIGNED;
  if (ws_bytes < sparda_workspace_bytes(s, batch, SPARDA_WS_PREFILL)) return SPARDA_ERR_WORKSPACE_TOO_SMALL;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  *a = PrefillArgs{static_cast<const __nv_bfloat16*>(ck), nullptr, nullptr, nullptr, seq_len, idx, cnt,
                   static_cast<float*>(ws), err, s->n_groups, w_cap(s), s->max_ctx, nb_cap(s), s->topk};
  return SPARDA_OK;
}

}  // namespace

extern "C" {

int32_t sparda_prefill_forecast_select(const sparda_shape* s, const void* ck, const void* forecast,
                                       const int32_t* seq_len, int32_t batch, int32_t* idx, int32_t* cnt, void* ws,
                                       size_t ws_bytes, void* stream) {
  PrefillArgs a;
  SPARDA_TRY(prepare_prefill(s, ck, forecast, seq_len, batch, idx, cnt, ws, ws_bytes, &a));
  a.f = static_cast<const __nv_bfloat16*>(forecast);
  launch_prefill_forecast_select(a, batch, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_prefill_multihead_select(const sparda_shape* s, const void* ck, const void* q,
                                        const int32_t* seq_len, int32_t batch, int32_t* idx, int32_t* cnt, void* ws,
                                        size_t ws_bytes, void* stream) {
  PrefillArgs a;
  SPARDA_TRY(prepare_prefill(s, ck, q, seq_len, batch, idx, cnt, ws, ws_bytes, &a));
  a.q = static_cast<const __nv_bfloat16*>(q);
  const uint64_t rows = (uint64_t)s->max_batch * s->n_groups * s->max_ctx;
  // every query row must fit a signed 32-bit TMA coordinate
  if (rows * kHeads >= ((uint64_t)1 << 31)) return SPARDA_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap mck, mq;
  SPARDA_TRY(make_kv_map(&mck, ck, (uint64_t)s->max_batch * s->n_groups * w_cap(s)));
  SPARDA_TRY(make_kv_map(&mq, q, rows * kHeads, 16));
  launch_prefill_multihead_select(a, mq, mck, batch, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}

int32_t sparda_prefill_attn(const sparda_shape* s, const sparda_layer_kv* L, const void* q, const int32_t* idx,
                            const int32_t* cnt, const int32_t* seq_len, int32_t batch, void* out, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  SPARDA_TRY(layer_status(L, true));
  if (L->on_host) return SPARDA_ERR_INVALID_ARG;              // prefill attends a resident layer
  if (!q || !idx || !cnt || !seq_len || !out) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(idx, 4) || !aligned(cnt, 4) || !aligned(seq_len, 4))
    return SPARDA_ERR_MISALIGNED;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  const uint64_t rows = (uint64_t)s->max_batch * s->n_groups * s->max_ctx;
  // every query row must fit a signed 32-bit TMA coordinate
  if (rows * kHeads >= ((uint64_t)1 << 31)) return SPARDA_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap mk, mv, mq;
  SPARDA_TRY(make_kv_map(&mk, L->k, rows));
  SPARDA_TRY(make_kv_map(&mv, L->v, rows));
  SPARDA_TRY(make_kv_map(&mq, q, rows * kHeads, 16));
  PrefillArgs a{nullptr, nullptr, static_cast<const __nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(out), seq_len,
                const_cast<int32_t*>(idx), const_cast<int32_t*>(cnt), nullptr, err, s->n_groups, w_cap(s),
                s->max_ctx, nb_cap(s), s->topk};
  launch_prefill_attn_tc(a, mq, mk, mv, batch, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}


// ------------------------------------------------------------------ cross-step block cache
int32_t sparda_prefetch_blocks_cached(const sparda_shape* s, const sparda_layer_kv* L, const int32_t* idx,
                                      const int32_t* cnt, const int32_t* seq_len, int32_t batch, void* cache_k,
                                      void* cache_v, int32_t* cache_blocks, int32_t n_cache, int32_t* slot,
                                      int32_t* fetch, unsigned long long* stats, int32_t n_ctas, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!L || !L->on_host) return SPARDA_ERR_INVALID_ARG;
  SPARDA_TRY(layer_status(L, true));
  if (!idx || !cnt || !seq_len || !cache_k || !cache_v || !cache_blocks || !slot || !fetch || n_ctas < 0 ||
      n_ctas > 4096)
    return SPARDA_ERR_INVALID_ARG;
  if (n_cache < kslots(s) || n_cache > 128) return SPARDA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(cache_k, 16) || !aligned(cache_v, 16) || !aligned(cache_blocks, 4) || !aligned(slot, 4) ||
      !aligned(fetch, 4) || !aligned(stats, 8))
    return SPARDA_ERR_MISALIGNED;
  int* err = dev_error_ptr();
  if (!err) return SPARDA_ERR_CUDA;
  CacheArgs a{static_cast<const __nv_bfloat16*>(L->k), static_cast<const __nv_bfloat16*>(L->v), idx, cnt, seq_len,
              cache_blocks, slot, fetch, stats, static_cast<__nv_bfloat16*>(cache_k),
              static_cast<__nv_bfloat16*>(cache_v), err, batch, s->n_groups, s->max_ctx, kslots(s), n_cache};
  launch_cache_gather(a, static_cast<cudaStream_t>(stream));   // one CTA per (b, g): n_ctas is not used
  return cuda_status(cudaGetLastError());
}

int32_t sparda_sparse_decode_attn_cached(const sparda_shape* s, const sparda_layer_kv* L, const void* cache_k,
                                         const void* cache_v, int32_t n_cache, const int32_t* slot, const void* q,
                                         const int32_t* idx, const int32_t* cnt, const int32_t* seq_len,
                                         int32_t batch, void* out, void* ws, size_t ws_bytes, void* stream) {
  if (!L || !L->on_host || !slot) return SPARDA_ERR_INVALID_ARG;
  if (n_cache < kslots(s) || n_cache > 128) return SPARDA_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(slot, 4)) return SPARDA_ERR_MISALIGNED;
  AttnArgs a;
  CUtensorMap mk, mv, hk, hv;
  SPARDA_TRY(prepare_attn(s, L, cache_k, cache_v, q, idx, cnt, seq_len, batch, out, ws, ws_bytes, &a, &mk, &mv,
                          &hk, &hv, n_cache));
  a.stage_slot = slot;
  a.stage_slots = n_cache;
  launch_sparse_attn(a, mk, mv, hk, hv, batch * s->n_groups, static_cast<cudaStream_t>(stream));
  return cuda_status(cudaGetLastError());
}


// ------------------------------------------------------------------ copy-engine gather
int32_t sparda_prefetch_blocks_copy_engine(const sparda_shape* s, const sparda_layer_kv* L, const int32_t* idx_host,
                                           const int32_t* cnt_host, const int32_t* seq_len_host, int32_t batch,
                                           void* staging_k, void* staging_v, int32_t* n_copies, void* stream) {
  SPARDA_TRY(shape_status(s));
  SPARDA_TRY(batch_status(s, batch));
  if (!L || !L->on_host) return SPARDA_ERR_INVALID_ARG;
  SPARDA_TRY(layer_status(L, true));
  if (!idx_host || !cnt_host || !seq_len_host || !staging_k || !staging_v) return SPARDA_ERR_INVALID_ARG;
  if (!aligned(staging_k, 16) || !aligned(staging_v, 16)) return SPARDA_ERR_MISALIGNED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ks = kslots(s);
  const size_t blk = (size_t)kBlock * kHeadDim * 2;                 // bytes of one block of K (or V)
  int copies = 0;
  for (int bg = 0; bg < batch * s->n_groups; ++bg) {
    const int T = seq_len_host[bg / s->n_groups];
    if (T < 1 || T > s->max_ctx) return SPARDA_ERR_INVALID_ARG;
    const int tb = (T - 1) / kBlock;
    const int n = cnt_host[bg] < 0 ? 0 : (cnt_host[bg] > ks ? ks : cnt_host[bg]);
    const int32_t* row = idx_host + (size_t)bg * ks;
    for (int sl = 0; sl < n;) {
      const int j = row[sl];
      if (j == 0 || j == tb) {
        ++sl;
        continue;
      }
      if (j < 0 || j > tb) return SPARDA_ERR_INVALID_ARG;
      // a run of consecutive blocks in consecutive slots is one contiguous range on both sides
      int e = sl + 1;
      while (e < n && row[e] == row[e - 1] + 1 && row[e] != tb) ++e;
      const size_t src = ((size_t)bg * s->max_ctx + (size_t)j * kBlock) * kHeadDim * 2;
      const size_t dst = ((size_t)bg * ks + sl) * blk;
      const size_t bytes = (size_t)(e - sl) * blk;
      SPARDA_TRY(cuda_status(cudaMemcpyAsync(static_cast<uint8_t*>(staging_k) + dst,
                                             static_cast<const uint8_t*>(L->k) + src, bytes, cudaMemcpyDefault, st)));
      SPARDA_TRY(cuda_status(cudaMemcpyAsync(static_cast<uint8_t*>(staging_v) + dst,
                                             static_cast<const uint8_t*>(L->v) + src, bytes, cudaMemcpyDefault, st)));
      copies += 2;
      sl = e;
    }
  }
  if (n_copies) *n_copies = copies;
  return SPARDA_OK;
}

}  // extern "C"
