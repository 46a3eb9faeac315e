/*
 * sparda.h -- C ABI of the forecast-driven block-sparse decode step (libsparda.so).
 *
 * SparDA ("SparDA: Sparse Decoupled Attention for Efficient Long-Context LLM Inference", as
 * described by three web pages: a bittide.aicompass.dev thread with the translated
 * abstract, the techwalker.com article "NVIDIA与MIT联手：让超长文本AI助手的'记忆搜索'快了5倍多"
 * and the 10100.com piece "不是我硬件不好 是你软件架构有硬伤") adds a fourth projection, the
 * Forecast, to every attention layer. Layer L's forecast picks the KV blocks that layer L+1
 * will attend, so those blocks can be fetched from host memory while layer L still runs.
 * This library implements one layer's decode-step pieces as CUDA kernels for sm_103a:
 *
 *   sparda_append_kv           store the new token's K/V, maintain the compressed keys
 *   sparda_compress_keys       build every compressed key of a cache at once (prefill)
 *   sparda_forecast_project    the forecast projection (one 128-wide head per KV group)
 *   sparda_forecast_select     forecast scoring + max-pool onto blocks + top-k
 *   sparda_sparse_decode_attn  block-sparse GQA decode attention over the selection
 *   sparda_prefetch_blocks     gather of selected blocks from pinned host memory (UVA)
 *   sparda_multihead_select    the baseline query-driven selector, for comparison
 *
 * Conventions shared by every call
 *   - All tensors are caller-owned. The library never allocates, frees or synchronises on
 *     these calls; kernels are enqueued on the stream given (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and the call returns at once.
 *   - bf16 means IEEE bfloat16 stored as 16-bit words. All layouts are dense, row-major,
 *     innermost dimension last.
 *   - B = batch (sequences), G = KV groups (KV heads), H = query heads per group,
 *     d = head dimension. Query head h belongs to group h / H.
 *   - seq_len is a DEVICE int32 array [B]: seq_len[b] = T, the number of tokens of
 *     sequence b's context INCLUDING the current decode token, which sits at position T-1.
 *     1 <= T <= shape->max_ctx is required; a sequence outside that range produces no
 *     output (cnt = 0, idx = -1, zero attention output) and sets SPARDA_DEV_BAD_SEQ_LEN in
 *     the device error word.
 *   - Pointers must be 16-byte aligned (KV caches, staging and hot buffers 1024-byte
 *     aligned); a violation returns SPARDA_ERR_MISALIGNED before anything is launched.
 *   - Every argument check is synchronous and happens before any launch. Errors inside a
 *     kernel (a bounded wait that ran out, an out-of-range seq_len or block index) never
 *     trap: the kernel skips the bad access, ORs a bit into a device-side error word and
 *     returns. sparda_device_error() reads that word.
 *   - Workspaces: calls that take a workspace need sparda_workspace_bytes() bytes of
 *     device memory, zero-filled before their first use (cudaMemset). Every call leaves
 *     the workspace's counters at zero again, so it can be reused without clearing.
 *     Two calls that may run at the same time must not share a workspace.
 *   - The library looks up the device address of its own device variables (the error word,
 *     the allocation-free entry's scratch) once per device and keeps it for the life of the
 *     process. A cudaDeviceReset() unloads the library's device code, which may come back at
 *     another address: do not call into the library after resetting a device it has used.
 */
#ifndef SPARDA_H_
#define SPARDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
#define SPARDA_OK                        0
#define SPARDA_ERR_INVALID_ARG          -1  /* null pointer, negative or zero size        */
#define SPARDA_ERR_UNSUPPORTED_SHAPE    -2  /* a shape this build does not support         */
#define SPARDA_ERR_MISALIGNED           -3  /* pointer alignment rule broken               */
#define SPARDA_ERR_NOT_MAPPED_HOST      -4  /* host KV not reachable by the device (UVA)   */
#define SPARDA_ERR_WORKSPACE_TOO_SMALL  -5
#define SPARDA_ERR_CUDA                 -6  /* a CUDA runtime/driver call failed           */
#define SPARDA_ERR_STATIC_SCRATCH_LIMIT -7  /* beyond the allocation-free entry's scratch  */

/* bits of the device error word (sparda_device_error) */
#define SPARDA_DEV_WAIT_TIMEOUT   1   /* a bounded wait on a copy's completion ran out      */
#define SPARDA_DEV_BAD_SEQ_LEN    2   /* seq_len[b] outside [1, max_ctx]                    */
#define SPARDA_DEV_BAD_INDEX      4   /* a block index outside the sequence's blocks        */

/* workspace kinds for sparda_workspace_bytes */
#define SPARDA_WS_SELECT      1
#define SPARDA_WS_ATTN        2
#define SPARDA_WS_MULTIHEAD   3
#define SPARDA_WS_PREFILL     4

/* ---------------------------------------------------------------- shapes */
/*
 * The decode-step geometry. This build supports head_dim 128, heads_per_group 16, block 64,
 * win_kernel 32, win_stride 16 (the compression window the techwalker article, section 四,
 * gives for inference), 1 <= topk <= 62, max_ctx a multiple of 64 up to 262144, any
 * n_groups >= 1 and max_batch >= 1. max_batch sizes the caches (their outer dimension);
 * a call may use any batch <= max_batch.
 */
typedef struct sparda_shape {
  int32_t n_groups;         /* G: KV groups (KV heads) of the layer                          */
  int32_t heads_per_group;  /* H: query heads sharing one KV head                            */
  int32_t head_dim;         /* d                                                             */
  int32_t block;            /* tokens per KV block                                           */
  int32_t win_kernel;       /* tokens per compression window                                 */
  int32_t win_stride;       /* stride between compression windows                            */
  int32_t topk;             /* scored blocks kept on top of block 0 and the tail block       */
  int32_t max_ctx;          /* token capacity per sequence                                   */
  int32_t max_batch;        /* sequence capacity of the caches                               */
} sparda_shape;

/*
 * One layer's KV state. W_cap = (max_ctx - win_kernel) / win_stride + 1 compressed-key
 * slots per sequence and group.
 *
 *   k, v   bf16 [max_batch, G, max_ctx, d]. Resident layer (on_host = 0): device memory.
 *          Offloaded layer (on_host = 1): pinned host memory allocated or registered with
 *          the mapped flag; pass the DEVICE pointer of that memory (cudaHostGetDevicePointer,
 *          equal to the host pointer under UVA). It holds every complete block.
 *   ck     bf16 [max_batch, G, W_cap, d], device memory (always resident): ck[.., i, :] is the
 *          mean of keys 16i .. 16i+31 rounded to bf16.
 *   hot_k, hot_v
 *          offloaded layers only (NULL otherwise): bf16 [max_batch, G, 3, block, d] device
 *          memory. Slot 0 holds block 0; the block j >= 1 that holds the newest token lives
 *          in slot 1 + (j & 1), and the block before it in the other of slots 1 and 2. The
 *          attention reads block 0 and the tail block from here, never from host memory.
 */
typedef struct sparda_layer_kv {
  void* k;
  void* v;
  void* ck;
  void* hot_k;
  void* hot_v;
  int32_t on_host;
  int32_t reserved;
} sparda_layer_kv;

/* ---------------------------------------------------------------- utilities */
int32_t sparda_abi_version(void);
const char* sparda_status_string(int32_t status);

/* SPARDA_OK if this build supports the shape, else SPARDA_ERR_UNSUPPORTED_SHAPE. */
int32_t sparda_check_shape(const sparda_shape* shape);

/* Bytes of workspace the call of the given kind (SPARDA_WS_*) needs for `batch`
 * sequences; 0 for an unsupported shape. */
size_t sparda_workspace_bytes(const sparda_shape* shape, int32_t batch, int32_t kind);

/* Byte offset, inside a SPARDA_WS_SELECT workspace, of its block scores: float32
 * [max_batch * G][max_ctx / 64], row b*G + g holding S[j] of (b, g). sparda_forecast_select,
 * sparda_forecast_score and sparda_attend_and_score leave the scores there, and
 * sparda_decode_prologue's top-k reads them, so a caller may inspect them or write its own
 * for the top-k to select from (entries j >= (T-1)/64 + 1 are not read for selection).
 * 0 for an unsupported shape. */
size_t sparda_block_scores_offset(const sparda_shape* shape);

/* Reads the device error word (bits SPARDA_DEV_*) of the current device into *flags and,
 * if clear != 0, resets it. Synchronous: waits for all work on the device. */
int32_t sparda_device_error(int32_t* flags, int32_t clear);

/* The stream-ordered status read: enqueues on `stream` (a cudaStream_t as void*) a one-thread
 * kernel that writes the device error word (bits SPARDA_DEV_*) into *dev_flag and, if
 * clear != 0, resets the word in the same atomic step. dev_flag: 4-byte aligned device memory,
 * or pinned host memory mapped into the device's address space (its device address equals
 * its host address). Nothing waits on the host: the value covers every kernel ordered before
 * this call in `stream` (and any other work the device had finished); read *dev_flag after
 * synchronising with the stream or with an event recorded behind the call. The call may be
 * captured into a CUDA graph. Errors: SPARDA_ERR_INVALID_ARG (null), SPARDA_ERR_MISALIGNED,
 * SPARDA_ERR_NOT_MAPPED_HOST (memory the device cannot address as given). */
int32_t sparda_get_device_status(int32_t* dev_flag, int32_t clear, void* stream);

/* Copy-CTA count the gather uses by default for a batch: 64 below batch 32, 152 (one per
 * GB300 SM) from 32 on. The techwalker article (section 三) uses 16 / 32 copy CTAs on H100;
 * the same batch-adaptive rule was re-measured here for this library's copy CTAs, which are
 * small enough (128 threads, no shared memory) to share an SM with the compute kernels:
 * while the selection and attention run beside it, the gather needs about 100 or more of
 * them to keep the host link saturated, at almost no cost to the compute. */
int32_t sparda_prefetch_default_ctas(int32_t batch);

/* ---------------------------------------------------------------- the decode step */

/*
 * sparda_append_kv -- store the current token's key and value and keep the compressed keys
 * up to date as tokens arrive (compression window kernel 32 / stride 16, techwalker §四).
 *
 * k_new, v_new: device bf16 [B, G, d]. For every sequence b (T = seq_len[b]) the token is
 * written at position T-1. When T >= 32 and (T - 32) % 16 == 0 a window completes and
 * ck[b, g, (T-32)/16, :] = bf16(mean of keys T-32 .. T-1) is written: the exact mean rounded
 * once to bf16, nearest even. Each dimension's window sum is formed exactly in a 64-bit
 * fixed-point integer (47 fractional bits) when every key of the window is zero or of
 * magnitude in [2^-40, 2^11); otherwise in float64, rounded to bf16 through a round-to-odd
 * float32 so that no double rounding occurs. Both give the same bf16 code as the exact mean.
 * Offloaded layers: the token goes to the hot tail slot; when it fills its block (T % 64
 * == 0) that block is also written to the host cache, so that a later gather finds it.
 */
int32_t sparda_append_kv(const sparda_shape* shape, const sparda_layer_kv* layer,
                         const void* k_new, const void* v_new, const int32_t* seq_len,
                         int32_t batch, void* stream);

/*
 * sparda_compress_keys -- write every compressed key that is complete within the first
 * seq_len[b] tokens of the cache (windows i < (T - 32) / 16 + 1), as sparda_append_kv would
 * have written them one by one. Used after a prefill. Offloaded layers read the keys from
 * the host cache over the host link (slow; a set-up step).
 */
int32_t sparda_compress_keys(const sparda_shape* shape, const sparda_layer_kv* layer,
                             const int32_t* seq_len, int32_t batch, void* stream);

/*
 * sparda_forecast_project -- the Forecast projection, the fourth per-layer projection
 * (bittide thread; techwalker §二): f[b, r] = bf16(sum_c W[r, c] * h[b, c]).
 *
 * W: device bf16 [rows, hidden] (rows = G * d: row g*d + c is component c of group g's
 * forecast head); h: device bf16 [batch, hidden]; f: device bf16 [batch, rows], i.e.
 * [batch, G, d]. Products and sums in float32 (tensor cores), output rounded to nearest
 * even. rows must be a multiple of 8 and hidden a multiple of 32.
 */
int32_t sparda_forecast_project(const void* W, const void* h, int32_t rows, int32_t hidden,
                                int32_t batch, void* f, void* stream);

/*
 * sparda_forecast_select -- the Forecast selector (bittide thread: one forecast head per
 * GQA group and no softmax; techwalker §二; 10100 "SparDA 的解法"), for the target layer
 * whose compressed keys are `ck` (layer L+1 under lookahead, layer 0 for its same-layer
 * forecast, techwalker §三).
 *
 * For each (b, g), with T = seq_len[b], tb = (T-1)/64 and W = the windows complete within
 * the first T-1 tokens (the current token's window does not exist yet in the target layer):
 *   s[i] = sum_c f[b,g,c] * ck[b,g,i,c]          (float32, i < W; no softmax, no scale)
 *   S[j] = max { s[i] : window i overlaps block j }   (windows 4j-1 .. 4j+3)
 *   chosen = the topk highest S[j] over 1 <= j < tb (ties -> lower j; -0 and +0 are equal
 *            scores; an infinity ranks above or below every finite score; a NaN score, which
 *            only inputs whose float32 products or sums overflow can produce, ranks above
 *            every number, all NaNs alike, and is still counted as a candidate)
 * Output idx: int32 [B, G, topk+2], the blocks {0, tb} U chosen sorted ascending, then -1
 * padding; cnt: int32 [B, G], the number of valid entries (min(topk, tb-1) + 2, or 1 when
 * tb = 0). forecast: device bf16 [B, G, d]. workspace: SPARDA_WS_SELECT.
 * Ordering: the call begins while the kernel before it in the stream still runs
 * (programmatic dependent launch). Its compressed-key loads do not wait for that kernel;
 * everything else (the forecast, seq_len, the workspace, idx, cnt) does. So the kernel just
 * before this call in the stream must not write the compressed keys it scores (the windows
 * i < W of every sequence). sparda_append_kv of the same layer writes only the window the
 * current token completes, which is not scored, and sparda_forecast_project writes only the
 * forecast: both may come just before it.
 */
int32_t sparda_forecast_select(const sparda_shape* shape, const void* ck, const void* forecast,
                               const int32_t* seq_len, int32_t batch, int32_t* idx,
                               int32_t* cnt, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * sparda_forecast_score -- sparda_forecast_select without its top-k: the block scores S[j]
 * (float32, j < (T-1)/64 + 1) are left in the workspace (SPARDA_WS_SELECT), for
 * sparda_decode_prologue's top-k (its ws_scores) to select from, as sparda_attend_and_score
 * leaves them. All SMs stream the compressed keys. Errors and the ordering rule (the
 * kernel just before this call must not write the compressed keys it scores): as
 * sparda_forecast_select.
 */
int32_t sparda_forecast_score(const sparda_shape* shape, const void* ck, const void* forecast,
                              const int32_t* seq_len, int32_t batch, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * sparda_sparse_decode_attn -- block-sparse GQA decode attention (bittide thread: the next
 * layer's own queries attend the selected blocks; techwalker §六: the sparse attention
 * itself is unchanged by SparDA). For every query head h of group g:
 *   o[b, g*H + h, :] = sum_t softmax_t(q . k_t / sqrt(d)) v_t
 * over the tokens t < T of the blocks idx[b, g, 0 .. cnt[b,g]-1].
 *
 * q: device bf16 [B, G*H, d]; out: device bf16 [B, G*H, d]; idx/cnt as produced by
 * sparda_forecast_select. Resident layer: K/V are read from the layer's cache. Offloaded
 * layer: staging_k / staging_v (device bf16 [max_batch, G, topk+2, 64, d], filled by
 * sparda_prefetch_blocks for the same idx) supply every selected block except block 0 and
 * the tail block, which come from the layer's hot buffers. QK^T and PV run on tensor cores
 * (bf16 operands, float32 accumulation); the softmax is float32. workspace: SPARDA_WS_ATTN
 * (partial results of (sequence, group)s split over several CTAs, and a counter per group,
 * zero between calls and left zero; when every group gets the same 2 to 8 CTAs, they form
 * one thread-block cluster and merge in distributed shared memory, and the workspace is
 * not touched).
 * Ordering: the call begins while the kernel before it in the stream still runs
 * (programmatic dependent launch) and reads nothing before that kernel has completed. It
 * lets the next launch in the stream begin as soon as it starts; every call of this library
 * that can begin that early waits for it to complete before touching its output, workspace
 * or error word. Such a following call may then also run beside the launch before this one:
 * between two sparda_attend_and_score calls, this call does not separate them (see there).
 */
int32_t sparda_sparse_decode_attn(const sparda_shape* shape, const sparda_layer_kv* layer,
                                  const void* staging_k, const void* staging_v, const void* q,
                                  const int32_t* idx, const int32_t* cnt,
                                  const int32_t* seq_len, int32_t batch, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparda_attend_and_select -- layer L's sparda_sparse_decode_attn and layer L+1's
 * sparda_forecast_select in one launch. Under lookahead the two are independent: layer L's
 * forecast exists when layer L attends (bittide thread; techwalker section 二). One
 * persistent grid of one CTA per SM is split between the two jobs in proportion to the
 * bytes each streams, so both run at once instead of one after the other.
 *
 * Arguments and results are exactly those of the two calls: (layer, staging_k, staging_v,
 * q, idx, cnt, out, ws_attn) as for sparda_sparse_decode_attn on layer L, and (ck_next,
 * forecast_next, idx_next, cnt_next, ws_sel) as for sparda_forecast_select on layer L+1's
 * compressed keys; seq_len and batch are shared. idx_next / cnt_next / ws_sel must be other
 * buffers than idx / cnt / ws_attn (SPARDA_ERR_INVALID_ARG otherwise).
 */
int32_t sparda_attend_and_select(const sparda_shape* shape, const sparda_layer_kv* layer,
                                 const void* staging_k, const void* staging_v, const void* q,
                                 const int32_t* idx, const int32_t* cnt, void* out, void* ws_attn,
                                 size_t ws_attn_bytes, const void* ck_next,
                                 const void* forecast_next, int32_t* idx_next, int32_t* cnt_next,
                                 void* ws_sel, size_t ws_sel_bytes, const int32_t* seq_len,
                                 int32_t batch, void* stream);

/*
 * The decode step as two launches per layer (a layer-pipelined split of the same work):
 *
 *   sparda_decode_prologue(L):   top-k of layer L's block scores -> idx[L], cnt[L]
 *                                append of layer L's token (as sparda_append_kv)
 *                                forecast for layer L+1 (as sparda_forecast_project)
 *   sparda_attend_and_score(L):  layer L's attention (as sparda_sparse_decode_attn) and the
 *                                block scores of layer L+1 (the selector's scoring and
 *                                max-pool, without its top-k)
 *
 * Under lookahead layer L's forecast scores layer L+1's blocks while layer L attends
 * (bittide thread; techwalker section 二); the top-k that turns those scores into layer
 * L+1's blocks only has to finish before layer L+1 attends, so it runs in layer L+1's
 * prologue beside that layer's append and projection instead of as a tail of layer L's
 * launch. Results are exactly those of the one-call-per-step entry points.
 */

/*
 * sparda_attend_and_score -- as sparda_attend_and_select, except that the selection half
 * stops after the block scores: for each (b, g) of layer L+1, S[j] (float32, the max-pooled
 * forecast scores, j < (T-1)/64 + 1) is left in ws_scores (a SPARDA_WS_SELECT workspace),
 * for sparda_decode_prologue of layer L+1 to select from. ws_scores must differ from
 * ws_attn (SPARDA_ERR_INVALID_ARG otherwise). l2_next (optional, NULL for none; 16-byte
 * aligned, l2_next_bytes a multiple of 16) names device memory that the next launches will
 * read, such as layer L+1's forecast weights for its prologue: the selection CTAs pull it
 * into L2 after issuing their last load. It changes no result. Every CTA lets the next
 * launch in the stream begin as soon as it starts (programmatic dependent launch), so a
 * following sparda_decode_prologue's projection starts on the SMs that finished CTAs free.
 * A run of these calls (or of sparda_attend_and_select) directly after one another in a
 * stream therefore overlaps: as many as fit on the GPU may run at once, so give each call of
 * such a run its own ws_scores (the selection's work queue lives there; ws_attn may be
 * shared); a sparda_sparse_decode_attn between two calls, which also lets the next launch
 * begin at once, counts as no separation. With a sparda_decode_prologue between two calls,
 * as in the decode step, the second begins only after the first has completed, and two
 * workspaces alternating suffice.
 */
int32_t sparda_attend_and_score(const sparda_shape* shape, const sparda_layer_kv* layer,
                                const void* staging_k, const void* staging_v, const void* q,
                                const int32_t* idx, const int32_t* cnt, void* out, void* ws_attn,
                                size_t ws_attn_bytes, const void* ck_next, const void* forecast_next,
                                void* ws_scores, size_t ws_scores_bytes, const void* l2_next,
                                size_t l2_next_bytes, const int32_t* seq_len, int32_t batch, void* stream);

/*
 * sparda_decode_prologue -- the small per-layer jobs of layer L in one launch:
 *   - if ws_scores != NULL: the top-k of the block scores that sparda_attend_and_score left
 *     there for this layer, written to idx / cnt exactly as sparda_forecast_select writes
 *     them (block 0, the tail block and the topk best others; ties to the lower block);
 *   - the append of k_new / v_new (device bf16 [B, G, d]) to `layer`, exactly as
 *     sparda_append_kv;
 *   - if W_next != NULL: forecast_next = bf16(W_next . h) for layer L+1, exactly as
 *     sparda_forecast_project with rows = G*d (W_next: device bf16 [G*d, hidden] row-major,
 *     h: device bf16 [B, hidden], forecast_next: device bf16 [B, G, d]; hidden a multiple of
 *     32).
 * The three jobs read and write disjoint buffers. Only the top-k waits for the previous
 * kernel in the stream to complete (the append waits too when ws_scores is NULL). The
 * projection and the append do not: when that kernel is sparda_attend_and_score or
 * sparda_attend_and_select (which let the next launch begin once all their CTAs run), they
 * run on the SMs it releases, beside its last CTAs. So the kernel just before this launch in
 * the stream must not write W_next, h, k_new or v_new, nor read forecast_next, the layer's
 * key/value at position T-1 or its compressed key of the window the token completes
 * (sparda_attend_and_score of the layer before reads only the windows below it). Errors:
 * as the three separate calls.
 */
int32_t sparda_decode_prologue(const sparda_shape* shape, const sparda_layer_kv* layer,
                               const void* k_new, const void* v_new, const void* ws_scores,
                               size_t ws_scores_bytes, int32_t* idx, int32_t* cnt, const void* W_next,
                               const void* h, int32_t hidden, void* forecast_next,
                               const int32_t* seq_len, int32_t batch, void* stream);

/*
 * sparda_prefetch_blocks -- the gather that hides the host-offload copy (bittide thread:
 * the next layer's blocks are fetched on a separate CUDA stream while the current layer
 * computes; techwalker §三: a persistent kernel with a few copy CTAs reads host memory
 * directly over unified virtual addressing, 16 CTAs below batch 32 and 32 from 32 on).
 *
 * For every (b, g) and slot s < cnt[b,g] whose block j = idx[b,g,s] is neither block 0 nor
 * the tail block, copies block j of the offloaded layer's host k and v into slot s of
 * staging_k / staging_v (device bf16 [max_batch, G, topk+2, 64, d]). n_ctas = 0 picks
 * sparda_prefetch_default_ctas(batch); any count from 1 to 4096 is allowed. Enqueue it on a side stream after an event recorded
 * behind the select call, and make the attention wait on an event recorded behind it.
 */
int32_t sparda_prefetch_blocks(const sparda_shape* shape, const sparda_layer_kv* layer,
                               const int32_t* idx, const int32_t* cnt, const int32_t* seq_len,
                               int32_t batch, void* staging_k, void* staging_v,
                               int32_t n_ctas, void* stream);

/*
 * sparda_copy -- a device-side copy of `bytes` bytes from src to dst, where each of them is
 * device memory or pinned host memory mapped into the device's address space (its device
 * address equals its host address). It serves the decode step's host I/O: the step's first
 * inputs in and its last outputs out, on the compute stream, where a DMA copy's start-up
 * latency (tens of microseconds on the host link) would sit on the critical path. Not an
 * operation of the pages: plumbing around the step.
 *
 * dst and src 16-byte aligned, bytes a positive multiple of 16, the ranges not overlapping.
 * Errors: SPARDA_ERR_INVALID_ARG (null pointer, zero or non-multiple-of-16 size),
 * SPARDA_ERR_MISALIGNED, SPARDA_ERR_NOT_MAPPED_HOST (a pointer the device cannot address as
 * given: pageable host memory, or pinned memory whose device address differs).
 */
int32_t sparda_copy(void* dst, const void* src, size_t bytes, void* stream);

/*
 * sparda_multihead_select -- the baseline query-driven selector the pages compare against
 * (bittide thread; 10100 "先把痛点讲透"): every query head of the group scores every
 * compressed key (scale 1/sqrt(d)), a softmax per head over the windows, a sum over the
 * group's heads, then the same max-pool and top-k as sparda_forecast_select.
 * q: device bf16 [B, G*H, d]. Outputs as sparda_forecast_select. workspace:
 * SPARDA_WS_MULTIHEAD.
 */
int32_t sparda_multihead_select(const sparda_shape* shape, const void* ck, const void* q,
                                const int32_t* seq_len, int32_t batch, int32_t* idx,
                                int32_t* cnt, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * sparda_forecast_select_static -- sparda_forecast_select without a workspace argument, for
 * callers that cannot allocate device memory: a plugin that its host engine hands only the
 * input and output tensors, or a serving loop that must not allocate once it runs. The
 * pages have no counterpart; this is a convenience of this library.
 *
 * Same inputs, outputs and results as sparda_forecast_select. Its scratch (per-group
 * counters and block scores) is a fixed array of SPARDA_STATIC_SCRATCH_BYTES in the
 * library's own device memory, which every device that loads the library holds until the
 * process exits. It serves batch * n_groups <= SPARDA_STATIC_MAX_GROUPS and
 * 4 * SPARDA_STATIC_MAX_GROUPS + 4 * batch * n_groups * (max_ctx / 64) <=
 * SPARDA_STATIC_SCRATCH_BYTES (for example batch 64, 2 groups, max_ctx 131072); larger
 * requests return SPARDA_ERR_STATIC_SCRATCH_LIMIT without launching anything.
 * The first call on a device looks up the array's device address (make that first call
 * before any stream capture). Each call clears the counters with an asynchronous memset on
 * `stream` and allocates nothing. All calls share the one array, which keeps the last
 * call's contents: calls that may overlap on the GPU (other streams, other threads) race
 * and must be serialized by the caller.
 */
#define SPARDA_STATIC_SCRATCH_BYTES (4 << 20)
#define SPARDA_STATIC_MAX_GROUPS 4096
int32_t sparda_forecast_select_static(const sparda_shape* shape, const void* ck,
                                      const void* forecast, const int32_t* seq_len,
                                      int32_t batch, int32_t* idx, int32_t* cnt, void* stream);

/*
 * sparda_prefetch_blocks_copy_engine -- the gather of sparda_prefetch_blocks done by the
 * copy engines instead of copy CTAs, for comparison: one cudaMemcpyAsync on `stream` per run
 * of consecutive selected blocks (K and V separately), into the same staging layout. The
 * selection must be on the HOST (idx_host int32 [B, G, topk+2], cnt_host int32 [B, G],
 * seq_len_host int32 [B]): the caller reads it back from the device and waits for it first,
 * which is the host-side indexing step the pages contrast SparDA with (techwalker section 五,
 * the InfiniGen paragraph); the GPU-side gather needs no such round trip. *n_copies (optional)
 * receives the number of copies issued. Host-synchronous argument checks; the copies are
 * asynchronous. Errors: as sparda_prefetch_blocks, plus SPARDA_ERR_INVALID_ARG for a host
 * seq_len or block index out of range (checked before each copy is issued) and
 * SPARDA_ERR_CUDA if a copy cannot be enqueued.
 */
int32_t sparda_prefetch_blocks_copy_engine(const sparda_shape* shape, const sparda_layer_kv* host_layer,
                                           const int32_t* idx_host, const int32_t* cnt_host,
                                           const int32_t* seq_len_host, int32_t batch, void* staging_k,
                                           void* staging_v, int32_t* n_copies, void* stream);

/* ---------------------------------------------------------------- cross-step block cache */
/*
 * An extension beyond the pages, for offloaded layers: consecutive decode steps often select
 * many of the same blocks, so each (b, g) of an offloaded layer keeps the blocks it gathered
 * in n_cache slots of HBM (topk + 2 <= n_cache <= 128), and only the selected blocks not held
 * there yet are read over the host link. The caller owns, per offloaded layer:
 *   cache_k, cache_v  device bf16 [max_batch, G, n_cache, 64, d] (the cached blocks);
 *   cache_blocks      device int32 [max_batch, G, n_cache]: the block each slot holds, -1 for
 *                     none. Fill with -1 before the first call (or after the layer's cache
 *                     content stops being valid, e.g. a new prompt in that sequence slot);
 *   slot              device int32 [B, G, topk+2]: written by the gather, read by the attention;
 *   fetch             device int32 [max_batch, G, n_cache]: scratch of the gather.
 */

/*
 * sparda_prefetch_blocks_cached -- sparda_prefetch_blocks with the block cache. For every
 * (b, g), a selected block (other than block 0 and the tail block, which the hot buffers
 * hold) already held in a slot keeps it; each other selected block, in idx order, takes the
 * lowest slot whose block is not selected now, and is copied there from the host cache.
 * slot[b, g, s] receives the cache slot of idx entry s (-1 for block 0, the tail block and
 * padding). stats (optional, NULL for none; device uint64 [2], 8-byte aligned) accumulates
 * the hits and the misses (blocks copied). One launch of one CTA per (b, g): the CTA assigns
 * its group's slots and copies its group's misses itself (four copy streams of 128 threads),
 * so the number of copy CTAs follows the batch; n_ctas is checked as for
 * sparda_prefetch_blocks (0 .. 4096) but not used.
 * Errors: as sparda_prefetch_blocks; SPARDA_ERR_UNSUPPORTED_SHAPE for n_cache out of range.
 */
int32_t sparda_prefetch_blocks_cached(const sparda_shape* shape, const sparda_layer_kv* host_layer,
                                      const int32_t* idx, const int32_t* cnt, const int32_t* seq_len,
                                      int32_t batch, void* cache_k, void* cache_v, int32_t* cache_blocks,
                                      int32_t n_cache, int32_t* slot, int32_t* fetch, unsigned long long* stats,
                                      int32_t n_ctas, void* stream);

/*
 * sparda_sparse_decode_attn_cached -- sparda_sparse_decode_attn of an offloaded layer whose
 * selected blocks sit in the block cache: the block of idx entry s is read from slot
 * slot[b, g, s] of cache_k / cache_v (as sparda_prefetch_blocks_cached left them), block 0
 * and the tail block from the hot buffers. Results are those of sparda_sparse_decode_attn on
 * the same blocks, bit for bit. A slot outside 0 .. n_cache-1 sets SPARDA_DEV_BAD_INDEX and
 * reads slot 0.
 */
int32_t sparda_sparse_decode_attn_cached(const sparda_shape* shape, const sparda_layer_kv* layer,
                                         const void* cache_k, const void* cache_v, int32_t n_cache,
                                         const int32_t* slot, const void* q, const int32_t* idx,
                                         const int32_t* cnt, const int32_t* seq_len, int32_t batch, void* out,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- chunked prefill */
/*
 * Prefill processes a whole prompt. The pages give its figures (bittide thread and abstract:
 * up to 1.25x faster prefill than the sparse offload baseline; techwalker section 五: in
 * prefill the block-sparse attention dominates, the block selection grows with the context
 * and nears it at 128K, and the Forecast indexer cuts the selection cost by up to 2.5x while
 * the attention is unchanged; 10100 "SparDA 的解法": in prefill all keys are already on the
 * GPU, so only the cheaper selection helps) but not the prefill selection itself. This
 * library takes these readings:
 *   - the prompt is split into chunks of 64 query tokens; chunk c = tokens 64c .. 64c+63
 *     (the last chunk of a sequence may be shorter), n_chunks = ceil(T / 64);
 *   - the tokens of a chunk share one selection: block 0, the chunk's own block c, and the
 *     topk best of blocks 1 .. c-1, ties to the lower block, ascending, -1 padded, scored
 *     over the compressed keys complete before the chunk (windows i < (64c - 32) / 16 + 1);
 *   - every token attends its chunk's blocks up to its own position (causal in block c).
 * Per-chunk outputs: idx int32 [B, G, max_ctx/64, topk+2] and cnt int32 [B, G, max_ctx/64]
 * (row c of (b, g) for chunk c; chunks past the prompt get cnt 0 and idx -1). seq_len[b] is
 * the prompt length T (1 <= T <= max_ctx). The compressed keys must hold every window of the
 * prompt (sparda_compress_keys with seq_len = T). workspace: SPARDA_WS_PREFILL (float32
 * block scores [max_batch * G, max_ctx/64, max_ctx/64]: 16 MiB per sequence-group at
 * max_ctx 131072; no zero-fill needed). The calls wait for the kernel before them in the
 * stream to finish (no programmatic overlap).
 */

/*
 * sparda_prefill_forecast_select -- the Forecast selector on prefill chunks: window i of
 * chunk c scores sum over the chunk's tokens t of f_t . ck_i (the decode score summed over
 * the chunk, no softmax, no scale), max-pooled onto blocks as in decode. forecast: device
 * bf16 [max_batch, max_ctx, G, d], the per-token forecast vectors (the fourth projection of
 * the prompt's hidden states, one head per group). The chunk's forecasts are summed in
 * float32 and the dot products run in float32.
 */
int32_t sparda_prefill_forecast_select(const sparda_shape* shape, const void* ck, const void* forecast,
                                       const int32_t* seq_len, int32_t batch, int32_t* idx, int32_t* cnt,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparda_prefill_multihead_select -- the baseline query-driven selector on prefill chunks:
 * every (token, head) query of the chunk gets its own softmax over the windows before the
 * chunk (logits scaled by 1/sqrt(d)), and the probabilities are summed over the chunk's
 * tokens and the group's heads; then the same max-pool and top-k. q: device bf16
 * [max_batch, max_ctx, G*H, d]. The logits run on tensor cores (tcgen05: bf16 operands,
 * float32 accumulation); the softmax and the sums are float32, the sums over rows in a
 * fixed order (the result does not vary from call to call). SPARDA_ERR_UNSUPPORTED_SHAPE
 * when max_batch * G * max_ctx * H reaches 2^31 (a query row's TMA coordinate).
 */
int32_t sparda_prefill_multihead_select(const sparda_shape* shape, const void* ck, const void* q,
                                        const int32_t* seq_len, int32_t batch, int32_t* idx, int32_t* cnt,
                                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * sparda_prefill_attn -- causal block-sparse prefill attention of a resident layer: for
 * every token t of chunk c and query head h of group g,
 *   out[b, t, g*H + h, :] = sum_u softmax_u(q[b, t, g*H + h] . k_u / sqrt(d)) v_u
 * over the tokens u <= t of the blocks idx[b, g, c, 0 .. cnt[b, g, c]-1] (as the prefill
 * selectors write them; a block index outside 0 .. c sets SPARDA_DEV_BAD_INDEX and reads
 * block 0 instead). q, out: device bf16 [max_batch, max_ctx, G*H, d]; the layer's k, v hold
 * the prompt's keys and values. QK^T and PV on tensor cores (bf16 operands, float32
 * accumulation), float32 softmax. SPARDA_ERR_INVALID_ARG for an offloaded layer.
 */
int32_t sparda_prefill_attn(const sparda_shape* shape, const sparda_layer_kv* layer, const void* q,
                            const int32_t* idx, const int32_t* cnt, const int32_t* seq_len, int32_t batch,
                            void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPARDA_H_ */
