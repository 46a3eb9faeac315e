// Compressed-key maintenance: storing a decode token's key/value and the mean-pooled keys of
// windows of kernel 32 / stride 16 (the inference-time key compression window of the
// techwalker article, section 四), either one token at a time (decode) or for a whole cache
// (after a prefill).
//
// Window means are summed in float64: for bf16 keys of ordinary range the sum of 32 keys is
// exact there, so the mean, and its bf16 rounding, does not depend on the order of the sum.
#include "common.cuh"
#include "kernels.h"

namespace sparda {

// Key `tok` of sequence-group `bg`, for the resident cache or an offloaded layer (where
// block 0 and the two newest blocks live in the hot ring, older blocks in host memory).
__device__ __forceinline__ uint32_t load_key2(const __nv_bfloat16* k, const __nv_bfloat16* hot_k,
                                              int on_host, size_t bg, int max_ctx, int tb,
                                              int tok, int dim2) {
  const __nv_bfloat16* row;
  const int j = tok / kBlock;
  if (!on_host || !(j == 0 || j == tb || j == tb - 1)) {
    row = k + ((bg * max_ctx) + tok) * kHeadDim;
  } else {
    row = hot_k + ((bg * kHotSlots + hot_slot(j)) * kBlock + (tok % kBlock)) * kHeadDim;
  }
  return reinterpret_cast<const uint32_t*>(row)[dim2];
}

// One CTA per (sequence, group), 64 threads, thread t owns dims 2t and 2t+1.
__global__ void __launch_bounds__(64) append_kv_kernel(AppendArgs a) {
  grid_dep_launch();                   // the attention may start its prologue
  const int bg = blockIdx.x;
  const int b = bg / a.G;
  const int t = threadIdx.x;
  const int T = a.seq_len[b];
  if (T < 1 || T > a.max_ctx) {
    if (t == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int p = T - 1;
  const int tb = p / kBlock;
  const uint32_t kn = reinterpret_cast<const uint32_t*>(a.k_new + (size_t)bg * kHeadDim)[t];
  const uint32_t vn = reinterpret_cast<const uint32_t*>(a.v_new + (size_t)bg * kHeadDim)[t];
  if (!a.on_host) {
    const size_t off = ((size_t)bg * a.max_ctx + p) * kHeadDim;
    reinterpret_cast<uint32_t*>(a.k + off)[t] = kn;
    reinterpret_cast<uint32_t*>(a.v + off)[t] = vn;
  } else {
    const size_t off = (((size_t)bg * kHotSlots + hot_slot(tb)) * kBlock + p % kBlock) * kHeadDim;
    reinterpret_cast<uint32_t*>(a.hot_k + off)[t] = kn;
    reinterpret_cast<uint32_t*>(a.hot_v + off)[t] = vn;
  }
  if (T >= kWinKernel && (T - kWinKernel) % kWinStride == 0) {
    const int i = (T - kWinKernel) / kWinStride;
    uint32_t xs[kWinKernel - 1];           // all loads in flight before the sums
#pragma unroll
    for (int u = 0; u < kWinKernel - 1; ++u)
      xs[u] = load_key2(a.k, a.hot_k, a.on_host, bg, a.max_ctx, tb, T - kWinKernel + u, t);
    double s0 = bf16_lo(kn), s1 = bf16_hi(kn);
#pragma unroll
    for (int u = 0; u < kWinKernel - 1; ++u) {
      s0 += bf16_lo(xs[u]);
      s1 += bf16_hi(xs[u]);
    }
    __nv_bfloat16* dst = a.ck + ((size_t)bg * a.W_cap + i) * kHeadDim + 2 * t;
    dst[0] = f64_to_bf16_rn(s0 / kWinKernel);
    dst[1] = f64_to_bf16_rn(s1 / kWinKernel);
  }
  // Offloaded layer: a block that just filled is written to the host cache, so that a
  // gather issued at a later step finds it there. Each thread copies its own two dims of
  // the 64 rows, which it wrote itself at earlier steps or just now.
  if (a.on_host && T % kBlock == 0) {
    const size_t src = ((size_t)bg * kHotSlots + hot_slot(tb)) * kBlock * kHeadDim;
    const size_t dst = ((size_t)bg * a.max_ctx + (size_t)tb * kBlock) * kHeadDim;
    const uint32_t* hk = reinterpret_cast<const uint32_t*>(a.hot_k + src);
    const uint32_t* hv = reinterpret_cast<const uint32_t*>(a.hot_v + src);
    uint32_t* ck = reinterpret_cast<uint32_t*>(a.k + dst);
    uint32_t* cv = reinterpret_cast<uint32_t*>(a.v + dst);
    for (int r = 0; r < kBlock; ++r) {
      ck[r * (kHeadDim / 2) + t] = hk[r * (kHeadDim / 2) + t];
      cv[r * (kHeadDim / 2) + t] = hv[r * (kHeadDim / 2) + t];
    }
  }
}

// grid (B*G, ceil(W_cap / kCompressWindows)), 64 threads; thread t owns dims 2t, 2t+1.
// Each CTA writes windows [i0, i1) from running half-window (16-token) sums, so that every
// key is read once.
constexpr int kCompressWindows = 64;

__global__ void __launch_bounds__(64) compress_keys_kernel(CompressArgs a) {
  const int bg = blockIdx.x;
  const int b = bg / a.G;
  const int t = threadIdx.x;
  const int T = a.seq_len[b];
  if (T < 1 || T > a.max_ctx) {
    if (t == 0 && blockIdx.y == 0) atomicOr(a.err, SPARDA_DEV_BAD_SEQ_LEN);
    return;
  }
  const int W = num_windows(T);
  const int tb = (T - 1) / kBlock;
  const int i0 = blockIdx.y * kCompressWindows;
  const int i1 = min(W, i0 + kCompressWindows);
  if (i0 >= i1) return;
  auto half_sum = [&](int h, double& s0, double& s1) {
    s0 = 0.0;
    s1 = 0.0;
    for (int tok = h * kWinStride; tok < (h + 1) * kWinStride; ++tok) {
      const uint32_t x = load_key2(a.k, a.hot_k, a.on_host, bg, a.max_ctx, tb, tok, t);
      s0 += bf16_lo(x);
      s1 += bf16_hi(x);
    }
  };
  double p0, p1;
  half_sum(i0, p0, p1);
  for (int i = i0; i < i1; ++i) {
    double n0, n1;
    half_sum(i + 1, n0, n1);
    __nv_bfloat16* dst = a.ck + ((size_t)bg * a.W_cap + i) * kHeadDim + 2 * t;
    dst[0] = f64_to_bf16_rn((p0 + n0) / kWinKernel);
    dst[1] = f64_to_bf16_rn((p1 + n1) / kWinKernel);
    p0 = n0;
    p1 = n1;
  }
}

void launch_append_kv(const AppendArgs& a, int bg_count, cudaStream_t s) {
  append_kv_kernel<<<bg_count, 64, 0, s>>>(a);
}

void launch_compress_keys(const CompressArgs& a, int bg_count, cudaStream_t s) {
  dim3 grid(bg_count, (a.W_cap + kCompressWindows - 1) / kCompressWindows);
  compress_keys_kernel<<<grid, 64, 0, s>>>(a);
}

}  // namespace sparda
