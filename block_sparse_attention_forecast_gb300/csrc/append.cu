// Compressed-key maintenance launches: the decode append (append_body.cuh) and the
// compression of a whole cache (after a prefill).
#include "append_body.cuh"

namespace sparda {

// One CTA per (sequence, group), 64 threads.
__global__ void __launch_bounds__(64) append_kv_kernel(AppendArgs a) {
  grid_dep_launch();                   // the attention may start its prologue
  append_token(a, blockIdx.x, threadIdx.x);
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
