// Compressed-key maintenance: storing a decode token's key/value and the mean-pooled keys of
// windows of kernel 32 / stride 16 (the inference-time key compression window of the
// techwalker article, section 四), one token at a time (decode).
//
// A window mean is the exact mean of 32 bf16 keys rounded once to bf16 (nearest, ties to
// even). The decode append sums each dimension exactly in a 64-bit fixed-point integer with
// 47 fractional bits and rounds that integer directly: every bf16 of magnitude in
// [2^-40, 2^11), and zero, converts without loss, and 32 of them cannot overflow. GB300
// issues float64 arithmetic at a small fraction of its integer rate, so the integer sum keeps
// the append short. A window holding any other value (a subnormal, a magnitude of 2^11 or
// more, a non-finite value) is summed in float64 instead, which is exact for bf16 keys of
// ordinary range, and rounded to bf16 without double rounding.
#pragma once

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

constexpr int kFixFrac = 47;          // fractional bits of the fixed-point window sums

// bf16 (given as its 16 bits) -> the integer x * 2^kFixFrac. Clears *in_range unless x is zero
// or of magnitude in [2^-40, 2^11) (biased exponent 87 .. 137), where the conversion is exact
// and the sum of 32 values stays below 2^63 in magnitude.
__device__ __forceinline__ long long bf16_to_fixed(uint32_t h, bool& in_range) {
  const int e = (int)((h >> 7) & 0xffu);
  const uint32_t m = h & 0x7fu;
  if (e == 0) {
    in_range = in_range && m == 0u;
    return 0;
  }
  in_range = in_range && e >= 87 && e <= 137;
  const int sh = min(max(e - 87, 0), 50);   // x = (128 + m) * 2^(e - 134)
  const long long v = (long long)(0x80u | m) << sh;
  return (h & 0x8000u) ? -v : v;
}

// bf16 bits of S * 2^-(kFixFrac + 5), rounded to nearest even: the mean of 32 values whose
// exact sum is S * 2^-kFixFrac (an exactly zero mean is +0).
__device__ __forceinline__ uint16_t fixed_mean_to_bf16(long long S) {
  if (S == 0) return 0u;
  const uint32_t sign = S < 0 ? 0x8000u : 0u;
  const unsigned long long A = S < 0 ? 0ull - (unsigned long long)S : (unsigned long long)S;
  const int p = 63 - __clzll((long long)A);      // A in [2^p, 2^(p+1))
  uint32_t m;                                    // the 8 leading bits, rounded: 128 .. 256
  if (p <= 7) {
    m = (uint32_t)(A << (7 - p));
  } else {
    const int sh = p - 7;
    m = (uint32_t)(A >> sh);
    const unsigned long long rem = A & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (m & 1u))) ++m;
  }
  // the mean is (m / 128) * 2^(p - 52); its biased exponent p - 52 + 127 lies in 75 .. 137.
  // m = 256 (rounded up to the next power of two) carries into the exponent.
  return (uint16_t)(sign + ((uint32_t)(p + 75) << 7) + (m - 128u));
}

// The append of sequence-group `bg` by 64 threads; thread t (0..63) owns dims 2t and 2t+1.
__device__ __forceinline__ void append_token(const AppendArgs& a, int bg, int t) {
  const int b = bg / a.G;
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
    bool in_range = true;
    long long S0 = bf16_to_fixed(kn & 0xffffu, in_range), S1 = bf16_to_fixed(kn >> 16, in_range);
#pragma unroll
    for (int u = 0; u < kWinKernel - 1; ++u) {
      S0 += bf16_to_fixed(xs[u] & 0xffffu, in_range);
      S1 += bf16_to_fixed(xs[u] >> 16, in_range);
    }
    uint32_t packed;
    if (in_range) {
      packed = (uint32_t)fixed_mean_to_bf16(S0) | ((uint32_t)fixed_mean_to_bf16(S1) << 16);
    } else {
      double s0 = 0.0 + bf16_lo(kn), s1 = 0.0 + bf16_hi(kn);    // an all-zero window gives +0
#pragma unroll
      for (int u = 0; u < kWinKernel - 1; ++u) {
        s0 += bf16_lo(xs[u]);
        s1 += bf16_hi(xs[u]);
      }
      const __nv_bfloat16 b0 = f64_to_bf16_rn(s0 / kWinKernel), b1 = f64_to_bf16_rn(s1 / kWinKernel);
      packed = (uint32_t)__bfloat16_as_ushort(b0) | ((uint32_t)__bfloat16_as_ushort(b1) << 16);
    }
    reinterpret_cast<uint32_t*>(a.ck + ((size_t)bg * a.W_cap + i) * kHeadDim)[t] = packed;
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

}  // namespace sparda
