// fa_prologue.cu -- pre-attention prologue: RMS-norm of every query and key
// head vector, then the rotary mix with per-position factors, writing the Q
// and K tensors the attention forward reads; and its backward.
//
// What it computes is the modded-nanogpt page qkv_rope.py (module docstring
// and `_qk_norm_rope_forward_kernel`, without its paired-heads and key-offset
// options; the backward is the norm/rotary part of
// `_qkv_norm_rope_pack_fp8_backward_kernel` without the fp8 packing):
//
//   x = qk[t][c][:]            (c < hq: query head c, else key head c - hq)
//   rstd = 1 / sqrt(mean_d x_d^2 + 2^-23),  n = rstd x
//   y_d  = f1[t][d] n_d + f2[t][d] n_(d xor 1)
//   backward:  gn_e = f1[t][e] g_e + f2[t][e xor 1] g_(e xor 1)
//              dx_e = rstd (gn_e - n_e mean_d(gn_d n_d))
//
// Elementwise with one row reduction, bound by HBM: each lane holds D/32
// consecutive elements of a head row, so the partner of every element
// (d xor 1) sits in the same lane and the only cross-lane traffic is the row
// sums (warp shuffles).  fp32 arithmetic, 16-bit (bf16 or fp16) inputs and
// outputs, fp32 factors.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 256;
constexpr float kEps = 1.1920928955078125e-7f;  // 2^-23

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// E = D / 32 elements per lane: 2 (one pair) or 4 (two pairs).
template <int E>
struct alignas(E * 2) Vec16 {
  uint16_t v[E];
};
template <int E>
struct alignas(E * 4) VecF {
  float v[E];
};

// One warp per token: the token's factors are read once into registers and
// serve all hq + hk head rows, which lie contiguously in memory.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fa_qk_norm_rope_fwd_kernel(const T* __restrict__ qk,
                                                                       const float* __restrict__ f1,
                                                                       const float* __restrict__ f2,
                                                                       T* __restrict__ q, T* __restrict__ k,
                                                                       int tokens, int hq, int hk) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int heads = hq + hk;
  const long nwarps = static_cast<long>(gridDim.x) * (kThreads / 32);
  for (long t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < tokens; t += nwarps) {
    const VecF<E> a = *reinterpret_cast<const VecF<E>*>(f1 + t * D + lane * E);
    const VecF<E> s = *reinterpret_cast<const VecF<E>*>(f2 + t * D + lane * E);
#pragma unroll 4
    for (int c = 0; c < heads; ++c) {
      const Vec16<E> xr = *reinterpret_cast<const Vec16<E>*>(qk + (t * heads + c) * D + lane * E);
      float x[E];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        x[e] = to_f<T>(*reinterpret_cast<const T*>(&xr.v[e]));
        ss = fmaf(x[e], x[e], ss);
      }
      const float rstd = rsqrtf(warp_sum(ss) * (1.f / D) + kEps);
      Vec16<E> yr;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const T yt = from_f<T>(a.v[e] * (x[e] * rstd) + s.v[e] * (x[e ^ 1] * rstd));
        yr.v[e] = *reinterpret_cast<const uint16_t*>(&yt);
      }
      T* dst = c < hq ? q + (t * hq + c) * D : k + (t * hk + (c - hq)) * D;
      *reinterpret_cast<Vec16<E>*>(dst + lane * E) = yr;
    }
  }
}

// Backward: one warp per (token, head) row.  With two dependent row sums per
// row, independent warps hide latency better than sharing the factors across
// a token's heads saves traffic (one warp per token measured 3.2 TB/s on
// GB300 against 4.8 for one per row; the factors then come from L2).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) fa_qk_norm_rope_bwd_kernel(const T* __restrict__ dq,
                                                                       const T* __restrict__ dk,
                                                                       const T* __restrict__ qk,
                                                                       const float* __restrict__ f1,
                                                                       const float* __restrict__ f2,
                                                                       T* __restrict__ dqk, int tokens, int hq,
                                                                       int hk) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int heads = hq + hk;
  const long rows = static_cast<long>(tokens) * heads;
  const long nwarps = static_cast<long>(gridDim.x) * (kThreads / 32);
  for (long r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const long t = r / heads;
    const int c = static_cast<int>(r - t * heads);
    const T* gsrc = c < hq ? dq + (t * hq + c) * D : dk + (t * hk + (c - hq)) * D;
    const Vec16<E> xr = *reinterpret_cast<const Vec16<E>*>(qk + r * D + lane * E);
    const Vec16<E> gr = *reinterpret_cast<const Vec16<E>*>(gsrc + lane * E);
    const VecF<E> a = *reinterpret_cast<const VecF<E>*>(f1 + t * D + lane * E);
    const VecF<E> s = *reinterpret_cast<const VecF<E>*>(f2 + t * D + lane * E);
    float x[E], g[E];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = to_f<T>(*reinterpret_cast<const T*>(&xr.v[e]));
      g[e] = to_f<T>(*reinterpret_cast<const T*>(&gr.v[e]));
      ss = fmaf(x[e], x[e], ss);
    }
    const float rstd = rsqrtf(warp_sum(ss) * (1.f / D) + kEps);
    float gn[E];
    float cs = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      gn[e] = a.v[e] * g[e] + s.v[e ^ 1] * g[e ^ 1];
      cs = fmaf(gn[e], x[e] * rstd, cs);
    }
    const float corr = warp_sum(cs) * (1.f / D);
    Vec16<E> dr;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const T v = from_f<T>(rstd * (gn[e] - (x[e] * rstd) * corr));
      dr.v[e] = *reinterpret_cast<const uint16_t*>(&v);
    }
    *reinterpret_cast<Vec16<E>*>(dqk + r * D + lane * E) = dr;
  }
}

int grid_for(long warps_of_work, int sms) {
  const long need = (warps_of_work + (kThreads / 32) - 1) / (kThreads / 32);
  const long cap = static_cast<long>(sms) * 16;  // 16 resident 256-thread CTAs per SM
  return static_cast<int>(need < cap ? need : cap);
}

template <typename T, int D>
cudaError_t fwd_t(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens, int hq, int hk,
                  int sms, cudaStream_t stream) {
  fa_qk_norm_rope_fwd_kernel<T, D><<<grid_for(tokens, sms), kThreads, 0, stream>>>(
      static_cast<const T*>(qk), f1, f2, static_cast<T*>(q), static_cast<T*>(k), tokens, hq, hk);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_t(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2, void* dqk,
                  int tokens, int hq, int hk, int sms, cudaStream_t stream) {
  fa_qk_norm_rope_bwd_kernel<T, D><<<grid_for(static_cast<long>(tokens) * (hq + hk), sms), kThreads, 0, stream>>>(
      static_cast<const T*>(dq), static_cast<const T*>(dk), static_cast<const T*>(qk), f1, f2, static_cast<T*>(dqk),
      tokens, hq, hk);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope_fwd(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens,
                                    int hq, int hk, int D, bool f16, int sms, cudaStream_t stream) {
  if (D == 64) return f16 ? fwd_t<__half, 64>(qk, f1, f2, q, k, tokens, hq, hk, sms, stream)
                          : fwd_t<__nv_bfloat16, 64>(qk, f1, f2, q, k, tokens, hq, hk, sms, stream);
  if (D == 128) return f16 ? fwd_t<__half, 128>(qk, f1, f2, q, k, tokens, hq, hk, sms, stream)
                           : fwd_t<__nv_bfloat16, 128>(qk, f1, f2, q, k, tokens, hq, hk, sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_qk_norm_rope_bwd(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2,
                                    void* dqk, int tokens, int hq, int hk, int D, bool f16, int sms,
                                    cudaStream_t stream) {
  if (D == 64) return f16 ? bwd_t<__half, 64>(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, sms, stream)
                          : bwd_t<__nv_bfloat16, 64>(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, sms, stream);
  if (D == 128) return f16 ? bwd_t<__half, 128>(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, sms, stream)
                           : bwd_t<__nv_bfloat16, 128>(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
