// fa_prologue.cu -- pre-attention prologue: RMS-norm of every query and key
// head vector, then the rotary mix with per-position factors, writing the Q
// and K tensors the attention forward reads; and its backward.
//
// What it computes is the modded-nanogpt page qkv_rope.py (module docstring
// and `_qk_norm_rope_forward_kernel`; the backward is the norm/rotary part of
// `_qkv_norm_rope_pack_fp8_backward_kernel` without the fp8 packing).  The
// plain kernels below take any hq, hk; the page's paired-heads and
// key-offset options have their own kernels further down:
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

// ------------------------------------------------------------------ options
//
// Paired heads and key offset (the same page's PAIRED and KEY_OFFSET
// branches; never both).  The projection holds `heads` query heads then
// `heads` key heads; logical head h = c mod heads.
//   paired:     factor rows 2*D wide, head h rotates with half h mod 2; the
//               output of (t, h) lands at token 2t + h div (heads/2), head
//               h mod (heads/2) of [2*tokens][heads/2][D] q and k.
//   key offset: a key row of token t > 0 takes its stationary dims d >= rot
//               from token t-1's normalised row of the same head, unrotated.
// The backward is the exact gradient of that forward: for a key row with
// key offset, n_e at e >= rot feeds only token t+1's output (and token 0's
// own rotated output), so its gradient there is g_{t+1, e} plus, at t = 0,
// the rotation term.

__device__ __forceinline__ size_t out_row(int t, int h, int heads, bool paired) {
  if (paired) {
    const int half = heads >> 1;
    return static_cast<size_t>(2 * t + h / half) * half + (h % half);
  }
  return static_cast<size_t>(t) * heads + h;
}

template <typename T, int E>
__device__ __forceinline__ float load_row(const T* row, int lane, float (&x)[E]) {
  const Vec16<E> xr = *reinterpret_cast<const Vec16<E>*>(row + lane * E);
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    x[e] = to_f<T>(*reinterpret_cast<const T*>(&xr.v[e]));
    ss = fmaf(x[e], x[e], ss);
  }
  return ss;
}

// One warp per token, as the plain forward: the token's factors (both
// halves when paired) stay in registers for its 2*heads rows.
template <typename T, int D, bool PAIRED, bool KEYOFF>
__global__ void __launch_bounds__(kThreads) fa_qk_norm_rope_fwd_opt_kernel(const T* __restrict__ qk,
                                                                           const float* __restrict__ f1,
                                                                           const float* __restrict__ f2,
                                                                           T* __restrict__ q, T* __restrict__ k,
                                                                           int tokens, int heads, int rot) {
  constexpr int E = D / 32;
  constexpr int F = PAIRED ? 2 * D : D;
  const int lane = threadIdx.x & 31;
  const long nwarps = static_cast<long>(gridDim.x) * (kThreads / 32);
  for (long t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < tokens; t += nwarps) {
    // factor halves 0 and 1 (the same half twice when not paired)
    const VecF<E> a0 = *reinterpret_cast<const VecF<E>*>(f1 + t * F + lane * E);
    const VecF<E> s0 = *reinterpret_cast<const VecF<E>*>(f2 + t * F + lane * E);
    const VecF<E> a1 = PAIRED ? *reinterpret_cast<const VecF<E>*>(f1 + t * F + D + lane * E) : a0;
    const VecF<E> s1 = PAIRED ? *reinterpret_cast<const VecF<E>*>(f2 + t * F + D + lane * E) : s0;
#pragma unroll 2
    for (int c = 0; c < 2 * heads; ++c) {
      const bool is_key = c >= heads;
      const int h = is_key ? c - heads : c;
      float x[E];
      const float rstd = rsqrtf(warp_sum(load_row<T, E>(qk + (t * 2 * heads + c) * D, lane, x)) * (1.f / D) + kEps);
      const bool odd = PAIRED && (h & 1);
      float y[E];
#pragma unroll
      for (int e = 0; e < E; ++e)
        y[e] = (odd ? a1.v[e] : a0.v[e]) * (x[e] * rstd) + (odd ? s1.v[e] : s0.v[e]) * (x[e ^ 1] * rstd);
      if (KEYOFF && is_key && t > 0) {
        float xp[E];
        const float rp =
            rsqrtf(warp_sum(load_row<T, E>(qk + ((t - 1) * 2 * heads + c) * D, lane, xp)) * (1.f / D) + kEps);
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (lane * E + e >= rot) y[e] = xp[e] * rp;
      }
      Vec16<E> yr;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const T yt = from_f<T>(y[e]);
        yr.v[e] = *reinterpret_cast<const uint16_t*>(&yt);
      }
      *reinterpret_cast<Vec16<E>*>((is_key ? k : q) + out_row(static_cast<int>(t), h, heads, PAIRED) * D +
                                   lane * E) = yr;
    }
  }
}

// One warp per (token, input head) row, as the plain backward.
template <typename T, int D, bool PAIRED, bool KEYOFF>
__global__ void __launch_bounds__(kThreads) fa_qk_norm_rope_bwd_opt_kernel(const T* __restrict__ dq,
                                                                           const T* __restrict__ dk,
                                                                           const T* __restrict__ qk,
                                                                           const float* __restrict__ f1,
                                                                           const float* __restrict__ f2,
                                                                           T* __restrict__ dqk, int tokens,
                                                                           int heads, int rot) {
  constexpr int E = D / 32;
  constexpr int F = PAIRED ? 2 * D : D;
  const int lane = threadIdx.x & 31;
  const long rows = static_cast<long>(tokens) * 2 * heads;
  const long nwarps = static_cast<long>(gridDim.x) * (kThreads / 32);
  for (long r = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const int t = static_cast<int>(r / (2 * heads));
    const int c = static_cast<int>(r - static_cast<long>(t) * 2 * heads);
    const bool is_key = c >= heads;
    const int h = is_key ? c - heads : c;
    const int hv = PAIRED ? (h & 1) : 0;
    float x[E], g[E];
    const float ss = load_row<T, E>(qk + r * D, lane, x);
    load_row<T, E>((is_key ? dk : dq) + out_row(t, h, heads, PAIRED) * D, lane, g);
    const VecF<E> a = *reinterpret_cast<const VecF<E>*>(f1 + static_cast<long>(t) * F + hv * D + lane * E);
    const VecF<E> s = *reinterpret_cast<const VecF<E>*>(f2 + static_cast<long>(t) * F + hv * D + lane * E);
    const float rstd = rsqrtf(warp_sum(ss) * (1.f / D) + kEps);
    float gn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) gn[e] = a.v[e] * g[e] + s.v[e ^ 1] * g[e ^ 1];
    if (KEYOFF && is_key) {
      float gnext[E];
#pragma unroll
      for (int e = 0; e < E; ++e) gnext[e] = 0.f;
      if (t + 1 < tokens) load_row<T, E>(dk + out_row(t + 1, h, heads, false) * D, lane, gnext);
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (lane * E + e >= rot) gn[e] = (t == 0 ? gn[e] : 0.f) + gnext[e];
    }
    float cs = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) cs = fmaf(gn[e], x[e] * rstd, cs);
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

template <typename T, int D>
cudaError_t fwd_opt_t(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens, int heads,
                      int rot, bool paired, bool key_offset, int sms, cudaStream_t stream) {
  const dim3 grid(grid_for(tokens, sms));
  const T* x = static_cast<const T*>(qk);
  T* qo = static_cast<T*>(q);
  T* ko = static_cast<T*>(k);
  if (paired)
    fa_qk_norm_rope_fwd_opt_kernel<T, D, true, false><<<grid, kThreads, 0, stream>>>(x, f1, f2, qo, ko, tokens,
                                                                                     heads, rot);
  else if (key_offset)
    fa_qk_norm_rope_fwd_opt_kernel<T, D, false, true><<<grid, kThreads, 0, stream>>>(x, f1, f2, qo, ko, tokens,
                                                                                     heads, rot);
  else
    fa_qk_norm_rope_fwd_opt_kernel<T, D, false, false><<<grid, kThreads, 0, stream>>>(x, f1, f2, qo, ko, tokens,
                                                                                      heads, rot);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t bwd_opt_t(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2, void* dqk,
                      int tokens, int heads, int rot, bool paired, bool key_offset, int sms, cudaStream_t stream) {
  const dim3 grid(grid_for(static_cast<long>(tokens) * 2 * heads, sms));
  const T* gq = static_cast<const T*>(dq);
  const T* gk = static_cast<const T*>(dk);
  const T* x = static_cast<const T*>(qk);
  T* dx = static_cast<T*>(dqk);
  if (paired)
    fa_qk_norm_rope_bwd_opt_kernel<T, D, true, false><<<grid, kThreads, 0, stream>>>(gq, gk, x, f1, f2, dx, tokens,
                                                                                     heads, rot);
  else if (key_offset)
    fa_qk_norm_rope_bwd_opt_kernel<T, D, false, true><<<grid, kThreads, 0, stream>>>(gq, gk, x, f1, f2, dx, tokens,
                                                                                     heads, rot);
  else
    fa_qk_norm_rope_bwd_opt_kernel<T, D, false, false><<<grid, kThreads, 0, stream>>>(gq, gk, x, f1, f2, dx,
                                                                                      tokens, heads, rot);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope_fwd_opt(const void* qk, const float* f1, const float* f2, void* q, void* k,
                                        int tokens, int heads, int D, int rot, bool paired, bool key_offset, bool f16,
                                        int sms, cudaStream_t stream) {
  if (D == 64) return f16 ? fwd_opt_t<__half, 64>(qk, f1, f2, q, k, tokens, heads, rot, paired, key_offset, sms, stream)
                          : fwd_opt_t<__nv_bfloat16, 64>(qk, f1, f2, q, k, tokens, heads, rot, paired, key_offset,
                                                          sms, stream);
  if (D == 128)
    return f16 ? fwd_opt_t<__half, 128>(qk, f1, f2, q, k, tokens, heads, rot, paired, key_offset, sms, stream)
               : fwd_opt_t<__nv_bfloat16, 128>(qk, f1, f2, q, k, tokens, heads, rot, paired, key_offset, sms,
                                                stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_qk_norm_rope_bwd_opt(const void* dq, const void* dk, const void* qk, const float* f1,
                                        const float* f2, void* dqk, int tokens, int heads, int D, int rot,
                                        bool paired, bool key_offset, bool f16, int sms, cudaStream_t stream) {
  if (D == 64)
    return f16 ? bwd_opt_t<__half, 64>(dq, dk, qk, f1, f2, dqk, tokens, heads, rot, paired, key_offset, sms, stream)
               : bwd_opt_t<__nv_bfloat16, 64>(dq, dk, qk, f1, f2, dqk, tokens, heads, rot, paired, key_offset, sms,
                                               stream);
  if (D == 128)
    return f16 ? bwd_opt_t<__half, 128>(dq, dk, qk, f1, f2, dqk, tokens, heads, rot, paired, key_offset, sms,
                                         stream)
               : bwd_opt_t<__nv_bfloat16, 128>(dq, dk, qk, f1, f2, dqk, tokens, heads, rot, paired, key_offset, sms,
                                                stream);
  return cudaErrorInvalidValue;
}

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
