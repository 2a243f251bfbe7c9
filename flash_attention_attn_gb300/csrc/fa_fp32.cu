// fa_fp32.cu -- fp32 attention forward and backward on the CUDA cores.
//
// The fp32 workloads need max-abs errors near 1e-5, which TF32 tensor-core
// products (10-bit mantissas) cannot give, so this dtype runs in plain FFMA.
// One warp owns one row; its 32 lanes split the head dimension (D/32 elements
// each) and dot products are finished with warp shuffles.  Same masking,
// block-free loop bounds and GQA map as the bf16 kernels; every sum is taken
// in a fixed order, so results are reproducible.
//
//   forward (one warp per query row): online softmax over the visible keys
//     (forge flash_attention.metal, flash_attn_fwd: m_new, corr, l, o);
//   dQ      (one warp per query row): p = exp(s - LSE), ds = p (dp - Delta)
//     (flash_attn_bwd_dq);
//   dK, dV  (one warp per key row, summing over the group's query heads)
//     (flash_attn_bwd_dv / flash_attn_bwd_dk).
#include <math_constants.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

__device__ __forceinline__ void visible_keys(const Shape& s, int i, int& jlo, int& jhi) {
  jlo = (s.window > 0) ? max(0, i - s.window + 1) : 0;
  jhi = s.causal ? min(i, s.Tk - 1) : s.Tk - 1;
}

__device__ __forceinline__ void visible_queries(const Shape& s, int j, int& ilo, int& ihi) {
  ilo = s.causal ? j : 0;
  ihi = (s.window > 0) ? min(s.T - 1, j + s.window - 1) : s.T - 1;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) fa_fwd_fp32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                                 const float* __restrict__ V, float* __restrict__ O,
                                                                 float* __restrict__ LSE, const Shape s) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int h = blockIdx.y, b = blockIdx.z;
  if (i >= s.T) return;
  const int g = h / (s.H / s.HKV);
  const float* qi = Q + ((static_cast<size_t>(b) * s.T + i) * s.H + h) * D;
  float q[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = qi[lane + 32 * e];
    o[e] = 0.f;
  }
  float m = -CUDART_INF_F, l = 0.f;
  int jlo, jhi;
  visible_keys(s, i, jlo, jhi);
  for (int j = jlo; j <= jhi; ++j) {
    const size_t kv = ((static_cast<size_t>(b) * s.Tk + j) * s.HKV + g) * D;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) part = fmaf(q[e], K[kv + lane + 32 * e], part);
    const float sc = warp_sum(part) * s.scale;
    const float m_new = fmaxf(m, sc);
    const float corr = expf(m - m_new);  // 0 on the first key (m = -inf)
    const float p = expf(sc - m_new);
    l = l * corr + p;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(o[e], corr, p * V[kv + lane + 32 * e]);
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* oi = O + ((static_cast<size_t>(b) * s.T + i) * s.H + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) oi[lane + 32 * e] = o[e] * inv;
  if (lane == 0) LSE[(static_cast<size_t>(b) * s.H + h) * s.T + i] = l > 0.f ? m + logf(l) : 0.f;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) fa_bwd_dq_fp32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                                    const float* __restrict__ V, const float* __restrict__ dO,
                                                                    const float* __restrict__ LSE,
                                                                    const float* __restrict__ Delta, float* __restrict__ dQ,
                                                                    const Shape s) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int h = blockIdx.y, b = blockIdx.z;
  if (i >= s.T) return;
  const int g = h / (s.H / s.HKV);
  const size_t qo = ((static_cast<size_t>(b) * s.T + i) * s.H + h) * D;
  const size_t ro = (static_cast<size_t>(b) * s.H + h) * s.T + i;
  const float lse = LSE[ro], delta = Delta[ro];
  float q[E], go[E], dq[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    q[e] = Q[qo + lane + 32 * e];
    go[e] = dO[qo + lane + 32 * e];
    dq[e] = 0.f;
  }
  int jlo, jhi;
  visible_keys(s, i, jlo, jhi);
  for (int j = jlo; j <= jhi; ++j) {
    const size_t kv = ((static_cast<size_t>(b) * s.Tk + j) * s.HKV + g) * D;
    float ps = 0.f, pd = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      ps = fmaf(q[e], K[kv + lane + 32 * e], ps);
      pd = fmaf(go[e], V[kv + lane + 32 * e], pd);
    }
    const float sc = warp_sum(ps) * s.scale;
    const float dp = warp_sum(pd);
    const float ds = expf(sc - lse) * (dp - delta);
#pragma unroll
    for (int e = 0; e < E; ++e) dq[e] = fmaf(ds, K[kv + lane + 32 * e], dq[e]);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) dQ[qo + lane + 32 * e] = dq[e] * s.scale;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) fa_bwd_dkdv_fp32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                                                                      const float* __restrict__ V, const float* __restrict__ dO,
                                                                      const float* __restrict__ LSE,
                                                                      const float* __restrict__ Delta, float* __restrict__ dK,
                                                                      float* __restrict__ dV, const Shape s) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int g = blockIdx.y, b = blockIdx.z;
  if (j >= s.Tk) return;
  const int rep = s.H / s.HKV;
  const size_t kvo = ((static_cast<size_t>(b) * s.Tk + j) * s.HKV + g) * D;
  float k[E], v[E], dk[E], dv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    k[e] = K[kvo + lane + 32 * e];
    v[e] = V[kvo + lane + 32 * e];
    dk[e] = 0.f;
    dv[e] = 0.f;
  }
  int ilo, ihi;
  visible_queries(s, j, ilo, ihi);
  for (int r = 0; r < rep; ++r) {
    const int h = g * rep + r;
    for (int i = ilo; i <= ihi; ++i) {
      const size_t qo = ((static_cast<size_t>(b) * s.T + i) * s.H + h) * D;
      const size_t ro = (static_cast<size_t>(b) * s.H + h) * s.T + i;
      float ps = 0.f, pd = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        ps = fmaf(Q[qo + lane + 32 * e], k[e], ps);
        pd = fmaf(dO[qo + lane + 32 * e], v[e], pd);
      }
      const float sc = warp_sum(ps) * s.scale;
      const float dp = warp_sum(pd);
      const float p = expf(sc - LSE[ro]);
      const float ds = p * (dp - Delta[ro]);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        dv[e] = fmaf(p, dO[qo + lane + 32 * e], dv[e]);
        dk[e] = fmaf(ds, Q[qo + lane + 32 * e], dk[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    dK[kvo + lane + 32 * e] = dk[e] * s.scale;
    dV[kvo + lane + 32 * e] = dv[e];
  }
}

template <int D>
cudaError_t fwd_d(const float* Q, const float* K, const float* V, float* O, float* LSE, const Shape& s,
                  cudaStream_t st) {
  dim3 grid(ceil_div(s.T, kWarps), s.H, s.B);
  fa_fwd_fp32_kernel<D><<<grid, kWarps * 32, 0, st>>>(Q, K, V, O, LSE, s);
  return cudaGetLastError();
}

template <int D>
cudaError_t dkdv_d(const float* Q, const float* K, const float* V, const float* dO, const float* LSE,
                   const float* Delta, float* dK, float* dV, const Shape& s, cudaStream_t st) {
  dim3 grid(ceil_div(s.Tk, kWarps), s.HKV, s.B);
  fa_bwd_dkdv_fp32_kernel<D><<<grid, kWarps * 32, 0, st>>>(Q, K, V, dO, LSE, Delta, dK, dV, s);
  return cudaGetLastError();
}

template <int D>
cudaError_t dq_d(const float* Q, const float* K, const float* V, const float* dO, const float* LSE,
                 const float* Delta, float* dQ, const Shape& s, cudaStream_t st) {
  dim3 grid(ceil_div(s.T, kWarps), s.H, s.B);
  fa_bwd_dq_fp32_kernel<D><<<grid, kWarps * 32, 0, st>>>(Q, K, V, dO, LSE, Delta, dQ, s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                            const Shape& s, cudaStream_t stream) {
  if (s.D == 64) return fwd_d<64>(Q, K, V, O, LSE, s, stream);
  if (s.D == 128) return fwd_d<128>(Q, K, V, O, LSE, s, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv_fp32(const float* Q, const float* K, const float* V, const float* dO,
                                 const float* LSE, const float* Delta, float* dK, float* dV, const Shape& s,
                                 cudaStream_t stream) {
  if (s.D == 64) return dkdv_d<64>(Q, K, V, dO, LSE, Delta, dK, dV, s, stream);
  if (s.D == 128) return dkdv_d<128>(Q, K, V, dO, LSE, Delta, dK, dV, s, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_fp32(const float* Q, const float* K, const float* V, const float* dO,
                               const float* LSE, const float* Delta, float* dQ, const Shape& s,
                               cudaStream_t stream) {
  if (s.D == 64) return dq_d<64>(Q, K, V, dO, LSE, Delta, dQ, s, stream);
  if (s.D == 128) return dq_d<128>(Q, K, V, dO, LSE, Delta, dQ, s, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
