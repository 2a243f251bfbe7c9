// fa_delta.cu -- backward preprocess: Delta[b,h,i] = sum_d dO[b,i,h,d] * O[b,i,h,d]
// (bf16, fp16 or fp32 elements, fp32 accumulation)
// (the identity rowsum(dO * O) = rowsum(dP * P) named in the forge page,
// flash_attention.metal, backward section; the Graphcore page computes the
// same D before its block loops).
//
// Pure HBM stream: 2 * B*T*H*D elements read, B*H*T floats written.  One
// 256-thread CTA covers 64 consecutive positions t of one (b, h): each row of
// D elements is read as 16-byte vectors by D*size/16 consecutive lanes (whole
// 32-byte sectors), every thread issues all of its loads before reducing, and
// the 64 results leave as one contiguous 256-byte store.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRowsPerCta = 64;
constexpr int kThreads = 256;

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, const __nv_bfloat16*) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fx = __bfloat1622float2(x[k]);
    const float2 fy = __bfloat1622float2(y[k]);
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, const __half*) {
  const __half2* x = reinterpret_cast<const __half2*>(&a);
  const __half2* y = reinterpret_cast<const __half2*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fx = __half22float2(x[k]);
    const float2 fy = __half22float2(y[k]);
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  return acc;
}

__device__ __forceinline__ float dot16(const uint4& a, const uint4& b, const float*) {
  const float4 x = *reinterpret_cast<const float4*>(&a);
  const float4 y = *reinterpret_cast<const float4*>(&b);
  return fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, x.w * y.w)));
}

// D: 64 or 128 lanes' worth of row; Dact <= D elements of it are real (the
// rest read as zeros).  EXACT: Dact == D, known at compile time.
template <typename T, int D, bool EXACT>
__global__ void __launch_bounds__(kThreads) fa_bwd_delta_kernel(const T* __restrict__ O, const T* __restrict__ dO,
                                                                float* __restrict__ Delta, int Tlen, int H, int Dact) {
  if (EXACT) Dact = D;
  constexpr int kVec = 16 / sizeof(T);               // elements per 16-byte load
  constexpr int kLanes = D / kVec;                   // lanes per row (8, 16 or 32)
  constexpr int kRowsPerPass = kThreads / kLanes;
  constexpr int kPasses = kRowsPerCta / kRowsPerPass;
  __shared__ float out[kRowsPerCta];

  const int t0 = blockIdx.x * kRowsPerCta;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int sub = threadIdx.x % kLanes;
  const int r0 = threadIdx.x / kLanes;

  uint4 xo[kPasses], xd[kPasses];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int t = t0 + ps * kRowsPerPass + r0;
    if (t < Tlen && sub * kVec < Dact) {
      const size_t off = ((static_cast<size_t>(b) * Tlen + t) * H + h) * Dact + sub * kVec;
      xo[ps] = __ldg(reinterpret_cast<const uint4*>(O + off));
      xd[ps] = __ldg(reinterpret_cast<const uint4*>(dO + off));
    } else {
      xo[ps] = make_uint4(0, 0, 0, 0);
      xd[ps] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    float acc = dot16(xo[ps], xd[ps], static_cast<const T*>(nullptr));
#pragma unroll
    for (int m = kLanes / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (sub == 0) out[ps * kRowsPerPass + r0] = acc;
  }
  __syncthreads();
  if (threadIdx.x < kRowsPerCta) {
    const int t = t0 + threadIdx.x;
    if (t < Tlen) Delta[(static_cast<size_t>(b) * H + h) * Tlen + t] = out[threadIdx.x];
  }
}

template <typename T, int D>
cudaError_t launch(const void* O, const void* dO, float* Delta, const Shape& s, cudaStream_t stream) {
  dim3 grid(ceil_div(s.T, kRowsPerCta), s.H, s.B);
  if (s.D == D)
    fa_bwd_delta_kernel<T, D, true><<<grid, kThreads, 0, stream>>>(static_cast<const T*>(O),
                                                                   static_cast<const T*>(dO), Delta, s.T, s.H, D);
  else
    fa_bwd_delta_kernel<T, D, false><<<grid, kThreads, 0, stream>>>(static_cast<const T*>(O),
                                                                    static_cast<const T*>(dO), Delta, s.T, s.H, s.D);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta(const void* O, const void* dO, float* Delta, const Shape& s, int elem,
                         cudaStream_t stream) {
  if (elem == 0) {  // bf16
    if (s.D <= 64) return launch<__nv_bfloat16, 64>(O, dO, Delta, s, stream);
    if (s.D <= 128) return launch<__nv_bfloat16, 128>(O, dO, Delta, s, stream);
  } else if (elem == 2) {  // fp16
    if (s.D <= 64) return launch<__half, 64>(O, dO, Delta, s, stream);
    if (s.D <= 128) return launch<__half, 128>(O, dO, Delta, s, stream);
  } else {  // fp32
    if (s.D == 64) return launch<float, 64>(O, dO, Delta, s, stream);
    if (s.D == 128) return launch<float, 128>(O, dO, Delta, s, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
