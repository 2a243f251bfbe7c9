// fa_internal.h -- declarations shared by the host library (fa_api.cu) and
// the kernels: tile planning, kernel parameter blocks and launchers.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace fa {

// Query rows per tile and key rows per block of the bf16 tensor-core kernels.
constexpr int kBM = 128;
constexpr int kBN = 128;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per pipeline wait

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

// Visible(i, j) = (!causal || j <= i) && (window == 0 || i - j < window),
// with query row i < Tq and key row j < Tk (Tq = Tk for self-attention; the
// library accepts Tq != Tk only without causal or window masking).  As index
// ranges, for per-element masking inside a block: query row i sees keys
// [lo, hi]; key j is seen by query rows [lo, hi] (empty, lo > hi, for a row
// or key past the end).
__host__ __device__ __forceinline__ void visible_keys(int Tq, int Tk, int causal, int window, int i, int& lo,
                                                      int& hi) {
  lo = window > 0 ? imax(0, i - window + 1) : 0;
  hi = causal ? imin(i, Tk - 1) : Tk - 1;
  if (i >= Tq) lo = hi + 1;
}
__host__ __device__ __forceinline__ void visible_queries(int Tq, int Tk, int causal, int window, int j, int& lo,
                                                         int& hi) {
  lo = causal ? j : 0;
  hi = window > 0 ? imin(Tq - 1, j + window - 1) : Tq - 1;
  if (j >= Tk) lo = hi + 1;
}

// KV blocks [lo, hi] that query tile qb must visit: blocks wholly above the
// causal diagonal or wholly before the window are skipped.
__host__ __device__ __forceinline__ void kv_range_for_q(int Tq, int Tk, int BM, int BN, int causal, int window,
                                                        int qb, int& lo, int& hi) {
  const int nkv = ceil_div(Tk, BN);
  const int row_lo = qb * BM;
  const int row_hi = imin(qb * BM + BM - 1, Tq - 1);
  hi = causal ? imin(nkv - 1, row_hi / BN) : nkv - 1;
  lo = window > 0 ? imax(0, row_lo - window + 1) / BN : 0;
}

// Query tiles [lo, hi] that see any key of KV block kb.
__host__ __device__ __forceinline__ void q_range_for_kv(int Tq, int Tk, int BM, int BN, int causal, int window,
                                                        int kb, int& lo, int& hi) {
  const int nq = ceil_div(Tq, BM);
  const int col_lo = kb * BN;
  const int col_hi = imin(kb * BN + BN - 1, Tk - 1);
  lo = causal ? col_lo / BM : 0;
  hi = window > 0 ? imin(nq - 1, (col_hi + window - 1) / BM) : nq - 1;
}

// Does block (qb, kb) hold any masked element (including rows >= Tq and
// keys >= Tk)?  Under causal masking with BM = BN these are the diagonal
// blocks: the block-offset k = qb*BM - kb*BN + 1 is the triu offset of that
// block.
__host__ __device__ __forceinline__ bool block_needs_mask(int Tq, int Tk, int BM, int BN, int causal, int window,
                                                          int qb, int kb) {
  const int row_lo = qb * BM, row_hi = qb * BM + BM - 1;
  const int col_lo = kb * BN, col_hi = kb * BN + BN - 1;
  if (row_hi >= Tq || col_hi >= Tk) return true;
  if (causal && col_hi > row_lo) return true;
  if (window > 0 && row_hi - col_lo >= window) return true;
  return false;
}

struct SchedCounter;  // fa_sched.cuh: the work counter of a persistent kernel (in the workspace)

struct Shape {
  int B, T, H, HKV, D;  // T: query rows
  float scale;
  int causal, window;
  int Tk;  // key rows (T for self-attention)
};

// ------------------------------------------------------------ bf16 kernels

struct FwdParams {
  Shape s;
  void* O;            // bf16 [B,T,H,D]
  float* LSE;         // [B,H,T]
  unsigned int* err;  // device error word
  float scale_log2;   // scale * log2(e)
  uint64_t timeout_ns;
  int inject_stall;
  int f16;            // elements are fp16 (else bf16)
  int pack_heads;     // two-tile kernel: the tiles are one query block of two heads (else two blocks of one head)
  int ctas;           // persistent kernels: CTAs to launch (at most one per SM; capped by the unit count)
  SchedCounter* sched;  // persistent kernels: their work counter in the workspace (zero between launches)
};

struct BwdParams {
  Shape s;
  int inject_stall;   // test hook: withhold the resident tile loads (the kernel's waits run out)
  const float* LSE;   // [B,H,T]
  const float* Delta; // [B,H,T]
  void* dQ;           // bf16 [B,T,H,D]
  void* dK;           // bf16 [B,T,HKV,D]
  void* dV;           // bf16 [B,T,HKV,D]
  unsigned int* err;
  float scale_log2;
  uint64_t timeout_ns;
  int f16;            // elements are fp16 (else bf16)
  int ctas;           // persistent kernels: CTAs to launch (at most one per SM; capped by the unit count)
  SchedCounter* sched;  // persistent kernels: their work counter in the workspace (zero between launches)
  float* dq_acc;        // fused backward: fp32 dQ accumulator [B,T,H,D] (workspace)
  unsigned int* turns;  // fused backward: turn counter per (b, h, query block) (workspace, zero between launches)
  int after_dkdv;       // dQ: launched as a programmatic dependent of the dK/dV kernel just before it on the stream
};

// 3-D views [B][T][heads*D] with boxes of 64 elements x R rows x 1 batch:
// R = 128 for the plain maps, R = 64 for the *64 maps.
struct TensorMaps {
  CUtensorMap q, k, v, dO;
};

// Raises a kernel's dynamic shared-memory limit (and, with carveout, its
// preferred carveout to the maximum) once per device: the attribute belongs
// to the kernel's instance on the current device.  `done` holds one bit per
// device ordinal.
inline cudaError_t set_smem_once(const void* kernel, int bytes, std::atomic<unsigned long long>& done,
                                 bool carveout = false) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && carveout)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_fwd_bf16(const TensorMaps& tm, const FwdParams& p, cudaStream_t stream);
// Pre-attention prologue (RMS-norm + rotary of the packed QK projection).
// Prologue with equally many query and key heads and the paired-heads or
// key-offset option (never both; neither = the plain prologue).
cudaError_t launch_qk_norm_rope_fwd_opt(const void* qk, const float* f1, const float* f2, void* q, void* k,
                                        int tokens, int heads, int D, int rot, bool paired, bool key_offset, bool f16,
                                        int sms, cudaStream_t stream);
cudaError_t launch_qk_norm_rope_bwd_opt(const void* dq, const void* dk, const void* qk, const float* f1,
                                        const float* f2, void* dqk, int tokens, int heads, int D, int rot,
                                        bool paired, bool key_offset, bool f16, int sms, cudaStream_t stream);
cudaError_t launch_qk_norm_rope_fwd(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens,
                                    int hq, int hk, int D, bool f16, int sms, cudaStream_t stream);
cudaError_t launch_qk_norm_rope_bwd(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2,
                                    void* dqk, int tokens, int hq, int hk, int D, bool f16, int sms,
                                    cudaStream_t stream);
// Whether the bf16 forward runs two query tiles per CTA for this shape.
// Forward kernel for a shape: 1 = one query tile per CTA, 2 = two tiles =
// two adjacent query blocks of one head, 3 = two tiles = one query block of
// two heads that share a KV head.
int fwd_mode(const Shape& s);
cudaError_t launch_bwd_dkdv_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream);
// Backward for head dims up to 64 under causal masking (self-attention,
// 16-bit elements): dK, dV and dQ in one kernel, dQ without the recompute of
// S and dP (fa_bwd_fused.cu).  acc_map: 4-D fp32 view of p.dq_acc with boxes
// of 32 elements x 1 head x 128 rows x 1 batch, 128-byte swizzle.
bool fused_backward_applies(const Shape& s, int f16_or_bf16);
cudaError_t launch_bwd_fused(const TensorMaps& tm, const CUtensorMap& acc_map, const BwdParams& p,
                             cudaStream_t stream);
cudaError_t launch_bwd_dq_bf16(const TensorMaps& tm, const BwdParams& p, cudaStream_t stream);

// Every host-side check fa_bwd makes (shape, pointers and their alignment,
// workspace size and alignment, device) without launching anything: FA_OK or
// the status fa_bwd would return for the same arguments.
int check_bwd_call(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                   void* dQ, void* dK, void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal,
                   int window, int dtype, void* workspace, size_t workspace_bytes);

// ---------------------------------------------------------- shared kernels

// Delta[b,h,i] = sum_d dO[b,i,h,d] * O[b,i,h,d], fp32 accumulation.
// elem: 0 bf16, 1 fp32, 2 fp16 (the fa_dtype values)
cudaError_t launch_delta(const void* O, const void* dO, float* Delta, const Shape& s, int elem,
                         cudaStream_t stream);

// ----------------------------------------------------------- fp32 kernels

cudaError_t launch_fwd_fp32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                            const Shape& s, cudaStream_t stream);
cudaError_t launch_bwd_dkdv_fp32(const float* Q, const float* K, const float* V, const float* dO,
                                 const float* LSE, const float* Delta, float* dK, float* dV, const Shape& s,
                                 cudaStream_t stream);
cudaError_t launch_bwd_dq_fp32(const float* Q, const float* K, const float* V, const float* dO,
                               const float* LSE, const float* Delta, float* dQ, const Shape& s,
                               cudaStream_t stream);

}  // namespace fa
