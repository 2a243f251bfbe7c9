// fa_api.cu -- the C ABI declared in include/fa.h: argument validation,
// workspace layout, TMA tensor-map encoding and kernel launches.  Nothing
// here computes attention; every arithmetic step runs in the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

using fa::Shape;

// The workspace's first 256 bytes: the device error word at 0, the work
// counters of the persistent kernels at kSchedOffset (forward, dK/dV, dQ;
// 8 bytes each); then Delta.
constexpr size_t kErrBytes = 256;
constexpr size_t kSchedOffset = 64;

fa::SchedCounter* sched_counter(void* workspace, int which) {
  return reinterpret_cast<fa::SchedCounter*>(static_cast<char*>(workspace) + kSchedOffset + 8 * which);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

std::atomic<unsigned long long> g_wait_ns{fa::kDefaultWaitNs};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_fwd_tiles{0};  // 0 = automatic
std::atomic<int> g_max_ctas{0};   // 0 = one CTA per SM

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Test hook: 1 = the next 16-bit forward launch, 2 = the next dK/dV launch,
// 3 = the next dQ launch withholds its first tile loads; taken (and cleared)
// by the launch it names.
int take_stall(int kind) {
  int expected = kind;
  return g_inject_stall.compare_exchange_strong(expected, 0) ? 1 : 0;
}

// T: query rows, Tk: key rows (T for self-attention).
int validate_shape(int B, int T, int Tk, int H, int HKV, int D, float scale, int causal, int window, int dtype) {
  if (B < 1 || T < 1 || Tk < 1 || H < 1 || HKV < 1 || D < 1) return FA_ERR_INVALID_ARG;
  if (H % HKV != 0) return FA_ERR_INVALID_ARG;
  if (window < 0 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  // queries and keys of different lengths: unmasked attention only (the
  // pages place no causal diagonal or window between two sequences)
  if (Tk != T && (causal || window)) return FA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale == INFINITY) return FA_ERR_INVALID_ARG;  // also rejects NaN
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP32 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_DTYPE_FP32) {
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  } else if (D < 16 || D > 128 || D % 8 != 0) {
    // 16-bit tensor-core path: the kernels run at 64 or 128 and read zeros
    // past D (TMA fill); D % 8 keeps every row 16-byte aligned
    return FA_ERR_UNSUPPORTED;
  }
  // grid limits (y = heads, z = batch) and 32-bit row indexing inside kernels
  if (H > 65535 || B > 65535) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * T * H * D >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Tk * HKV * D >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) + window >= (1ll << 30) || Tk >= (1 << 30)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t delta_bytes(int B, int T, int H) { return round_up(sizeof(float) * static_cast<size_t>(B) * H * T, 256); }

// The fused backward (head dims up to 64, 16-bit elements, causal) also keeps
// an fp32 dQ accumulator [B,T,H,D] and one turn counter per (b, h, query
// block) in the workspace, after Delta.
bool fused_sizes(int head_dim, int dtype) { return dtype != FA_DTYPE_FP32 && head_dim <= 64; }
size_t acc_bytes(int B, int T, int H, int D) { return round_up(sizeof(float) * static_cast<size_t>(B) * T * H * D, 256); }
size_t turn_bytes(int B, int T, int H) {
  return round_up(sizeof(unsigned) * static_cast<size_t>(B) * H * fa::ceil_div(T, fa::kBM), 256);
}
size_t bwd_base_bytes(int B, int T, int H) { return kErrBytes + delta_bytes(B, T, H); }
size_t bwd_full_bytes(int B, int T, int H, int D, int dtype) {
  return bwd_base_bytes(B, T, H) + (fused_sizes(D, dtype) ? acc_bytes(B, T, H, D) + turn_bytes(B, T, H) : 0);
}

// ---------------------------------------------------------------- devices

struct DeviceInfo {
  bool probed = false;
  bool sm103 = false;
  int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_ok(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    d.sm103 = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_CUDA;
    d.probed = true;
  }
  *dev_out = dev;
  return d.sm103 ? FA_OK : FA_ERR_UNSUPPORTED;
}

// CTAs of a persistent kernel on device `dev`: one per SM, or the number
// the test hook sets (the launch takes at most one CTA per work unit).
int persistent_ctas(int dev) {
  const int cap = g_max_ctas.load();
  const int sms = g_dev[dev].sms > 0 ? g_dev[dev].sms : 1;
  return cap > 0 ? cap : sms;
}

int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return FA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return FA_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return FA_OK;
}

// 4-D 16-bit (bf16 or fp16) view [B][T][heads][D] of a [B,T,heads,D] tensor;
// boxes of 64 elements x 1 head x 128 rows x 1 batch, 128-byte swizzle.
// Elements past D (head dims below 64 or 128) and rows past T read as zeros.
int encode_map(CUtensorMap* map, const void* base, int B, int T, int heads, int D, int dtype) {
  const cuuint64_t row = static_cast<cuuint64_t>(heads) * D * 2;  // bytes per position
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, row, row * static_cast<cuuint64_t>(T)};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      dtype == FA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = g_encode(map, ty, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

namespace fa {
int fwd_mode(const Shape& s) {
  const int forced = g_fwd_tiles.load();
  if (forced == 1 || forced == 2) return forced;
  // automatic (0) and head pairs asked for (3): head pairs need an even
  // number of query heads per KV head
  if ((s.H / s.HKV) % 2 == 0) return 3;
  return ceil_div(s.T, kBM) >= 2 ? 2 : 1;
}
}  // namespace fa

extern "C" {

size_t fa_workspace_size(int op, int B, int T, int H, int HKV, int head_dim, int dtype) {
  if (validate_shape(B, T, T, H, HKV, head_dim, 1.f, 1, 0, dtype) != FA_OK) return 0;
  if (op == FA_OP_FWD) return kErrBytes;
  if (op == FA_OP_BWD) return bwd_base_bytes(B, T, H);
  if (op == FA_OP_BWD_FUSED) return fused_sizes(head_dim, dtype) ? bwd_full_bytes(B, T, H, head_dim, dtype) : 0;
  return 0;
}

}  // extern "C"

namespace {

int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int T, int Tk, int H, int HKV,
             int head_dim, float scale, int causal, int window, int dtype, void* workspace, size_t workspace_bytes,
             void* stream) {
  int st = validate_shape(B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype);
  if (st != FA_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE)) return FA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < fa_workspace_size(FA_OP_FWD, B, T, H, HKV, head_dim, dtype))
    return FA_ERR_WORKSPACE;
  int dev;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Shape shp{B, T, H, HKV, head_dim, scale, causal, window, Tk};
  if (dtype == FA_DTYPE_FP32)
    return status_of(fa::launch_fwd_fp32(static_cast<const float*>(Q), static_cast<const float*>(K),
                                         static_cast<const float*>(V), static_cast<float*>(O), LSE, shp, s));
  if ((st = get_encoder()) != FA_OK) return st;
  fa::TensorMaps tm;
  if ((st = encode_map(&tm.q, Q, B, T, H, head_dim, dtype)) != FA_OK) return st;
  if ((st = encode_map(&tm.k, K, B, Tk, HKV, head_dim, dtype)) != FA_OK) return st;
  if ((st = encode_map(&tm.v, V, B, Tk, HKV, head_dim, dtype)) != FA_OK) return st;
  fa::FwdParams p;
  p.s = shp;
  p.O = O;
  p.LSE = LSE;
  p.err = static_cast<unsigned int*>(workspace);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_wait_ns.load();
  p.inject_stall = take_stall(1);
  p.f16 = dtype == FA_DTYPE_FP16;
  p.ctas = persistent_ctas(dev);
  p.sched = sched_counter(workspace, 0);
  return status_of(fa::launch_fwd_bf16(tm, p, s));
}

// Shared checks of the backward stages; fills the shape and the Delta pointer.
int bwd_prologue(const void* const* ptrs, int nptr, int B, int T, int Tk, int H, int HKV, int head_dim, float scale,
                 int causal, int window, int dtype, void* workspace, size_t workspace_bytes, Shape* shp,
                 float** delta) {
  int st = validate_shape(B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype);
  if (st != FA_OK) return st;
  for (int i = 0; i < nptr; ++i)
    if (!ptrs[i] || !aligned16(ptrs[i])) return FA_ERR_INVALID_ARG;
  // the error word and Delta (the fused backward checks for its accumulator
  // and turn counters itself)
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < bwd_base_bytes(B, T, H))
    return FA_ERR_WORKSPACE;
  int dev;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  *shp = Shape{B, T, H, HKV, head_dim, scale, causal, window, Tk};
  *delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + kErrBytes);
  return FA_OK;
}

}  // namespace

namespace fa {
int check_bwd_call(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                   void* dQ, void* dK, void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal,
                   int window, int dtype, void* workspace, size_t workspace_bytes) {
  const void* ptrs[] = {Q, K, V, O, LSE, dO, dQ, dK, dV};
  Shape shp;
  float* delta;
  return bwd_prologue(ptrs, 9, B, T, T, H, HKV, head_dim, scale, causal, window, dtype, workspace, workspace_bytes,
                      &shp, &delta);
}
}  // namespace fa

namespace {

int bwd_maps(fa::TensorMaps* tm, const void* Q, const void* K, const void* V, const void* dO, const Shape& s,
             int dtype) {
  int st;
  if ((st = get_encoder()) != FA_OK) return st;
  if ((st = encode_map(&tm->q, Q, s.B, s.T, s.H, s.D, dtype)) != FA_OK) return st;
  if ((st = encode_map(&tm->k, K, s.B, s.Tk, s.HKV, s.D, dtype)) != FA_OK) return st;
  if ((st = encode_map(&tm->v, V, s.B, s.Tk, s.HKV, s.D, dtype)) != FA_OK) return st;
  if ((st = encode_map(&tm->dO, dO, s.B, s.T, s.H, s.D, dtype)) != FA_OK) return st;
  return FA_OK;
}

fa::BwdParams bwd_params(const Shape& s, const float* LSE, const float* delta, void* dQ, void* dK, void* dV,
                         void* workspace, int dtype, int stall_kind) {
  fa::BwdParams p{};
  int dev = 0;
  cudaGetDevice(&dev);  // already checked by bwd_prologue
  p.ctas = persistent_ctas(dev);
  p.sched = sched_counter(workspace, stall_kind == 2 ? 1 : 2);  // the dK/dV or the dQ kernel's counter
  p.s = s;
  p.inject_stall = take_stall(stall_kind);
  p.LSE = LSE;
  p.Delta = delta;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.err = static_cast<unsigned int*>(workspace);
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.timeout_ns = g_wait_ns.load();
  p.f16 = dtype == FA_DTYPE_FP16;
  return p;
}

int preprocess_impl(const void* O, const void* dO, int B, int T, int H, int HKV, int head_dim, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {O, dO};
  Shape shp;
  float* delta;
  int st = bwd_prologue(ptrs, 2, B, T, T, H, HKV, head_dim, 1.f, 1, 0, dtype, workspace, workspace_bytes, &shp,
                        &delta);
  if (st != FA_OK) return st;
  return status_of(fa::launch_delta(O, dO, delta, shp, dtype, static_cast<cudaStream_t>(stream)));
}

int dkdv_impl(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dK, void* dV,
              int B, int T, int Tk, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
              void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {Q, K, V, LSE, dO, dK, dV};
  Shape shp;
  float* delta;
  int st = bwd_prologue(ptrs, 7, B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                        workspace_bytes, &shp, &delta);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_FP32)
    return status_of(fa::launch_bwd_dkdv_fp32(static_cast<const float*>(Q), static_cast<const float*>(K),
                                              static_cast<const float*>(V), static_cast<const float*>(dO), LSE,
                                              delta, static_cast<float*>(dK), static_cast<float*>(dV), shp, s));
  fa::TensorMaps tm;
  if ((st = bwd_maps(&tm, Q, K, V, dO, shp, dtype)) != FA_OK) return st;
  return status_of(fa::launch_bwd_dkdv_bf16(tm, bwd_params(shp, LSE, delta, nullptr, dK, dV, workspace, dtype, 2), s));
}

int dq_impl(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ, int B, int T,
            int Tk, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype, void* workspace,
            size_t workspace_bytes, void* stream, bool after_dkdv = false) {
  const void* ptrs[] = {Q, K, V, LSE, dO, dQ};
  Shape shp;
  float* delta;
  int st = bwd_prologue(ptrs, 6, B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                        workspace_bytes, &shp, &delta);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_FP32)
    return status_of(fa::launch_bwd_dq_fp32(static_cast<const float*>(Q), static_cast<const float*>(K),
                                            static_cast<const float*>(V), static_cast<const float*>(dO), LSE, delta,
                                            static_cast<float*>(dQ), shp, s));
  fa::TensorMaps tm;
  if ((st = bwd_maps(&tm, Q, K, V, dO, shp, dtype)) != FA_OK) return st;
  fa::BwdParams p = bwd_params(shp, LSE, delta, dQ, nullptr, nullptr, workspace, dtype, 3);
  p.after_dkdv = after_dkdv ? 1 : 0;
  return status_of(fa::launch_bwd_dq_bf16(tm, p, s));
}

// 4-D fp32 view [B][T][heads][D] of the dQ accumulator; boxes of 32
// elements x 1 head x 128 rows x 1 batch, 128-byte swizzle (the layout the
// fused kernel stages its partials in).
int encode_acc_map(CUtensorMap* map, const float* base, int B, int T, int heads, int D) {
  const cuuint64_t row = static_cast<cuuint64_t>(heads) * D * 4;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 4, row, row * static_cast<cuuint64_t>(T)};
  cuuint32_t box[4] = {32, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// dK, dV and dQ in one launch (the fused backward); Delta must be in the
// workspace already.  FA_ERR_UNSUPPORTED if the shape does not take it,
// FA_ERR_WORKSPACE if the workspace lacks the accumulator.
int fused_impl(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ, void* dK,
               void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
               void* workspace, size_t workspace_bytes, void* stream) {
  int st = validate_shape(B, T, T, H, HKV, head_dim, scale, causal, window, dtype);
  if (st != FA_OK) return st;
  if (!fa::fused_backward_applies(Shape{B, T, H, HKV, head_dim, scale, causal, window, T}, dtype != FA_DTYPE_FP32))
    return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < bwd_full_bytes(B, T, H, head_dim, dtype)) return FA_ERR_WORKSPACE;
  const void* ptrs[] = {Q, K, V, LSE, dO, dQ, dK, dV};
  Shape shp;
  float* delta;
  if ((st = bwd_prologue(ptrs, 8, B, T, T, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                         workspace_bytes, &shp, &delta)) != FA_OK)
    return st;
  int dev;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  fa::TensorMaps tm;
  if ((st = bwd_maps(&tm, Q, K, V, dO, shp, dtype)) != FA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  float* acc = reinterpret_cast<float*>(ws + bwd_base_bytes(B, T, H));
  unsigned* turns = reinterpret_cast<unsigned*>(ws + bwd_base_bytes(B, T, H) + acc_bytes(B, T, H, head_dim));
  CUtensorMap acc_map;
  if ((st = encode_acc_map(&acc_map, acc, B, T, H, head_dim)) != FA_OK) return st;
  // every launch starts its turn counters at zero (a launch that gave up on
  // a wait may have left some advanced)
  if (cudaMemsetAsync(turns, 0, turn_bytes(B, T, H), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  fa::BwdParams p = bwd_params(shp, LSE, delta, dQ, dK, dV, workspace, dtype, 2);
  p.sched = sched_counter(workspace, 3);
  p.dq_acc = acc;
  p.turns = turns;
  // a cooperative launch: at most one CTA per SM, all resident together
  const int sms = g_dev[dev].sms > 0 ? g_dev[dev].sms : 1;
  p.ctas = fa::imin(p.ctas, sms);
  return status_of(fa::launch_bwd_fused(tm, acc_map, p, static_cast<cudaStream_t>(stream)));
}

int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO, void* dQ,
             void* dK, void* dV, int B, int T, int Tk, int H, int HKV, int head_dim, float scale, int causal,
             int window, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  // validate every argument before the first launch, so that a bad call
  // launches nothing
  const void* ptrs[] = {Q, K, V, O, LSE, dO, dQ, dK, dV};
  Shape shp;
  float* delta;
  int st = bwd_prologue(ptrs, 9, B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                        workspace_bytes, &shp, &delta);
  if (st != FA_OK) return st;
  if ((st = preprocess_impl(O, dO, B, T, H, HKV, head_dim, dtype, workspace, workspace_bytes, stream)) != FA_OK)
    return st;
  if ((st = dkdv_impl(Q, K, V, LSE, dO, dK, dV, B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                      workspace_bytes, stream)) != FA_OK)
    return st;
  // dQ reads nothing that dK/dV writes: its CTAs may start on the SMs that
  // the dK/dV kernel leaves idle (fewer units than SMs, or its tail)
  return dq_impl(Q, K, V, LSE, dO, dQ, B, T, Tk, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                 workspace_bytes, stream, /*after_dkdv=*/true);
}

}  // namespace

extern "C" {

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int T, int H, int HKV,
           int head_dim, float scale, int causal, int window, int dtype, void* workspace, size_t workspace_bytes,
           void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, T, T, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                  workspace_bytes, stream);
}

int fa_fwd_cross(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Tq, int Tk, int H,
                 int HKV, int head_dim, float scale, int dtype, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, Tq, Tk, H, HKV, head_dim, scale, 0, 0, dtype, workspace, workspace_bytes,
                  stream);
}

int fa_bwd_preprocess(const void* O, const void* dO, int B, int T, int H, int HKV, int head_dim, int dtype,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return preprocess_impl(O, dO, B, T, H, HKV, head_dim, dtype, workspace, workspace_bytes, stream);
}

int fa_bwd_dkdv(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dK, void* dV,
                int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
                void* workspace, size_t workspace_bytes, void* stream) {
  return dkdv_impl(Q, K, V, LSE, dO, dK, dV, B, T, T, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                   workspace_bytes, stream);
}

int fa_bwd_dq(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ, int B, int T,
              int H, int HKV, int head_dim, float scale, int causal, int window, int dtype, void* workspace,
              size_t workspace_bytes, void* stream) {
  return dq_impl(Q, K, V, LSE, dO, dQ, B, T, T, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                 workspace_bytes, stream);
}

int fa_bwd_dkdv_dq(const void* Q, const void* K, const void* V, const float* LSE, const void* dO, void* dQ, void* dK,
                   void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream) {
  return fused_impl(Q, K, V, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype, workspace,
                    workspace_bytes, stream);
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO, void* dQ,
           void* dK, void* dV, int B, int T, int H, int HKV, int head_dim, float scale, int causal, int window,
           int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, LSE, dO, dQ, dK, dV, B, T, T, H, HKV, head_dim, scale, causal, window, dtype,
                  workspace, workspace_bytes, stream);
}

int fa_bwd_cross(const void* Q, const void* K, const void* V, const void* O, const float* LSE, const void* dO,
                 void* dQ, void* dK, void* dV, int B, int Tq, int Tk, int H, int HKV, int head_dim, float scale,
                 int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, LSE, dO, dQ, dK, dV, B, Tq, Tk, H, HKV, head_dim, scale, 0, 0, dtype, workspace,
                  workspace_bytes, stream);
}

int fa_check_status(void* workspace, void* stream, unsigned int* raw_word) {
  if (!workspace) return FA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (raw_word) *raw_word = word;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel wait timed out";
    case FA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
  }
}

int fa_plan_kv_range(int T, int BM, int BN, int causal, int window, int qb, int* lo, int* hi) {
  if (T < 1 || BM < 1 || BN < 1 || window < 0 || !lo || !hi || qb < 0 || qb >= fa::ceil_div(T, BM))
    return FA_ERR_INVALID_ARG;
  fa::kv_range_for_q(T, T, BM, BN, causal, window, qb, *lo, *hi);
  return FA_OK;
}

int fa_plan_q_range(int T, int BM, int BN, int causal, int window, int kb, int* lo, int* hi) {
  if (T < 1 || BM < 1 || BN < 1 || window < 0 || !lo || !hi || kb < 0 || kb >= fa::ceil_div(T, BN))
    return FA_ERR_INVALID_ARG;
  fa::q_range_for_kv(T, T, BM, BN, causal, window, kb, *lo, *hi);
  return FA_OK;
}

int fa_plan_row_keys(int Tq, int Tk, int causal, int window, int i, int* lo, int* hi) {
  if (Tq < 1 || Tk < 1 || window < 0 || i < 0 || !lo || !hi) return FA_ERR_INVALID_ARG;
  fa::visible_keys(Tq, Tk, causal, window, i, *lo, *hi);
  return FA_OK;
}

int fa_plan_key_rows(int Tq, int Tk, int causal, int window, int j, int* lo, int* hi) {
  if (Tq < 1 || Tk < 1 || window < 0 || j < 0 || !lo || !hi) return FA_ERR_INVALID_ARG;
  fa::visible_queries(Tq, Tk, causal, window, j, *lo, *hi);
  return FA_OK;
}

int fa_plan_block_mask(int T, int BM, int BN, int causal, int window, int qb, int kb) {
  if (T < 1 || BM < 1 || BN < 1 || window < 0 || qb < 0 || kb < 0) return -FA_ERR_INVALID_ARG;
  return fa::block_needs_mask(T, T, BM, BN, causal, window, qb, kb) ? 1 : 0;
}

int fa_qk_norm_rope_fwd(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens, int hq,
                        int hk, int head_dim, int dtype, void* stream) {
  if (tokens < 1 || hq < 1 || hk < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(tokens) * (hq + hk) * head_dim >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
  const void* ptrs[5] = {qk, f1, f2, q, k};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  int dev, st;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  return status_of(fa::launch_qk_norm_rope_fwd(qk, f1, f2, q, k, tokens, hq, hk, head_dim, dtype == FA_DTYPE_FP16,
                                               g_dev[dev].sms, static_cast<cudaStream_t>(stream)));
}

int fa_qk_norm_rope_bwd(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2, void* dqk,
                        int tokens, int hq, int hk, int head_dim, int dtype, void* stream) {
  if (tokens < 1 || hq < 1 || hk < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(tokens) * (hq + hk) * head_dim >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
  const void* ptrs[6] = {dq, dk, qk, f1, f2, dqk};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  int dev, st;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  return status_of(fa::launch_qk_norm_rope_bwd(dq, dk, qk, f1, f2, dqk, tokens, hq, hk, head_dim,
                                               dtype == FA_DTYPE_FP16, g_dev[dev].sms,
                                               static_cast<cudaStream_t>(stream)));
}

namespace {
int qk_opt_check(int tokens, int heads, int head_dim, int rotary_dim, int paired, int key_offset, int dtype) {
  if (tokens < 1 || heads < 1) return FA_ERR_INVALID_ARG;
  if (paired && key_offset) return FA_ERR_INVALID_ARG;  // the options are exclusive
  if (paired && heads % 2) return FA_ERR_INVALID_ARG;
  if (key_offset && (rotary_dim < 0 || rotary_dim > head_dim || rotary_dim % 2)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(tokens) * 2 * heads * head_dim >= (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}
}  // namespace

int fa_qk_norm_rope_fwd_opt(const void* qk, const float* f1, const float* f2, void* q, void* k, int tokens,
                            int heads, int head_dim, int rotary_dim, int paired, int key_offset, int dtype,
                            void* stream) {
  int st = qk_opt_check(tokens, heads, head_dim, rotary_dim, paired, key_offset, dtype);
  if (st != FA_OK) return st;
  const void* ptrs[5] = {qk, f1, f2, q, k};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  int dev;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  return status_of(fa::launch_qk_norm_rope_fwd_opt(qk, f1, f2, q, k, tokens, heads, head_dim, rotary_dim,
                                                   paired != 0, key_offset != 0, dtype == FA_DTYPE_FP16,
                                                   g_dev[dev].sms, static_cast<cudaStream_t>(stream)));
}

int fa_qk_norm_rope_bwd_opt(const void* dq, const void* dk, const void* qk, const float* f1, const float* f2,
                            void* dqk, int tokens, int heads, int head_dim, int rotary_dim, int paired, int key_offset,
                            int dtype, void* stream) {
  int st = qk_opt_check(tokens, heads, head_dim, rotary_dim, paired, key_offset, dtype);
  if (st != FA_OK) return st;
  const void* ptrs[6] = {dq, dk, qk, f1, f2, dqk};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  int dev;
  if ((st = device_ok(&dev)) != FA_OK) return st;
  return status_of(fa::launch_qk_norm_rope_bwd_opt(dq, dk, qk, f1, f2, dqk, tokens, heads, head_dim, rotary_dim,
                                                   paired != 0, key_offset != 0, dtype == FA_DTYPE_FP16,
                                                   g_dev[dev].sms, static_cast<cudaStream_t>(stream)));
}

int fa_tile_m(void) { return fa::kBM; }
int fa_tile_n(void) { return fa::kBN; }

int fa_debug_max_ctas(int ctas) {
  if (ctas < 0) return FA_ERR_INVALID_ARG;
  g_max_ctas.store(ctas);
  return FA_OK;
}

int fa_debug_fwd_tiles(int tiles) {
  if (tiles < 0 || tiles > 3) return FA_ERR_INVALID_ARG;
  g_fwd_tiles.store(tiles);
  return FA_OK;
}

int fa_debug_config(unsigned long long wait_timeout_ns, int inject_stall) {
  g_wait_ns.store(wait_timeout_ns ? wait_timeout_ns : fa::kDefaultWaitNs);
  if (inject_stall < 0 || inject_stall > 3) return FA_ERR_INVALID_ARG;
  g_inject_stall.store(inject_stall);
  return FA_OK;
}

}  // extern "C"
