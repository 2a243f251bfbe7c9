// fa_static_scratch.cu -- fa_bwd for callers that cannot allocate device memory.
//
// fa_bwd needs scratch beyond its inputs and outputs: Delta = rowsum(dO * O)
// (B*H*T floats) and a 4-byte device error word, which callers normally pass
// as a workspace they allocated.  Some callers cannot call cudaMalloc at all:
// code running inside another allocator's callback, plugins of host programs
// that own every device allocation, or paths that must not touch the
// allocator while a CUDA graph is being built.  fa_bwd_static_scratch gives
// them the same backward with its scratch in the fixed device array below,
// which the library carries in its own image: every GPU that loads the
// library keeps these bytes allocated until the process exits.
//
// The array's name means a device address only in device code.  In host
// code it is a host-side shadow symbol; passing it to a kernel would fault
// or, where the GPU can reach host memory, silently use the wrong memory.
// Host code must ask the runtime for the device address, once per device,
// with that device current (cudaGetSymbolAddress), which is what
// scratch_address() does and caches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// 256 bytes for the error word (the layout fa_workspace_size describes),
// then room for Delta of up to FA_STATIC_SCRATCH_MAX_ROWS rows.
constexpr size_t kErrBytes = 256;
constexpr size_t kScratchBytes = kErrBytes + sizeof(float) * static_cast<size_t>(FA_STATIC_SCRATCH_MAX_ROWS);

static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};  // id of the context g_addr[dev] belongs to (0 = none)
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

// Id of the current context (unique for the life of the process), or 0 if it
// cannot be read.  A context torn down and created again (cudaDeviceReset)
// gets a new id, and the module holding the array is loaded again there.
unsigned long long current_ctx_id() {
  if (g_ctx_get_id == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return 0;
    g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  }
  unsigned long long id = 0;
  return g_ctx_get_id(nullptr, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_static_scratch in the current device's current
// context, looked up once per (device, context), or nullptr if the runtime
// could not provide it.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  const unsigned long long id = current_ctx_id();
  if (g_addr[dev] != nullptr && id != 0 && g_ctx[dev] == id) return g_addr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
  // the lookup above made the device's primary context current if none was
  g_addr[dev] = p;
  g_ctx[dev] = current_ctx_id();
  return p;
}

}  // namespace

extern "C" int fa_bwd_static_scratch(const void* Q, const void* K, const void* V, const void* O, const float* LSE,
                                     const void* dO, void* dQ, void* dK, void* dV, int B, int T, int H, int HKV,
                                     int head_dim, float scale, int causal, int window, int dtype,
                                     unsigned int* err_word, void* stream) {
  if (B < 1 || T < 1 || H < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * T > FA_STATIC_SCRATCH_MAX_ROWS) return FA_ERR_WORKSPACE;
  const size_t need = fa_workspace_size(FA_OP_BWD, B, T, H, HKV, head_dim, dtype);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kScratchBytes) return FA_ERR_WORKSPACE;
  if (err_word && (reinterpret_cast<uintptr_t>(err_word) & 3u)) return FA_ERR_INVALID_ARG;
  void* ws = scratch_address();
  if (ws == nullptr) return FA_ERR_CUDA;
  // every check fa_bwd makes, before anything goes onto the stream: a call
  // that fails here has launched nothing
  int st = fa::check_bwd_call(Q, K, V, O, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype,
                              ws, kScratchBytes);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left: the error word must
  // start at zero for this call (Delta is fully rewritten before it is read).
  if (cudaMemsetAsync(ws, 0, sizeof(unsigned int), s) != cudaSuccess) return FA_ERR_CUDA;
  st = fa_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, T, H, HKV, head_dim, scale, causal, window, dtype, ws,
              kScratchBytes, stream);
  if (st != FA_OK) return st;
  if (err_word && cudaMemcpyAsync(err_word, ws, sizeof(unsigned int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
