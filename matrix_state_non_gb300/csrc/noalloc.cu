// m2rnn_backward_noalloc: the backward scan for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a workspace: code running inside a
// runtime that owns all device allocations (and hands out none), plug-ins
// loaded into a host that forbids cudaMalloc, or code paths that must not
// allocate because an allocation would synchronise or fail at that point.
// For them this entry point keeps its scratch in a fixed array inside the
// library's device image, so the caller passes only inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kStaticScratchBytes) until the process exits.  In host
// code its name is only a host-side handle, so the device address is looked
// up with cudaGetSymbolAddress (with the device current) on the first call
// made on a device, and passed to the kernels.  The address is kept per
// device together with the identity of the context it belongs to; if that
// context is replaced (cudaDeviceReset, then a new primary context), the next
// call looks the address up again instead of using a stale one.
//
// All calls share the one array and it keeps the previous call's contents:
// the status block is cleared at the start of each call, everything else is
// fully overwritten before it is read.  Calls that overlap on the GPU (on
// different streams, or from different host threads without ordering) race
// on the array and corrupt each other's results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace m2rnn {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

struct DeviceScratch {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;
};
std::mutex g_addr_mu;
DeviceScratch g_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Identity of the current context (0 if the driver cannot tell).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch on the current device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return M2RNN_ERR_UNSUPPORTED;
  // 0 while this thread has no current context yet: then the lookup below
  // (which makes the device's primary context current) runs.
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_addr_mu);
  DeviceScratch& e = g_addr[dev];
  if (e.addr == nullptr || ctx == 0 || e.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return M2RNN_ERR_CUDA;
    e.addr = p;
    e.ctx_id = current_context_id();
  }
  *out = e.addr;
  return M2RNN_OK;
}

// Stream-ordered read (and clear) of the array's status block.
int read_status(StatusBlock* status, cudaStream_t s, uint32_t* detail) {
  unsigned int host[2] = {0u, 0u};
  if (cudaMemcpyAsync(host, status, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(host), s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (detail != nullptr) *detail = host[1];
  if (host[0] == 0u) return M2RNN_OK;
  return host[0] == kStatusTimeout ? M2RNN_ERR_TIMEOUT : M2RNN_ERR_DEVICE;
}

inline size_t round256(size_t x) { return (x + 255) / 256 * 256; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace m2rnn

using namespace m2rnn;

extern "C" int m2rnn_backward_noalloc(const void* q, const void* k, const void* v, const void* f,
                                      const void* W, const void* w_r, const float* dy, const float* dH_T,
                                      const float* ckpt, int ckpt_every, float* dq, float* dk, float* dv,
                                      float* df, float* dW, float* dw_r, int64_t B, int64_t T, int64_t N,
                                      int64_t K, int64_t V, m2rnn_dtype dtype, int sync, void* cuda_stream) {
  if (B < 1 || T < 1 || N < 1 || B > (1 << 20) || N > (1 << 20) || T > (int64_t(1) << 30))
    return M2RNN_ERR_INVALID_ARG;
  if (dtype != M2RNN_BF16 || !mma_backward_supported(static_cast<int>(K), static_cast<int>(V)))
    return M2RNN_ERR_UNSUPPORTED;
  if (ckpt_every < 1 || ckpt_every > mma_backward_max_chunk()) return M2RNN_ERR_UNSUPPORTED;
  const int64_t nck = (T - 1) / ckpt_every;
  if (nck > 0 && ckpt == nullptr) return M2RNN_ERR_INVALID_ARG;  // checkpoints must come from the forward
  const void* req[] = {q, k, v, f, W, w_r, dy, dq, dk, dv, df, dW, dw_r};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return M2RNN_ERR_INVALID_ARG;
  if ((dH_T && !aligned16(dH_T)) || (ckpt && !aligned16(ckpt))) return M2RNN_ERR_INVALID_ARG;

  const int parts = static_cast<int>(K) / 16;
  const size_t status_bytes = sizeof(StatusBlock);
  const size_t dwp_bytes = round256(sizeof(float) * static_cast<size_t>(B * N * parts) * V * V);
  const size_t dwr_bytes = round256(sizeof(float) * static_cast<size_t>(B * N) * V);
  const size_t scr_bytes = round256(mma_backward_scratch_bytes(static_cast<int>(B), static_cast<int>(T),
                                                               static_cast<int>(N), static_cast<int>(K),
                                                               static_cast<int>(V), ckpt_every));
  if (status_bytes + dwp_bytes + dwr_bytes + scr_bytes > kStaticScratchBytes)
    return M2RNN_ERR_WORKSPACE;  // the problem needs more scratch than the built-in array holds

  void* base = nullptr;
  const int st = scratch_address(&base);
  if (st != M2RNN_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(base);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  StatusBlock* status = reinterpret_cast<StatusBlock*>(ws);
  if (cudaMemsetAsync(status, 0, status_bytes, s) != cudaSuccess) return M2RNN_ERR_CUDA;

  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.f = f; a.W = W; a.w_r = w_r;
  a.dy = dy; a.dH_T = dH_T; a.ckpt = ckpt; a.ckpt_every = ckpt_every; a.n_ckpt = nck;
  a.dq = dq; a.dk = dk; a.dv = dv; a.df = df; a.dW = dW; a.dw_r = dw_r;
  a.B = static_cast<int>(B); a.T = static_cast<int>(T); a.N = static_cast<int>(N);
  a.K = static_cast<int>(K); a.V = static_cast<int>(V);
  a.dtype = dtype;
  a.status = status;
  a.dW_part = reinterpret_cast<float*>(ws + status_bytes);
  a.dwr_part = reinterpret_cast<float*>(ws + status_bytes + dwp_bytes);
  a.scratch = reinterpret_cast<float*>(ws + status_bytes + dwp_bytes + dwr_bytes);
  a.parts = parts;
  if (launch_mma_backward(a, s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (launch_reduce_partials(a, s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (!sync) return M2RNN_OK;
  return read_status(status, s, nullptr);
}

extern "C" int m2rnn_backward_noalloc_status(void* cuda_stream, uint32_t* detail) {
  void* base = nullptr;
  const int st = scratch_address(&base);
  if (st != M2RNN_OK) return st;
  return read_status(reinterpret_cast<StatusBlock*>(base), static_cast<cudaStream_t>(cuda_stream), detail);
}
