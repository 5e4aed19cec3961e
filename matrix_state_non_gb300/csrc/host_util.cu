// Host-side helpers shared by the kernel launchers: TMA tensor-map encoding
// through the driver entry point (no link-time dependency on libcuda), and the
// process-wide switches for tests and measurements.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "mma_common.cuh"

namespace m2rnn {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}
}  // namespace

bool make_tensor_map_btnx(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int B,
                          int T, int N, int X, int bx, int by) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(X), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(X) * esize, static_cast<cuuint64_t>(N) * X * esize,
                           static_cast<cuuint64_t>(T) * N * X * esize};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(bx), 1, static_cast<cuuint32_t>(by), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {
// -2 = not yet read from the environment.
std::atomic<int> g_kernel_family{-2};
std::atomic<int> g_stall_tile{-2};
std::once_flag g_env_once;

void read_env_once() {
  std::call_once(g_env_once, [] {
    int fam = -1;
    if (const char* e = std::getenv("M2RNN_KERNEL")) {
      if (std::strcmp(e, "tcgen05") == 0) fam = 1;
      else if (std::strcmp(e, "mma") == 0) fam = 2;
      else if (std::strcmp(e, "simt") == 0) fam = 0;
    }
    int stall = -1;
    if (const char* e = std::getenv("M2RNN_TEST_STALL_TILE")) stall = std::atoi(e);
    int expect = -2;
    g_kernel_family.compare_exchange_strong(expect, fam);
    expect = -2;
    g_stall_tile.compare_exchange_strong(expect, stall);
  });
}
}  // namespace

int option_kernel_family() {
  read_env_once();
  return g_kernel_family.load(std::memory_order_relaxed);
}

int option_test_stall_tile() {
  read_env_once();
  return g_stall_tile.load(std::memory_order_relaxed);
}

int set_option(int option, int value, int* previous) {
  read_env_once();
  if (option == M2RNN_OPT_KERNEL_FAMILY) {
    if (value < -1 || value > 2) return M2RNN_ERR_INVALID_ARG;
    const int old = g_kernel_family.exchange(value);
    if (previous != nullptr) *previous = old;
    return M2RNN_OK;
  }
  if (option == M2RNN_OPT_TEST_STALL_TILE) {
    if (value < -1) return M2RNN_ERR_INVALID_ARG;
    const int old = g_stall_tile.exchange(value);
    if (previous != nullptr) *previous = old;
    return M2RNN_OK;
  }
  return M2RNN_ERR_INVALID_ARG;
}

}  // namespace m2rnn
