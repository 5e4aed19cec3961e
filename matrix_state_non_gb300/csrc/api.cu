// C-ABI entry points of libm2rnn.so (declared in include/m2rnn.h): argument
// validation, workspace carving and kernel dispatch.  Every step of both
// scans runs in this library's CUDA kernels; nothing runs on the host CPU.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "gate.cuh"
#include "internal.h"

using namespace m2rnn;

namespace {

constexpr size_t kStatusBytes = sizeof(StatusBlock);
constexpr int kMaxDim = 128;
constexpr int kMaxCkptEvery = 4096;

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(int64_t B, int64_t T, int64_t N, int64_t K, int64_t V) {
  if (B < 1 || T < 1 || N < 1 || K < 1 || V < 1) return false;
  if (B > INT_MAX / 8 || T > INT_MAX || N > INT_MAX / 8) return false;
  if (B * N > INT_MAX / 8) return false;
  return true;
}

bool dtype_ok(int dt) { return dt == M2RNN_F32 || dt == M2RNN_BF16; }

constexpr int kPathSimt = 0, kPathTc = 1, kPathMma = 2;

// Kernel family override for tests and benchmarks (m2rnn_set_option; first
// read from M2RNN_KERNEL = auto | tcgen05 | mma | simt).  A family that does
// not support the shape falls back to the automatic choice.
int kernel_override() {
  switch (option_kernel_family()) {
    case 1: return kPathTc;
    case 2: return kPathMma;
    case 0: return kPathSimt;
    default: return -1;
  }
}

// Which family runs the forward: 2 = warp-MMA, 1 = tcgen05, 0 = SIMT fp32, <0 = error.
int choose_path(int64_t K, int64_t V, int dt) {
  if (!dtype_ok(dt)) return M2RNN_ERR_INVALID_ARG;
  if (K < 1 || V < 1) return M2RNN_ERR_INVALID_ARG;
  if (K > kMaxDim || V > kMaxDim) return M2RNN_ERR_UNSUPPORTED;
  if (dt != M2RNN_BF16) return kPathSimt;
  const int k = static_cast<int>(K), v = static_cast<int>(V);
  const bool mma = mma_forward_supported(k, v), tc = tc_forward_supported(k, v);
  switch (kernel_override()) {
    case kPathTc: if (tc) return kPathTc; break;
    case kPathMma: if (mma) return kPathMma; break;
    case kPathSimt: return kPathSimt;
    default: break;
  }
  // V = 64: both tensor-core forwards hold ~16 state rows per SM and are
  // bound by the step latency; the warp-MMA scan with its readout on
  // separate warps measured ~9 % shorter (196 vs 216 ns per step on the
  // T = 16384 workload).  It also writes the Z stash.
  if (mma) return kPathMma;  // V = 64 and V = 16: the register-resident warp-MMA scans
  if (tc) return kPathTc;    // wide heads: tensor throughput matters
  return kPathSimt;
}

// Backward family (the tensor-core backwards cover fewer shapes and chunk
// lengths than the forwards).
int choose_bwd_path(int64_t K, int64_t V, int dt, int ckpt_every) {
  const int path = choose_path(K, V, dt);
  if (path < 0) return path;
  const int k = static_cast<int>(K), v = static_cast<int>(V);
  const bool mma = (v == 16) ? mv_backward_supported(k, v, ckpt_every)
                             : mma_backward_supported(k, v) && ckpt_every <= mma_backward_max_chunk();
  const bool tc = tc_backward_supported(k, v);
  if (path == kPathMma && mma) return kPathMma;
  if (path == kPathTc && tc) return kPathTc;
  if (dt == M2RNN_BF16 && kernel_override() != kPathSimt) {
    if (mma) return kPathMma;
    if (tc) return kPathTc;
  }
  return kPathSimt;
}

cudaError_t launch_forward_path(int path, const FwdArgs& a, cudaStream_t s) {
  if (path == kPathMma) return launch_mma_forward(a, s);
  if (path == kPathTc) return launch_tc_forward(a, s);
  return launch_simt_forward(a, s);
}

struct BwdLayout {
  size_t ckpt_off, dwp_off, dwrp_off, scratch_off, qk_off, gate_off, total;
};

// shared_qk: one q/k for every head; the per-head dq, dk go to the workspace
// ([B,T,N,K] each) and are summed over heads into the caller's [B,T,1,K].
BwdLayout bwd_layout(int64_t B, int64_t T, int64_t N, int64_t K, int64_t V, int dt, int C,
                     bool have_ckpt, bool shared_qk = false) {
  BwdLayout l{};
  const int path = choose_bwd_path(K, V, dt, C);
  const int64_t nck = (T - 1) / C;
  const int b = static_cast<int>(B), nn = static_cast<int>(N), k = static_cast<int>(K),
            v = static_cast<int>(V);
  size_t off = kStatusBytes;
  l.ckpt_off = off;
  if (!have_ckpt) off = align256(off + sizeof(float) * static_cast<size_t>(B * N * nck * K * V));
  const int parts = (path == kPathSimt) ? 1 : (path == kPathMma ? k / 16 : tc_backward_parts(k, v));
  l.dwp_off = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(B * N * parts * V * V));
  l.dwrp_off = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(B * N * V));
  l.scratch_off = off;
  if (path == kPathMma)
    off = align256(off + mma_backward_scratch_bytes(b, static_cast<int>(T), nn, k, v, C));
  else if (path == kPathTc)
    off = align256(off + tc_backward_scratch_bytes(b, nn, k, v, C));
  else
    off = align256(off + simt_backward_scratch_bytes(b, nn, k, v, C));
  l.qk_off = off;
  if (shared_qk) off = align256(off + 2 * sizeof(float) * static_cast<size_t>(B * T * N * K));
  l.gate_off = off;  // gate-backward partials (used by the gated backward only)
  off = align256(off + 2 * sizeof(float) * static_cast<size_t>(N) * gate_backward_parts(B * T));
  l.total = off;
  return l;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? M2RNN_OK : M2RNN_ERR_CUDA; }

// Shapes whose forward can leave Z_t for the backward (the tcgen05 forward at V = 64, the
// register-resident warp-MMA forward at V = 16).
bool stash_ok(int64_t K, int64_t V, int dt) {
  return dt == M2RNN_BF16 && (V == 64 || V == 16) && K >= 16 && K <= kMaxDim && K % 16 == 0;
}

}  // namespace

extern "C" {

int m2rnn_version(void) { return 10000; }

const char* m2rnn_status_string(int status) {
  switch (status) {
    case M2RNN_OK: return "ok";
    case M2RNN_ERR_INVALID_ARG: return "invalid argument";
    case M2RNN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case M2RNN_ERR_WORKSPACE: return "workspace missing or too small";
    case M2RNN_ERR_CUDA: return "CUDA error";
    case M2RNN_ERR_TIMEOUT: return "device wait timed out";
    case M2RNN_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
  }
}

int64_t m2rnn_checkpoint_count(int64_t T, int ckpt_every) {
  if (T < 1 || ckpt_every < 1) return -1;
  return (T - 1) / ckpt_every;
}

int m2rnn_path(int64_t K, int64_t V, m2rnn_dtype dtype) { return choose_path(K, V, dtype); }

int m2rnn_set_option(int option, int value, int* previous) { return set_option(option, value, previous); }

size_t m2rnn_forward_workspace_size(int64_t B, int64_t T, int64_t N, int64_t K, int64_t V,
                                    m2rnn_dtype dtype) {
  if (!dims_ok(B, T, N, K, V) || choose_path(K, V, dtype) < 0) return 0;
  return kStatusBytes;
}

size_t m2rnn_backward_workspace_size(int64_t B, int64_t T, int64_t N, int64_t K, int64_t V,
                                     m2rnn_dtype dtype, int ckpt_every, int have_ckpt) {
  if (!dims_ok(B, T, N, K, V) || choose_path(K, V, dtype) < 0) return 0;
  if (ckpt_every < 1 || ckpt_every > kMaxCkptEvery) return 0;
  return bwd_layout(B, T, N, K, V, dtype, ckpt_every, have_ckpt != 0).total;
}

size_t m2rnn_backward_state_workspace_size(int64_t B, int64_t T, int64_t N, int64_t qk_heads,
                                           int64_t K, int64_t V, m2rnn_dtype dtype, int ckpt_every,
                                           int have_ckpt) {
  if (!dims_ok(B, T, N, K, V) || choose_path(K, V, dtype) < 0) return 0;
  if (ckpt_every < 1 || ckpt_every > kMaxCkptEvery || (qk_heads != 1 && qk_heads != N)) return 0;
  return bwd_layout(B, T, N, K, V, dtype, ckpt_every, have_ckpt != 0, qk_heads == 1 && N > 1).total;
}

}  // extern "C"

namespace {

// The forget gate as the caller gives it: f itself, or (a, alpha, beta).
struct GateIn {
  const void* f;
  const void* a;
  const float* alpha;
  const float* beta;
  bool ok() const {
    if (a == nullptr) return f != nullptr && aligned16(f);
    return f == nullptr && aligned16(a) && alpha != nullptr && beta != nullptr && aligned16(alpha) &&
           aligned16(beta);
  }
};

int forward_impl(const void* q, const void* k, const void* v, const GateIn& gate, const void* W,
                 const void* w_r, const float* H_0, float* y, float* H_T, float* ckpt, int ckpt_every,
                 void* z_stash, int64_t B, int64_t T, int64_t N, int64_t qk_heads, int64_t K, int64_t V,
                 m2rnn_dtype dtype, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!dtype_ok(dtype) || !dims_ok(B, T, N, K, V)) return M2RNN_ERR_INVALID_ARG;
  if (qk_heads != 1 && qk_heads != N) return M2RNN_ERR_INVALID_ARG;
  int path = choose_path(K, V, dtype);
  if (path < 0) return path;
  if (z_stash != nullptr) {
    if (!stash_ok(K, V, dtype)) return M2RNN_ERR_UNSUPPORTED;
    if (!aligned16(z_stash)) return M2RNN_ERR_INVALID_ARG;
    path = kPathMma;  // the kernels that write the stash: the warp-MMA forwards (V = 64, V = 16)
  }
  const void* req[] = {q, k, v, W, w_r, y};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return M2RNN_ERR_INVALID_ARG;
  if (!gate.ok()) return M2RNN_ERR_INVALID_ARG;
  if ((H_T && !aligned16(H_T)) || (ckpt && !aligned16(ckpt)) || (H_0 && !aligned16(H_0)))
    return M2RNN_ERR_INVALID_ARG;
  if (ckpt && (ckpt_every < 1 || ckpt_every > kMaxCkptEvery)) return M2RNN_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < kStatusBytes)
    return M2RNN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  StatusBlock* status = static_cast<StatusBlock*>(workspace);
  cudaError_t e = cudaMemsetAsync(status, 0, kStatusBytes, s);
  if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  FwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.f = gate.f; a.W = W; a.w_r = w_r;
  a.gate_a = gate.a; a.gate_alpha = gate.alpha; a.gate_beta = gate.beta;
  a.H0 = H_0; a.qkN = static_cast<int>(qk_heads); a.y = y; a.H_T = H_T; a.ckpt = ckpt;
  a.zstash = static_cast<uint16_t*>(z_stash);
  a.ckpt_every = ckpt ? ckpt_every : 1;
  a.n_ckpt = ckpt ? (T - 1) / ckpt_every : 0;
  a.B = static_cast<int>(B); a.T = static_cast<int>(T); a.N = static_cast<int>(N);
  a.K = static_cast<int>(K); a.V = static_cast<int>(V);
  a.dtype = dtype;
  a.status = status;
  e = launch_forward_path(path, a, s);
  return cuda_status(e);
}

}  // namespace

extern "C" {

int m2rnn_forward_state(const void* q, const void* k, const void* v, const void* f, const void* W,
                        const void* w_r, const float* H_0, float* y, float* H_T, float* ckpt,
                        int ckpt_every, void* z_stash, int64_t B, int64_t T, int64_t N, int64_t qk_heads, int64_t K,
                        int64_t V, m2rnn_dtype dtype, void* workspace, size_t workspace_bytes,
                        void* cuda_stream) {
  if (f == nullptr) return M2RNN_ERR_INVALID_ARG;
  return forward_impl(q, k, v, GateIn{f, nullptr, nullptr, nullptr}, W, w_r, H_0, y, H_T, ckpt, ckpt_every,
                      z_stash, B, T, N, qk_heads, K, V, dtype, workspace, workspace_bytes, cuda_stream);
}

int m2rnn_forward_gated(const void* q, const void* k, const void* v, const void* a, const float* alpha,
                        const float* beta, const void* W, const void* w_r, const float* H_0, float* y,
                        float* H_T, float* ckpt, int ckpt_every, void* z_stash, int64_t B, int64_t T, int64_t N,
                        int64_t qk_heads, int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace,
                        size_t workspace_bytes, void* cuda_stream) {
  if (a == nullptr) return M2RNN_ERR_INVALID_ARG;
  return forward_impl(q, k, v, GateIn{nullptr, a, alpha, beta}, W, w_r, H_0, y, H_T, ckpt, ckpt_every, z_stash,
                      B, T, N, qk_heads, K, V, dtype, workspace, workspace_bytes, cuda_stream);
}

int m2rnn_forward(const void* q, const void* k, const void* v, const void* f, const void* W,
                  const void* w_r, float* y, float* H_T, float* ckpt, int ckpt_every, int64_t B,
                  int64_t T, int64_t N, int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace,
                  size_t workspace_bytes, void* cuda_stream) {
  return m2rnn_forward_state(q, k, v, f, W, w_r, nullptr, y, H_T, ckpt, ckpt_every, nullptr, B, T, N, N, K, V,
                             dtype, workspace, workspace_bytes, cuda_stream);
}

int m2rnn_decode_step(float* H, const void* q, const void* k, const void* v, const void* f,
                      const void* W, const void* w_r, float* y, int64_t B, int64_t N, int64_t qk_heads,
                      int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* cuda_stream) {
  if (H == nullptr || (qk_heads != 1 && qk_heads != N)) return M2RNN_ERR_INVALID_ARG;
  if (dtype_ok(dtype) && dims_ok(B, 1, N, K, V) && decode_kernel_supported(static_cast<int>(K), static_cast<int>(V), dtype) &&
      kernel_override() < 0) {
    const void* req[] = {H, q, k, v, f, W, w_r, y};
    for (const void* p : req)
      if (!aligned16(p)) return M2RNN_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < kStatusBytes)
      return M2RNN_ERR_WORKSPACE;
    return cuda_status(launch_decode_step(H, q, k, v, f, W, w_r, y, static_cast<int>(B), static_cast<int>(N),
                                          static_cast<int>(K), static_cast<int>(qk_heads),
                                          static_cast<StatusBlock*>(workspace),
                                          static_cast<cudaStream_t>(cuda_stream)));
  }
  // Otherwise the scan kernels with T = 1, from H to H: every kernel reads a
  // state element before the same thread block overwrites it.
  return m2rnn_forward_state(q, k, v, f, W, w_r, H, y, H, nullptr, 0, nullptr, B, 1, N, qk_heads, K, V, dtype,
                             workspace, workspace_bytes, cuda_stream);
}

}  // extern "C"

namespace {

// df receives the gradient of f; with a gate given as (a, alpha, beta) it
// then becomes da in place, and dalpha, dbeta [N] are written.
int backward_impl(const void* q, const void* k, const void* v, const GateIn& gate, const void* W,
                  const void* w_r, const float* H_0, const float* dy, const float* dH_T, const float* ckpt,
                  int ckpt_every, const void* z_stash, float* dq, float* dk, float* dv, float* df, float* dalpha, float* dbeta,
                  float* dW, float* dw_r, float* dH_0, float state_grad_clip, int64_t B, int64_t T, int64_t N,
                  int64_t qk_heads, int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace,
                  size_t workspace_bytes, void* cuda_stream) {
  if (!(state_grad_clip >= 0.f)) return M2RNN_ERR_INVALID_ARG;  // also rejects NaN
  if (!dtype_ok(dtype) || !dims_ok(B, T, N, K, V)) return M2RNN_ERR_INVALID_ARG;
  if (qk_heads != 1 && qk_heads != N) return M2RNN_ERR_INVALID_ARG;
  const bool shared_qk = qk_heads == 1 && N > 1;
  const int path = choose_path(K, V, dtype);
  if (path < 0) return path;
  int bpath = choose_bwd_path(K, V, dtype, ckpt_every);
  if (ckpt_every < 1 || ckpt_every > kMaxCkptEvery) return M2RNN_ERR_INVALID_ARG;
  if (z_stash != nullptr) {
    const bool chunk_ok = (V == 16) ? mv_backward_supported(static_cast<int>(K), 16, ckpt_every)
                                    : ckpt_every <= mma_backward_max_chunk();
    if (!stash_ok(K, V, dtype) || !chunk_ok) return M2RNN_ERR_UNSUPPORTED;
    if (!aligned16(z_stash)) return M2RNN_ERR_INVALID_ARG;
    if (ckpt == nullptr && (T - 1) / ckpt_every > 0) return M2RNN_ERR_INVALID_ARG;  // stash and checkpoints go together
    bpath = kPathMma;  // the kernel that reads the stash
  }
  const void* req[] = {q, k, v, W, w_r, dy, dq, dk, dv, df, dW, dw_r};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return M2RNN_ERR_INVALID_ARG;
  if (!gate.ok()) return M2RNN_ERR_INVALID_ARG;
  if (gate.a != nullptr && (dalpha == nullptr || dbeta == nullptr || !aligned16(dalpha) || !aligned16(dbeta)))
    return M2RNN_ERR_INVALID_ARG;
  if (gate.a != nullptr && N > 65535) return M2RNN_ERR_UNSUPPORTED;  // heads index the grid's y dimension
  if ((dH_T && !aligned16(dH_T)) || (ckpt && !aligned16(ckpt)) || (H_0 && !aligned16(H_0)) ||
      (dH_0 && !aligned16(dH_0)))
    return M2RNN_ERR_INVALID_ARG;
  const BwdLayout l = bwd_layout(B, T, N, K, V, dtype, ckpt_every, ckpt != nullptr, shared_qk);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < l.total)
    return M2RNN_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  StatusBlock* status = reinterpret_cast<StatusBlock*>(ws);
  cudaError_t e = cudaMemsetAsync(status, 0, kStatusBytes, s);
  if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  const int64_t nck = (T - 1) / ckpt_every;
  float* ck = const_cast<float*>(ckpt);
  if (ck == nullptr) {
    ck = reinterpret_cast<float*>(ws + l.ckpt_off);
    if (nck > 0) {
      // Checkpoint pass: the forward without the readout.
      FwdArgs fa{};
      fa.q = q; fa.k = k; fa.v = v; fa.f = gate.f; fa.W = W; fa.w_r = w_r;
      fa.gate_a = gate.a; fa.gate_alpha = gate.alpha; fa.gate_beta = gate.beta;
      fa.H0 = H_0; fa.qkN = static_cast<int>(qk_heads); fa.y = nullptr; fa.H_T = nullptr; fa.ckpt = ck;
      fa.ckpt_every = ckpt_every; fa.n_ckpt = nck;
      fa.B = static_cast<int>(B); fa.T = static_cast<int>(T); fa.N = static_cast<int>(N);
      fa.K = static_cast<int>(K); fa.V = static_cast<int>(V);
      fa.dtype = dtype; fa.status = status;
      e = launch_forward_path(path, fa, s);
      if (e != cudaSuccess) return M2RNN_ERR_CUDA;
    }
  }
  BwdArgs a{};
  a.q = q; a.k = k; a.v = v; a.f = gate.f; a.W = W; a.w_r = w_r;
  a.gate_a = gate.a; a.gate_alpha = gate.alpha; a.gate_beta = gate.beta;
  a.dy = dy; a.dH_T = dH_T; a.H0 = H_0; a.ckpt = ck; a.ckpt_every = ckpt_every; a.n_ckpt = nck;
  a.zstash = static_cast<const uint16_t*>(z_stash);
  a.dq = dq; a.dk = dk; a.dv = dv; a.df = df; a.dW = dW; a.dw_r = dw_r; a.dH0 = dH_0;
  a.clip = state_grad_clip;
  a.qkN = static_cast<int>(qk_heads);
  float* dq_heads = reinterpret_cast<float*>(ws + l.qk_off);
  float* dk_heads = dq_heads + B * T * N * K;
  if (shared_qk) {  // per-head gradients first, summed over the heads below
    a.dq = dq_heads;
    a.dk = dk_heads;
  }
  a.B = static_cast<int>(B); a.T = static_cast<int>(T); a.N = static_cast<int>(N);
  a.K = static_cast<int>(K); a.V = static_cast<int>(V);
  a.dtype = dtype; a.status = status;
  a.dW_part = reinterpret_cast<float*>(ws + l.dwp_off);
  a.dwr_part = reinterpret_cast<float*>(ws + l.dwrp_off);
  a.scratch = reinterpret_cast<float*>(ws + l.scratch_off);
  a.parts = (bpath == kPathSimt) ? 1 : (bpath == kPathMma ? a.K / 16 : tc_backward_parts(a.K, a.V));
  if (bpath == kPathMma)
    e = launch_mma_backward(a, s);
  else if (bpath == kPathTc)
    e = launch_tc_backward(a, s);
  else
    e = launch_simt_backward(a, s);
  if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  if (shared_qk) {
    e = launch_sum_qk_heads(dq_heads, dk_heads, dq, dk, B * T, static_cast<int>(N), static_cast<int>(K), s);
    if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  }
  e = launch_reduce_partials(a, s);
  if (e != cudaSuccess) return M2RNN_ERR_CUDA;
  if (gate.a != nullptr) {
    const GateSrc gs{nullptr, gate.a, gate.alpha, gate.beta, dtype == M2RNN_BF16};
    e = launch_gate_backward(gs, df, dalpha, dbeta, reinterpret_cast<float*>(ws + l.gate_off), B * T,
                             static_cast<int>(N), s);
  }
  return cuda_status(e);
}

}  // namespace

extern "C" {

int m2rnn_backward_state(const void* q, const void* k, const void* v, const void* f,
                         const void* W, const void* w_r, const float* H_0, const float* dy,
                         const float* dH_T, const float* ckpt, int ckpt_every, const void* z_stash, float* dq,
                         float* dk, float* dv, float* df, float* dW, float* dw_r, float* dH_0,
                         float state_grad_clip, int64_t B, int64_t T, int64_t N, int64_t qk_heads,
                         int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* cuda_stream) {
  if (f == nullptr) return M2RNN_ERR_INVALID_ARG;
  return backward_impl(q, k, v, GateIn{f, nullptr, nullptr, nullptr}, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every,
                       z_stash, dq, dk, dv, df, nullptr, nullptr, dW, dw_r, dH_0, state_grad_clip, B, T, N, qk_heads, K,
                       V, dtype, workspace, workspace_bytes, cuda_stream);
}

int m2rnn_backward_gated(const void* q, const void* k, const void* v, const void* a, const float* alpha,
                         const float* beta, const void* W, const void* w_r, const float* H_0, const float* dy,
                         const float* dH_T, const float* ckpt, int ckpt_every, const void* z_stash, float* dq, float* dk, float* dv,
                         float* da, float* dalpha, float* dbeta, float* dW, float* dw_r, float* dH_0,
                         float state_grad_clip, int64_t B, int64_t T, int64_t N, int64_t qk_heads, int64_t K,
                         int64_t V, m2rnn_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* cuda_stream) {
  if (a == nullptr) return M2RNN_ERR_INVALID_ARG;
  return backward_impl(q, k, v, GateIn{nullptr, a, alpha, beta}, W, w_r, H_0, dy, dH_T, ckpt, ckpt_every, z_stash,
                       dq, dk,
                       dv, da, dalpha, dbeta, dW, dw_r, dH_0, state_grad_clip, B, T, N, qk_heads, K, V, dtype,
                       workspace, workspace_bytes, cuda_stream);
}

size_t m2rnn_z_stash_size(int64_t B, int64_t T, int64_t N, int64_t K, int64_t V, m2rnn_dtype dtype) {
  if (!dims_ok(B, T, N, K, V) || !stash_ok(K, V, dtype)) return 0;
  return static_cast<size_t>(B) * T * N * K * V * 2;
}

size_t m2rnn_output_norm_backward_workspace_size(int64_t B, int64_t T, int64_t N, int64_t V) {
  if (!dims_ok(B, T, N, 1, V) || N * V > output_norm_max_width()) return 0;
  const int64_t rows = B * T;
  const int d = static_cast<int>(N * V);
  return align256(sizeof(float) * static_cast<size_t>(output_norm_backward_parts(rows, d)) * d);
}

int m2rnn_output_norm(const float* y, const void* g, const float* w, float eps, float* out, float* rstd,
                      int64_t B, int64_t T, int64_t N, int64_t V, m2rnn_dtype dtype, void* cuda_stream) {
  if (!dtype_ok(dtype) || !dims_ok(B, T, N, 1, V) || !(eps >= 0.f)) return M2RNN_ERR_INVALID_ARG;
  if (N * V > output_norm_max_width()) return M2RNN_ERR_UNSUPPORTED;
  const void* req[] = {y, g, w, out};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return M2RNN_ERR_INVALID_ARG;
  if (rstd && !aligned16(rstd)) return M2RNN_ERR_INVALID_ARG;
  return cuda_status(launch_output_norm(y, g, w, eps, out, rstd, B * T, static_cast<int>(N * V),
                                        dtype == M2RNN_BF16, static_cast<cudaStream_t>(cuda_stream)));
}

int m2rnn_output_norm_backward(const float* y, const void* g, const float* w, const float* dout, float eps,
                               float* dy, float* dg, float* dw, int64_t B, int64_t T, int64_t N, int64_t V,
                               m2rnn_dtype dtype, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!dtype_ok(dtype) || !dims_ok(B, T, N, 1, V) || !(eps >= 0.f)) return M2RNN_ERR_INVALID_ARG;
  if (N * V > output_norm_max_width()) return M2RNN_ERR_UNSUPPORTED;
  const void* req[] = {y, g, w, dout, dy, dg, dw};
  for (const void* p : req)
    if (p == nullptr || !aligned16(p)) return M2RNN_ERR_INVALID_ARG;
  const size_t need = m2rnn_output_norm_backward_workspace_size(B, T, N, V);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return M2RNN_ERR_WORKSPACE;
  return cuda_status(launch_output_norm_backward(y, g, w, dout, eps, dy, dg, dw, static_cast<float*>(workspace),
                                                 B * T, static_cast<int>(N * V), dtype == M2RNN_BF16,
                                                 static_cast<cudaStream_t>(cuda_stream)));
}

int m2rnn_backward(const void* q, const void* k, const void* v, const void* f, const void* W,
                   const void* w_r, const float* dy, const float* dH_T, const float* ckpt,
                   int ckpt_every, float* dq, float* dk, float* dv, float* df, float* dW,
                   float* dw_r, int64_t B, int64_t T, int64_t N, int64_t K, int64_t V,
                   m2rnn_dtype dtype, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return m2rnn_backward_state(q, k, v, f, W, w_r, nullptr, dy, dH_T, ckpt, ckpt_every, nullptr, dq, dk, dv,
                              df, dW, dw_r, nullptr, 0.f, B, T, N, N, K, V, dtype, workspace,
                              workspace_bytes, cuda_stream);
}

int m2rnn_sync_status(void* workspace, void* cuda_stream, uint32_t* detail) {
  if (workspace == nullptr || !aligned16(workspace)) return M2RNN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  StatusBlock host{};
  if (cudaMemcpyAsync(&host, workspace, 8, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return M2RNN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, 8, s) != cudaSuccess) return M2RNN_ERR_CUDA;
  if (detail) *detail = host.detail;
  if (host.code == 0) return M2RNN_OK;
  return host.code == kStatusTimeout ? M2RNN_ERR_TIMEOUT : M2RNN_ERR_DEVICE;
}

}  // extern "C"
