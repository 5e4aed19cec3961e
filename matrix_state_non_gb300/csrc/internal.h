// Internal launcher interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/m2rnn.h"
#include "status.cuh"

namespace m2rnn {

// Everything a forward launch needs, already validated by the C-ABI layer.
struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* f;
  const void* W;
  const void* w_r;
  const float* H0;  // initial state [B,N,K,V] fp32; null = zero
  int qkN;          // heads of q and k: 1 = one q/k shared by every head, else N
  const void* gate_a;        // non-null: f = exp(-alpha softplus(a + beta)) from a [B,T,N] (input dtype)
  const float* gate_alpha;   // [N]
  const float* gate_beta;    // [N]
  uint16_t* zstash;  // V = 64 warp-MMA forward: fp16 Z_t of every step for the backward, or null
  float* y;      // may be null (checkpoint-only pass)
  float* H_T;    // may be null
  float* ckpt;   // may be null
  int ckpt_every;
  int64_t n_ckpt;
  int B, T, N, K, V;
  m2rnn_dtype dtype;
  StatusBlock* status;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* f;
  const void* W;
  const void* w_r;
  const float* dy;
  const float* dH_T;  // may be null
  const float* H0;    // initial state; null = zero
  float* dH0;         // gradient of the initial state; may be null
  int qkN;            // heads of q and k (1 = shared); dq/dk are per head here either way
  const void* gate_a;        // as in FwdArgs
  const float* gate_alpha;
  const float* gate_beta;
  float clip;         // > 0: every new C_{t-1} clamped to [-clip, clip]; else no clipping
  const float* ckpt;  // never null here (recomputed by the caller layer if needed)
  const uint16_t* zstash;  // the forward's Z stash (V = 64 warp-MMA backward), or null: rerun the forward
  int ckpt_every;
  int64_t n_ckpt;
  float* dq;
  float* dk;
  float* dv;
  float* df;
  float* dW;
  float* dw_r;
  int B, T, N, K, V;
  m2rnn_dtype dtype;
  StatusBlock* status;
  // Scratch carved from the workspace by the C-ABI layer.
  float* dW_part;    // [B*N*parts][V][V]
  float* dwr_part;   // [B*N][V]
  float* scratch;    // kernel-specific (SIMT: per-chain chunk states)
  int parts;         // dW partials per chain
};

// Process-wide switches (m2rnn_set_option), first read from the environment
// variables M2RNN_KERNEL and M2RNN_TEST_STALL_TILE once.  Kernel family: -1
// automatic, 0 fp32 CUDA cores, 1 tcgen05, 2 warp MMA.  Stall tile: -1 off.
int option_kernel_family();
int option_test_stall_tile();
int set_option(int option, int value, int* previous);

// fp32 CUDA-core kernels (any K, V in [1, 128]).
cudaError_t launch_simt_forward(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_simt_backward(const BwdArgs& a, cudaStream_t s);
size_t simt_backward_scratch_bytes(int B, int N, int K, int V, int ckpt_every);

// Fixed-order sum of per-chain partials over b (and parts): dW, dw_r.
cudaError_t launch_reduce_partials(const BwdArgs& a, cudaStream_t s);

// Register-resident warp-MMA kernels (bf16 inputs, V = 64).
bool mma_forward_supported(int K, int V);
cudaError_t launch_mma_forward(const FwdArgs& a, cudaStream_t s);
// Head of q/k that head n reads: 0 when one q/k is shared by every head.
__host__ __device__ inline int qk_head(int qkN, int n) { return qkN == 1 ? 0 : n; }
__host__ __device__ inline int qk_heads(int qkN, int N) { return qkN == 1 ? 1 : N; }

// One decoding step (bf16, V = 64, K % 16 == 0, K <= 128), state in place.
bool decode_kernel_supported(int K, int V, m2rnn_dtype dtype);
cudaError_t launch_decode_step(float* H, const void* q, const void* k, const void* v, const void* f,
                               const void* W, const void* w_r, float* y, int B, int N, int K, int qkN,
                               StatusBlock* status, cudaStream_t stream);
// dq[b,t,0,:] = sum over heads n of dq_heads[b,t,n,:] (fixed order), same for dk.
cudaError_t launch_sum_qk_heads(const float* dq_heads, const float* dk_heads, float* dq, float* dk,
                                int64_t BT, int N, int K, cudaStream_t stream);

// Register-resident forward for V = 16 (one warp per 16 key rows, no exchange).
bool mv_forward_supported(int K, int V);
// The pipelined V = 16 forward (compute and readout warps per row block), for
// K <= 64 with the readout y requested; launch_mv_forward runs it there.
bool mv_forward_pipe_supported(int K, int V, bool readout);
cudaError_t launch_mv_forward_pipe(const FwdArgs& a, cudaStream_t s);
cudaError_t launch_mv_forward(const FwdArgs& a, cudaStream_t s);

// Register-resident backward for V = 16 (chunks of up to 32 steps, 16 with K > 64).
bool mv_backward_supported(int K, int V, int ckpt_every);
cudaError_t launch_mv_backward(const BwdArgs& a, cudaStream_t s);
// The pipelined V = 16 backward (rebuild and chain warps per row block);
// launch_mv_backward runs it where it applies (chunks of up to 20 steps for
// K <= 64, 10 for K <= 128).
bool mv_backward_pipe_supported(int K, int V, int ckpt_every);
cudaError_t launch_mv_backward_pipe(const BwdArgs& a, cudaStream_t s);

bool mma_backward_supported(int K, int V);
size_t mma_backward_scratch_bytes(int B, int T, int N, int K, int V, int ckpt_every);
int mma_backward_max_chunk();
cudaError_t launch_mma_backward(const BwdArgs& a, cudaStream_t s);

// tcgen05 tensor-core kernels (bf16 inputs).
bool tc_forward_supported(int K, int V);
cudaError_t launch_tc_forward(const FwdArgs& a, cudaStream_t s);
bool tc_backward_supported(int K, int V);
int tc_backward_parts(int K, int V);
size_t tc_backward_scratch_bytes(int B, int N, int K, int V, int ckpt_every);
cudaError_t launch_tc_backward(const BwdArgs& a, cudaStream_t s);
// K = V = 128 with chunks of at most 16 steps: every product on tcgen05
// (launch_tc_backward routes there).
bool tc_backward128_supported(int K, int V, int ckpt_every);
size_t tc_backward128_scratch_bytes(int B, int N, int ckpt_every);
cudaError_t launch_tc_backward128(const BwdArgs& a, cudaStream_t s);

// Gate backward: grad holds df on entry, da on exit; part holds
// 2 * N * gate_backward_parts(BT) floats of scratch.
struct GateSrc;
int gate_backward_parts(int64_t BT);
cudaError_t launch_gate_backward(const GateSrc& gs, float* grad, float* dalpha, float* dbeta, float* part,
                                 int64_t BT, int N, cudaStream_t s);
// Gated RMSNorm output path over rows of d elements.
int output_norm_max_width();
int output_norm_backward_parts(int64_t rows, int d);
cudaError_t launch_output_norm(const float* y, const void* g, const float* w, float eps, float* out, float* rstd,
                               int64_t rows, int d, bool bf16, cudaStream_t s);
cudaError_t launch_output_norm_backward(const float* y, const void* g, const float* w, const float* dout, float eps,
                                        float* dy, float* dg, float* dw, float* part, int64_t rows, int d,
                                        bool bf16, cudaStream_t s);

}  // namespace m2rnn
