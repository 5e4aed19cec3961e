// fp32 CUDA-core kernels for the M2RNN scans: any K, V in [1, 128], fp32 or
// bf16 inputs, fp32 arithmetic throughout (tanhf, fmaf).  One CTA per
// (batch, head) chain.  They serve the all-fp32 workloads and every shape the
// tensor-core kernels do not take.
//
// Forward: Eq. 10-12 of "M2RNN: Non-Linear RNNs with Matrix-Valued States for
// Scalable Language Modeling" (reading notes section 2.1).  Backward: the
// chain-rule recursion of the notes' section 2.7, with per-chunk recompute
// from stored states (section 2.6 describes the paper's recompute-and-cache
// scheme; here only one chunk of states is cached at a time).
#include <cuda_runtime.h>

#include "gate.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace m2rnn {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_in(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p, int64_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float ld_in<uint16_t>(const uint16_t* p, int64_t i) {
  return bf16_bits_to_f32(p[i]);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) simt_forward_kernel(FwdArgs a) {
  extern __shared__ float sm[];
  const int K = a.K, V = a.V, T = a.T, N = a.N;
  const int KV = K * V;
  const int chain = blockIdx.x;
  const int b = chain / N, n = chain % N;
  float* Ws = sm;          // [V][V]
  float* Ha = Ws + V * V;  // [K][V]
  float* Hb = Ha + KV;     // [K][V]
  float* ks = Hb + KV;     // [K]
  float* qs = ks + K;      // [K]
  float* vs = qs + K;      // [V]
  float* fs = vs + V;      // [1]
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  const GateSrc gs{a.f, a.gate_a, a.gate_alpha, a.gate_beta, sizeof(Tin) == 2};
  const Tin* W = static_cast<const Tin*>(a.W) + static_cast<int64_t>(n) * V * V;
  const Tin* w_r = static_cast<const Tin*>(a.w_r) + static_cast<int64_t>(n) * V;

  for (int e = threadIdx.x; e < V * V; e += kThreads) Ws[e] = ld_in(W, e);
  for (int e = threadIdx.x; e < KV; e += kThreads) Ha[e] = a.H0 ? a.H0[static_cast<int64_t>(chain) * KV + e] : 0.f;
  __syncthreads();
  float* Hc = Ha;
  float* Hn = Hb;
  for (int t = 0; t < T; ++t) {
    const int64_t row = (static_cast<int64_t>(b) * T + t) * N + n;
    const int64_t rowqk = (static_cast<int64_t>(b) * T + t) * qk_heads(a.qkN, N) + qk_head(a.qkN, n);
    for (int i = threadIdx.x; i < K; i += kThreads) {
      ks[i] = ld_in(k, rowqk * K + i);
      qs[i] = ld_in(q, rowqk * K + i);
    }
    for (int j = threadIdx.x; j < V; j += kThreads) vs[j] = ld_in(v, row * V + j);
    if (threadIdx.x == 0) fs[0] = gate_value(gs, row, n);
    __syncthreads();
    const float ft = fs[0];
    for (int e = threadIdx.x; e < KV; e += kThreads) {
      const int i = e / V, j = e % V;
      float acc = 0.f;
      for (int m = 0; m < V; ++m) acc = fmaf(Hc[i * V + m], Ws[m * V + j], acc);  // (H W)_ij
      acc = fmaf(ks[i], vs[j], acc);                                                  // + k_i v_j
      const float z = tanhf(acc);                                                     // Eq. 10
      Hn[e] = ft * Hc[e] + (1.f - ft) * z;                                            // Eq. 11
    }
    __syncthreads();
    if (a.y != nullptr) {
      for (int j = threadIdx.x; j < V; j += kThreads) {
        float s = 0.f;
        for (int i = 0; i < K; ++i) s = fmaf(qs[i], Hn[i * V + j], s);
        a.y[row * V + j] = s + ld_in(w_r, j) * vs[j];  // Eq. 12
      }
    }
    if (a.ckpt != nullptr && (t + 1) % a.ckpt_every == 0 && t + 1 < T) {
      float* dst = a.ckpt + (static_cast<int64_t>(chain) * a.n_ckpt + (t + 1) / a.ckpt_every - 1) * KV;
      for (int e = threadIdx.x; e < KV; e += kThreads) dst[e] = Hn[e];
    }
    float* tmp = Hc;
    Hc = Hn;
    Hn = tmp;
    __syncthreads();
  }
  if (a.H_T != nullptr) {
    for (int e = threadIdx.x; e < KV; e += kThreads) a.H_T[static_cast<int64_t>(chain) * KV + e] = Hc[e];
  }
}

__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = x;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];  // fixed order
  }
  return s;  // valid in thread 0 only
}

// Backward: per chain, chunks in reverse; each chunk is recomputed from its
// starting state (zero for chunk 0, else the stored checkpoint) into the
// chain's scratch (states H_{s0..s0+L} and candidates Z), then walked in
// reverse with the recursion R -> D -> C_{t-1}.
template <typename Tin>
__global__ void __launch_bounds__(kThreads) simt_backward_kernel(BwdArgs a) {
  extern __shared__ float sm[];
  const int K = a.K, V = a.V, T = a.T, N = a.N, CL = a.ckpt_every;
  const int KV = K * V;
  const int chain = blockIdx.x;
  const int b = chain / N, n = chain % N;
  float* Ws = sm;          // [V][V]
  float* Cm = Ws + V * V;  // [K][V] state gradient C (then R)
  float* Dm = Cm + KV;     // [K][V] D (recompute: current H)
  float* ks = Dm + KV;     // [K]
  float* qs = ks + K;      // [K]
  float* vs = qs + K;      // [V]
  float* us = vs + V;      // [V]
  float* red = us + V;     // [32]
  float* fs = red + 32;    // [1]
  const Tin* q = static_cast<const Tin*>(a.q);
  const Tin* k = static_cast<const Tin*>(a.k);
  const Tin* v = static_cast<const Tin*>(a.v);
  const GateSrc gs{a.f, a.gate_a, a.gate_alpha, a.gate_beta, sizeof(Tin) == 2};
  const Tin* W = static_cast<const Tin*>(a.W) + static_cast<int64_t>(n) * V * V;
  const Tin* w_r = static_cast<const Tin*>(a.w_r) + static_cast<int64_t>(n) * V;
  float* Hs = a.scratch + static_cast<int64_t>(chain) * (2 * CL + 1) * KV;  // [CL+1][K][V]
  float* Zs = Hs + static_cast<int64_t>(CL + 1) * KV;                       // [CL][K][V]
  float* dWp = a.dW_part + static_cast<int64_t>(chain) * V * V;
  float* dwrp = a.dwr_part + static_cast<int64_t>(chain) * V;

  for (int e = threadIdx.x; e < V * V; e += kThreads) {
    Ws[e] = ld_in(W, e);
    dWp[e] = 0.f;
  }
  for (int j = threadIdx.x; j < V; j += kThreads) dwrp[j] = 0.f;
  for (int e = threadIdx.x; e < KV; e += kThreads)
    Cm[e] = a.dH_T ? a.dH_T[static_cast<int64_t>(chain) * KV + e] : 0.f;
  __syncthreads();

  const int nchunks = (T + CL - 1) / CL;
  for (int c = nchunks - 1; c >= 0; --c) {
    const int s0 = c * CL;
    const int L = min(CL, T - s0);
    // ---- recompute the chunk's states ----
    const float* Hstart = (c == 0) ? (a.H0 ? a.H0 + static_cast<int64_t>(chain) * KV : nullptr)
                                   : a.ckpt + (static_cast<int64_t>(chain) * a.n_ckpt + (c - 1)) * KV;
    for (int e = threadIdx.x; e < KV; e += kThreads) {
      const float h = Hstart ? Hstart[e] : 0.f;
      Dm[e] = h;
      Hs[e] = h;
    }
    __syncthreads();
    for (int s = 0; s < L; ++s) {
      const int64_t row = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
      const int64_t rowqk = (static_cast<int64_t>(b) * T + s0 + s) * qk_heads(a.qkN, N) + qk_head(a.qkN, n);
      for (int i = threadIdx.x; i < K; i += kThreads) ks[i] = ld_in(k, rowqk * K + i);
      for (int j = threadIdx.x; j < V; j += kThreads) vs[j] = ld_in(v, row * V + j);
      if (threadIdx.x == 0) fs[0] = gate_value(gs, row, n);
      __syncthreads();
      const float ft = fs[0];
      for (int e = threadIdx.x; e < KV; e += kThreads) {
        const int i = e / V, j = e % V;
        float acc = 0.f;
        for (int m = 0; m < V; ++m) acc = fmaf(Dm[i * V + m], Ws[m * V + j], acc);
        acc = fmaf(ks[i], vs[j], acc);
        const float z = tanhf(acc);
        Zs[static_cast<int64_t>(s) * KV + e] = z;
        Hs[static_cast<int64_t>(s + 1) * KV + e] = ft * Dm[e] + (1.f - ft) * z;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < KV; e += kThreads) Dm[e] = Hs[static_cast<int64_t>(s + 1) * KV + e];
      __syncthreads();
    }
    // ---- reverse walk over the chunk ----
    for (int s = L - 1; s >= 0; --s) {
      const int64_t row = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
      const int64_t rowqk = (static_cast<int64_t>(b) * T + s0 + s) * qk_heads(a.qkN, N) + qk_head(a.qkN, n);
      for (int i = threadIdx.x; i < K; i += kThreads) {
        ks[i] = ld_in(k, rowqk * K + i);
        qs[i] = ld_in(q, rowqk * K + i);
      }
      for (int j = threadIdx.x; j < V; j += kThreads) {
        vs[j] = ld_in(v, row * V + j);
        us[j] = a.dy[row * V + j];
      }
      if (threadIdx.x == 0) fs[0] = gate_value(gs, row, n);
      __syncthreads();
      const float ft = fs[0];
      const float* Hprev = Hs + static_cast<int64_t>(s) * KV;
      const float* Hcur = Hs + static_cast<int64_t>(s + 1) * KV;
      const float* Z = Zs + static_cast<int64_t>(s) * KV;
      float dfp = 0.f;
      for (int e = threadIdx.x; e < KV; e += kThreads) {
        const int i = e / V, j = e % V;
        const float R = fmaf(qs[i], us[j], Cm[e]);        // R = C + q u^T
        const float z = Z[e];
        Dm[e] = (1.f - ft) * R * (1.f - z * z);            // D
        Cm[e] = R;
        dfp = fmaf(R, Hprev[e] - z, dfp);                  // <R, H_{t-1} - Z>
      }
      __syncthreads();
      const float dfs = block_sum(dfp, red);
      if (threadIdx.x == 0) a.df[row] = dfs;
      for (int i = threadIdx.x; i < K; i += kThreads) {
        float sq = 0.f, sk = 0.f;
        for (int j = 0; j < V; ++j) {
          sq = fmaf(Hcur[i * V + j], us[j], sq);  // dq = H_t u
          sk = fmaf(Dm[i * V + j], vs[j], sk);    // dk = D v
        }
        a.dq[row * K + i] = sq;
        a.dk[row * K + i] = sk;
      }
      for (int j = threadIdx.x; j < V; j += kThreads) {
        float sv = 0.f;
        for (int i = 0; i < K; ++i) sv = fmaf(Dm[i * V + j], ks[i], sv);  // D^T k
        a.dv[row * V + j] = sv + ld_in(w_r, j) * us[j];
        dwrp[j] += us[j] * vs[j];
      }
      for (int e = threadIdx.x; e < V * V; e += kThreads) {
        const int m = e / V, j = e % V;
        float s2 = 0.f;
        for (int i = 0; i < K; ++i) s2 = fmaf(Hprev[i * V + m], Dm[i * V + j], s2);  // H^T D
        dWp[e] += s2;
      }
      for (int e = threadIdx.x; e < KV; e += kThreads) {
        const int i = e / V, m = e % V;
        float s3 = 0.f;
        for (int j = 0; j < V; ++j) s3 = fmaf(Dm[i * V + j], Ws[m * V + j], s3);  // D W^T
        const float cn = ft * Cm[e] + s3;
        Cm[e] = (a.clip > 0.f) ? fminf(fmaxf(cn, -a.clip), a.clip) : cn;  // per-step clipping
      }
      __syncthreads();
    }
  }
  if (a.dH0 != nullptr)  // C_0, the state gradient left after step 1
    for (int e = threadIdx.x; e < KV; e += kThreads) a.dH0[static_cast<int64_t>(chain) * KV + e] = Cm[e];
}

// dW[n] = sum_b sum_p part[b][n][p], dw_r[n] = sum_b wpart[b][n], fixed order.
__global__ void reduce_partials_kernel(const float* __restrict__ dWp, const float* __restrict__ dwrp,
                                       float* __restrict__ dW, float* __restrict__ dw_r, int B,
                                       int N, int P, int V) {
  const int64_t VV = static_cast<int64_t>(V) * V;
  const int64_t total = static_cast<int64_t>(N) * VV;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = e / VV, x = e % VV;
    float s = 0.f;
    for (int b = 0; b < B; ++b)
      for (int p = 0; p < P; ++p) s += dWp[((static_cast<int64_t>(b) * N + n) * P + p) * VV + x];
    dW[e] = s;
  }
  const int64_t total2 = static_cast<int64_t>(N) * V;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total2;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = e / V, j = e % V;
    float s = 0.f;
    for (int b = 0; b < B; ++b) s += dwrp[(static_cast<int64_t>(b) * N + n) * V + j];
    dw_r[e] = s;
  }
}

size_t fwd_smem_bytes(int K, int V) { return sizeof(float) * (V * V + 2 * K * V + 2 * K + V + 4); }
size_t bwd_smem_bytes(int K, int V) {
  return sizeof(float) * (V * V + 2 * K * V + 2 * K + 2 * V + 32 + 4);
}

template <typename Tin>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  const size_t smem = fwd_smem_bytes(a.K, a.V);
  cudaError_t e = cudaFuncSetAttribute(simt_forward_kernel<Tin>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  simt_forward_kernel<Tin><<<a.B * a.N, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = bwd_smem_bytes(a.K, a.V);
  cudaError_t e = cudaFuncSetAttribute(simt_backward_kernel<Tin>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  simt_backward_kernel<Tin><<<a.B * a.N, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_forward(const FwdArgs& a, cudaStream_t s) {
  return a.dtype == M2RNN_F32 ? launch_fwd_t<float>(a, s) : launch_fwd_t<uint16_t>(a, s);
}

cudaError_t launch_simt_backward(const BwdArgs& a, cudaStream_t s) {
  return a.dtype == M2RNN_F32 ? launch_bwd_t<float>(a, s) : launch_bwd_t<uint16_t>(a, s);
}

size_t simt_backward_scratch_bytes(int B, int N, int K, int V, int ckpt_every) {
  return sizeof(float) * static_cast<size_t>(B) * N * (2 * static_cast<size_t>(ckpt_every) + 1) * K * V;
}

cudaError_t launch_reduce_partials(const BwdArgs& a, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(a.N) * a.V * a.V;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
  reduce_partials_kernel<<<blocks, 256, 0, s>>>(a.dW_part, a.dwr_part, a.dW, a.dw_r, a.B, a.N,
                                                a.parts, a.V);
  return cudaGetLastError();
}

}  // namespace m2rnn

namespace m2rnn {
namespace {
__global__ void sum_qk_heads_kernel(const float* __restrict__ dqh, const float* __restrict__ dkh,
                                    float* __restrict__ dq, float* __restrict__ dk, int64_t BT, int N, int K) {
  const int64_t total = BT * K;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t bt = e / K, i = e % K;
    float sq = 0.f, sk = 0.f;
    for (int n = 0; n < N; ++n) {  // fixed order over the heads
      sq += dqh[(bt * N + n) * K + i];
      sk += dkh[(bt * N + n) * K + i];
    }
    dq[e] = sq;
    dk[e] = sk;
  }
}
}  // namespace

cudaError_t launch_sum_qk_heads(const float* dq_heads, const float* dk_heads, float* dq, float* dk,
                                int64_t BT, int N, int K, cudaStream_t stream) {
  const int64_t total = BT * K;
  const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 152 * 16));
  sum_qk_heads_kernel<<<blocks, 256, 0, stream>>>(dq_heads, dk_heads, dq, dk, BT, N, K);
  return cudaGetLastError();
}
}  // namespace m2rnn
