// The two state-free pieces around the scan ("M2RNN: Non-Linear RNNs with
// Matrix-Valued States for Scalable Language Modeling", sections 2.2 and 2.3
// of the reading notes, Appendix C):
//
//  * gate backward: with x = a + beta[n], s = softplus(x), f = exp(-alpha s),
//      da = df f (-alpha) sigmoid(x),  dalpha[n] = sum_{b,t} df f (-s),
//      dbeta[n] = sum_{b,t} da;
//    the forward gate itself runs inside the scan kernels (gate.cuh).
//  * output path: x = y * g, rms-normalised over the full token width
//    d = N V (the statistic spans every head), times a per-channel weight:
//      s = (sum x^2 / d + eps)^(-1/2),  out = w x s;
//    backward with p = w dout and r = sum p x:
//      dx = s p - r s^3 x / d,  dy = dx g,  dg = dx y,  dw = sum_{b,t} dout x s.
//
// All of it is HBM-bound elementwise work plus per-row and per-column sums.
// Every sum runs in a fixed order that depends only on the shape, so results
// are bitwise reproducible.
#include <cuda_runtime.h>

#include <cstdint>

#include "gate.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace m2rnn {
namespace {

constexpr int kGateThreads = 256;

// Fixed-order block sum of two values; every thread gets the totals.
template <int kThreads>
__device__ __forceinline__ float2 block_sum2(float a, float b, float2* red) {
  static_assert(kThreads % 32 == 0 && kThreads <= 1024, "block size");
  constexpr int kWarps = kThreads / 32;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = make_float2(a, b);
  __syncthreads();
  float2 t = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) {
    t.x += red[i].x;
    t.y += red[i].y;
  }
  __syncthreads();  // red may be reused right after
  return t;
}

// Grid (P, N): block (p, n) takes rows i = p * 256 + tid, stepping P * 256,
// of head n; grad holds df on entry and da on exit.  Block partials of
// dalpha, dbeta go to part[n][p]; gate_finish_kernel sums them in order.
__global__ void __launch_bounds__(kGateThreads) gate_backward_kernel(GateSrc gs, float* grad, float2* part,
                                                                     int64_t BT, int N) {
  __shared__ float2 red[kGateThreads / 32];
  const int n = blockIdx.y, P = gridDim.x;
  const float al = gs.alpha[n], be = gs.beta[n];
  float sa = 0.f, sb = 0.f;
#pragma unroll 4
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kGateThreads + threadIdx.x; i < BT;
       i += static_cast<int64_t>(P) * kGateThreads) {
    const int64_t idx = i * N + n;
    const float x = (gs.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(gs.a)[idx])
                             : static_cast<const float*>(gs.a)[idx]) + be;
    const float s = softplus_f(x);
    const float f = gate_value(gs, idx, n);  // the forward's own f, bit for bit
    const float sig = 1.f / (1.f + expf(-x));
    const float g = grad[idx] * f;
    const float d = -al * g * sig;
    grad[idx] = d;
    sa -= g * s;
    sb += d;
  }
  const float2 t = block_sum2<kGateThreads>(sa, sb, red);
  if (threadIdx.x == 0) part[static_cast<int64_t>(n) * P + blockIdx.x] = t;
}

__global__ void gate_finish_kernel(const float2* part, float* dalpha, float* dbeta, int P, int N) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float2 t = part[static_cast<int64_t>(n) * P];
  for (int p = 1; p < P; ++p) {
    const float2 u = part[static_cast<int64_t>(n) * P + p];
    t.x += u.x;
    t.y += u.y;
  }
  dalpha[n] = t.x;
  dbeta[n] = t.y;
}

// ---------------------------------------------------------------------------
// Output path.  One row = one token (b, t) of d = N V elements, held in
// registers as groups of 4 consecutive elements: thread i owns groups
// i, i + kThreads, ... (kPer of them).
// ---------------------------------------------------------------------------

struct NormArgs {
  const float* y;   // [rows][d]
  const void* g;    // [rows][d], input dtype
  const float* w;   // [d]
  const float* dout;  // backward only
  float* out;       // forward: [rows][d]
  float* rstd;      // forward: [rows] or null
  float* dy;        // backward: [rows][d]
  float* dg;        // backward: [rows][d]
  float* dw_part;   // backward: [gridDim.x][d]
  int64_t rows;
  int d;
  float eps;
  bool bf16;
  bool vec;  // d % 4 == 0: 16-byte loads
};

__device__ __forceinline__ float4 ld4_f32(const float* p, int64_t base, int j, int d, bool vec) {
  if (vec) return *reinterpret_cast<const float4*>(p + base + j);
  float4 r;
  r.x = j < d ? p[base + j] : 0.f;
  r.y = j + 1 < d ? p[base + j + 1] : 0.f;
  r.z = j + 2 < d ? p[base + j + 2] : 0.f;
  r.w = j + 3 < d ? p[base + j + 3] : 0.f;
  return r;
}

__device__ __forceinline__ float4 ld4_in(const NormArgs& A, const void* p, int64_t base, int j) {
  if (!A.bf16) return ld4_f32(static_cast<const float*>(p), base, j, A.d, A.vec);
  const uint16_t* h = static_cast<const uint16_t*>(p) + base;
  if (A.vec) {
    const uint2 u = *reinterpret_cast<const uint2*>(h + j);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  }
  float4 r;
  r.x = j < A.d ? bf16_bits_to_f32(h[j]) : 0.f;
  r.y = j + 1 < A.d ? bf16_bits_to_f32(h[j + 1]) : 0.f;
  r.z = j + 2 < A.d ? bf16_bits_to_f32(h[j + 2]) : 0.f;
  r.w = j + 3 < A.d ? bf16_bits_to_f32(h[j + 3]) : 0.f;
  return r;
}

__device__ __forceinline__ void st4(float* p, int64_t base, int j, int d, bool vec, float4 v) {
  if (vec) {
    *reinterpret_cast<float4*>(p + base + j) = v;
    return;
  }
  if (j < d) p[base + j] = v.x;
  if (j + 1 < d) p[base + j + 1] = v.y;
  if (j + 2 < d) p[base + j + 2] = v.z;
  if (j + 3 < d) p[base + j + 3] = v.w;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

template <int kThreads, int kPer>
__global__ void __launch_bounds__(kThreads) output_norm_kernel(NormArgs A) {
  __shared__ float2 red[kThreads / 32];
  const int d = A.d;
  float4 wv[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 4 * (threadIdx.x + i * kThreads);
    wv[i] = j < d ? ld4_f32(A.w, 0, j, d, A.vec) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t row = blockIdx.x; row < A.rows; row += gridDim.x) {
    const int64_t base = row * d;
    float4 x[kPer];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (threadIdx.x + i * kThreads);
      if (j < d) {
        x[i] = mul4(ld4_f32(A.y, base, j, d, A.vec), ld4_in(A, A.g, base, j));
      } else {
        x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      ss += dot4(x[i], x[i]);
    }
    const float tot = block_sum2<kThreads>(ss, 0.f, red).x;
    const float s = rsqrtf(tot / static_cast<float>(d) + A.eps);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (threadIdx.x + i * kThreads);
      if (j < d) {
        const float4 o = mul4(wv[i], x[i]);
        st4(A.out, base, j, d, A.vec, make_float4(o.x * s, o.y * s, o.z * s, o.w * s));
      }
    }
    if (A.rstd != nullptr && threadIdx.x == 0) A.rstd[row] = s;
  }
}

// Pass 1 keeps y and g in registers; pass 2 reads w and dout again (from L1
// or L2: the block has just read them), which keeps the widest rows
// (d = 16384 at 512 threads) free of spills.
template <int kThreads, int kPer>
__global__ void __launch_bounds__(kThreads) output_norm_backward_kernel(NormArgs A) {
  __shared__ float2 red[kThreads / 32];
  const int d = A.d;
  const float inv_d = 1.f / static_cast<float>(d);
  float4 dwa[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) dwa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t row = blockIdx.x; row < A.rows; row += gridDim.x) {
    const int64_t base = row * d;
    float4 yv[kPer], gv[kPer];
    float ss = 0.f, rr = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (threadIdx.x + i * kThreads);
      float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < d) {
        yv[i] = ld4_f32(A.y, base, j, d, A.vec);
        gv[i] = ld4_in(A, A.g, base, j);
        p = mul4(ld4_f32(A.w, 0, j, d, A.vec), ld4_f32(A.dout, base, j, d, A.vec));
      } else {
        yv[i] = gv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const float4 x = mul4(yv[i], gv[i]);
      ss += dot4(x, x);
      rr += dot4(p, x);
    }
    const float2 t = block_sum2<kThreads>(ss, rr, red);
    const float s = rsqrtf(t.x * inv_d + A.eps);
    const float c = t.y * s * s * s * inv_d;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (threadIdx.x + i * kThreads);
      if (j < d) {
        const float4 x = mul4(yv[i], gv[i]);
        const float4 o = ld4_f32(A.dout, base, j, d, A.vec);
        const float4 p = mul4(ld4_f32(A.w, 0, j, d, A.vec), o);
        const float4 dx = make_float4(s * p.x - c * x.x, s * p.y - c * x.y, s * p.z - c * x.z, s * p.w - c * x.w);
        st4(A.dy, base, j, d, A.vec, mul4(dx, gv[i]));
        st4(A.dg, base, j, d, A.vec, mul4(dx, yv[i]));
        dwa[i].x += o.x * x.x * s;
        dwa[i].y += o.y * x.y * s;
        dwa[i].z += o.z * x.z * s;
        dwa[i].w += o.w * x.w * s;
      }
    }
  }
  float* part = A.dw_part + static_cast<int64_t>(blockIdx.x) * d;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 4 * (threadIdx.x + i * kThreads);
    if (j < d) st4(part, 0, j, d, A.vec, dwa[i]);
  }
}

// Rows of up to 1024 elements: one warp per row, lane l owning groups
// l, l + 32, ... (kPer of them), eight warps per block; only shuffles in the
// row sums.  Warp w takes rows w, w + (total warps), ...
constexpr int kRowWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int kPer>
__global__ void __launch_bounds__(32 * kRowWarps) norm_rows_kernel(NormArgs A) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int d = A.d;
  float4 wv[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 4 * (lane + 32 * i);
    wv[i] = j < d ? ld4_f32(A.w, 0, j, d, A.vec) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); row < A.rows;
       row += nw) {
    const int64_t base = row * d;
    float4 x[kPer];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (lane + 32 * i);
      x[i] = j < d ? mul4(ld4_f32(A.y, base, j, d, A.vec), ld4_in(A, A.g, base, j))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      ss += dot4(x[i], x[i]);
    }
    const float s = rsqrtf(warp_sum(ss) / static_cast<float>(d) + A.eps);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (lane + 32 * i);
      if (j < d) {
        const float4 o = mul4(wv[i], x[i]);
        st4(A.out, base, j, d, A.vec, make_float4(o.x * s, o.y * s, o.z * s, o.w * s));
      }
    }
    if (A.rstd != nullptr && lane == 0) A.rstd[row] = s;
  }
}

// dw: each lane accumulates its columns over the warp's rows; the block's
// eight warps are summed in warp order through shared memory, one partial
// row per block.
template <int kPer>
__global__ void __launch_bounds__(32 * kRowWarps) norm_rows_backward_kernel(NormArgs A) {
  __shared__ float dws[kRowWarps][128 * kPer];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int d = A.d;
  const float inv_d = 1.f / static_cast<float>(d);
  float4 wv[kPer], dwa[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 4 * (lane + 32 * i);
    wv[i] = j < d ? ld4_f32(A.w, 0, j, d, A.vec) : make_float4(0.f, 0.f, 0.f, 0.f);
    dwa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + wib; row < A.rows; row += nw) {
    const int64_t base = row * d;
    float4 yv[kPer], gv[kPer], ov[kPer];
    float ss = 0.f, rr = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (lane + 32 * i);
      if (j < d) {
        yv[i] = ld4_f32(A.y, base, j, d, A.vec);
        gv[i] = ld4_in(A, A.g, base, j);
        ov[i] = ld4_f32(A.dout, base, j, d, A.vec);
      } else {
        yv[i] = gv[i] = ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const float4 x = mul4(yv[i], gv[i]);
      ss += dot4(x, x);
      rr += dot4(mul4(wv[i], ov[i]), x);
    }
    ss = warp_sum(ss);
    rr = warp_sum(rr);
    const float s = rsqrtf(ss * inv_d + A.eps);
    const float c = rr * s * s * s * inv_d;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = 4 * (lane + 32 * i);
      if (j < d) {
        const float4 x = mul4(yv[i], gv[i]);
        const float4 p = mul4(wv[i], ov[i]);
        const float4 dx = make_float4(s * p.x - c * x.x, s * p.y - c * x.y, s * p.z - c * x.z, s * p.w - c * x.w);
        st4(A.dy, base, j, d, A.vec, mul4(dx, gv[i]));
        st4(A.dg, base, j, d, A.vec, mul4(dx, yv[i]));
        dwa[i].x += ov[i].x * x.x * s;
        dwa[i].y += ov[i].y * x.y * s;
        dwa[i].z += ov[i].z * x.z * s;
        dwa[i].w += ov[i].w * x.w * s;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 4 * (lane + 32 * i);
    *reinterpret_cast<float4*>(&dws[wib][j]) = dwa[i];
  }
  __syncthreads();
  float* part = A.dw_part + static_cast<int64_t>(blockIdx.x) * d;
  for (int j = threadIdx.x; j < d; j += 32 * kRowWarps) {
    float t = dws[0][j];
#pragma unroll
    for (int w = 1; w < kRowWarps; ++w) t += dws[w][j];
    part[j] = t;
  }
}

// dw[j] = sum over the P block partials part[p][j]: block b takes columns
// 32 b .. 32 b + 31 (one per lane); its 32 warps each sum a contiguous
// 32nd of p in order, then the 32 are added in warp order.
constexpr int kSumWarps = 32;

__global__ void __launch_bounds__(32 * kSumWarps) sum_columns_kernel(const float* part, float* out, int P, int d) {
  __shared__ float red[kSumWarps][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + lane;
  const int per = (P + kSumWarps - 1) / kSumWarps, p0 = w * per, p1 = min(P, p0 + per);
  float acc = 0.f;
  if (j < d) {
#pragma unroll 4
    for (int p = p0; p < p1; ++p) acc += part[static_cast<int64_t>(p) * d + j];
  }
  red[w][lane] = acc;
  __syncthreads();
  if (w == 0 && j < d) {
    float t = red[0][lane];
#pragma unroll
    for (int i = 1; i < kSumWarps; ++i) t += red[i][lane];
    out[j] = t;
  }
}

// Launch shape for a row width d: threads per block and register groups per
// thread; d <= 16384 (N V with V <= 128 and N <= 128) always fits.
struct NormShape {
  int threads, per;
};

// threads == 0: one warp per row (norm_rows_*), per = groups per lane.
NormShape norm_shape(int d) {
  const int groups = (d + 3) / 4;
  if (groups <= 32) return {0, 1};
  if (groups <= 64) return {0, 2};
  if (groups <= 128) return {0, 4};
  if (groups <= 256) return {0, 8};
  if (groups <= 512) return {256, 2};
  if (groups <= 1024) return {256, 4};
  if (groups <= 2048) return {256, 8};
  return {512, 8};
}

cudaError_t launch_norm(bool backward, const NormArgs& A, int grid, cudaStream_t s) {
  const NormShape sh = norm_shape(A.d);
#define M2RNN_ROWS_CASE(PER)                                                            \
  if (sh.threads == 0 && sh.per == PER) {                                               \
    if (backward)                                                                       \
      norm_rows_backward_kernel<PER><<<grid, 32 * kRowWarps, 0, s>>>(A);                \
    else                                                                                \
      norm_rows_kernel<PER><<<grid, 32 * kRowWarps, 0, s>>>(A);                         \
    return cudaGetLastError();                                                          \
  }
  M2RNN_ROWS_CASE(1)
  M2RNN_ROWS_CASE(2)
  M2RNN_ROWS_CASE(4)
  M2RNN_ROWS_CASE(8)
#undef M2RNN_ROWS_CASE
#define M2RNN_NORM_CASE(TH, PER)                                                   \
  if (sh.threads == TH && sh.per == PER) {                                         \
    if (backward)                                                                  \
      output_norm_backward_kernel<TH, PER><<<grid, TH, 0, s>>>(A);                 \
    else                                                                           \
      output_norm_kernel<TH, PER><<<grid, TH, 0, s>>>(A);                          \
    return cudaGetLastError();                                                     \
  }
  M2RNN_NORM_CASE(256, 2)
  M2RNN_NORM_CASE(256, 4)
  M2RNN_NORM_CASE(256, 8)
  M2RNN_NORM_CASE(512, 8)
#undef M2RNN_NORM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

int output_norm_max_width() { return 4 * 512 * 8; }

// Backward partial count: a fixed function of the shape, enough blocks to
// cover every SM a few times over.
int output_norm_backward_parts(int64_t rows, int d) {
  const NormShape sh = norm_shape(d);
  const int64_t want = sh.threads == 0 ? (rows + kRowWarps - 1) / kRowWarps : rows;
  const int64_t cap = sh.threads == 0 ? 608 : (sh.threads <= 256 ? 608 : 304);
  return static_cast<int>(want < cap ? want : cap);
}

int gate_backward_parts(int64_t BT) {
  const int64_t p = (BT + 4 * kGateThreads - 1) / (4 * kGateThreads);
  return static_cast<int>(p < 128 ? p : 128);
}

cudaError_t launch_gate_backward(const GateSrc& gs, float* grad, float* dalpha, float* dbeta, float* part,
                                 int64_t BT, int N, cudaStream_t s) {
  const int P = gate_backward_parts(BT);
  gate_backward_kernel<<<dim3(P, N), kGateThreads, 0, s>>>(gs, grad, reinterpret_cast<float2*>(part), BT, N);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gate_finish_kernel<<<(N + 127) / 128, 128, 0, s>>>(reinterpret_cast<const float2*>(part), dalpha, dbeta, P, N);
  return cudaGetLastError();
}

cudaError_t launch_output_norm(const float* y, const void* g, const float* w, float eps, float* out, float* rstd,
                               int64_t rows, int d, bool bf16, cudaStream_t s) {
  NormArgs A{};
  A.y = y; A.g = g; A.w = w; A.out = out; A.rstd = rstd;
  A.rows = rows; A.d = d; A.eps = eps; A.bf16 = bf16; A.vec = (d % 4) == 0;
  const NormShape sh = norm_shape(d);
  const int64_t want = sh.threads == 0 ? (rows + kRowWarps - 1) / kRowWarps : rows;
  const int64_t cap = 152 * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  return launch_norm(false, A, grid, s);
}

cudaError_t launch_output_norm_backward(const float* y, const void* g, const float* w, const float* dout, float eps,
                                        float* dy, float* dg, float* dw, float* part, int64_t rows, int d,
                                        bool bf16, cudaStream_t s) {
  NormArgs A{};
  A.y = y; A.g = g; A.w = w; A.dout = dout; A.dy = dy; A.dg = dg; A.dw_part = part;
  A.rows = rows; A.d = d; A.eps = eps; A.bf16 = bf16; A.vec = (d % 4) == 0;
  const int P = output_norm_backward_parts(rows, d);
  cudaError_t e = launch_norm(true, A, P, s);
  if (e != cudaSuccess) return e;
  sum_columns_kernel<<<(d + 31) / 32, 32 * kSumWarps, 0, s>>>(part, dw, P, d);
  return cudaGetLastError();
}

}  // namespace m2rnn
