// One decoding step (Eq. 10-12 of "M2RNN: Non-Linear RNNs with
// Matrix-Valued States for Scalable Language Modeling", reading notes
// section 2.1) for a batch of (b, n) states: the fixed-size recurrent state
// of section 2.6 advanced by one token, in place.
//
// One CTA per (b, n), one warp per 16 key rows.  A warp holds all 64 value
// columns of its rows, so the accumulator layout of its eight n-tiles is
// the A-operand layout of the next MMA's four k-tiles: the state never
// leaves the warp (no shared-memory exchange, no barrier on the chain).
//   acc = k v^T + bf16(H_{t-1}) W   (32 warp MMAs; W staged once per CTA in
//                                    shared memory, fragments by ldmatrix)
//   Z = tanh(acc); H_t = f H_{t-1} + (1 - f) Z        (fp32)
//   y = H_t^T q + w_r * v: row sums over the warp's 16 rows by shuffles,
//       then over the row blocks in shared memory, in a fixed order.
// Used for bf16 inputs, V = 64 and K a multiple of 16 (at most 128).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 64;
constexpr int kMaxWarps = 8;  // K <= 128

__global__ void __launch_bounds__(kMaxWarps * 32) decode_step_kernel(
    float* __restrict__ H, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const uint16_t* __restrict__ f, const uint16_t* __restrict__ W,
    const uint16_t* __restrict__ w_r, float* __restrict__ y, int N, int K, int qkN, StatusBlock* status) {
  // Nothing in this kernel waits, so it has no device error to report: it
  // only clears the caller's status block, as every call does.
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    status->code = 0u;
    status->detail = 0u;
  }
  __shared__ float ypart[kMaxWarps][kV];
  __shared__ __align__(128) uint8_t wtile[4][2048];  // W as four 16 x 64 fp16 k-tiles (swizzled)
  const int chain = blockIdx.x, n = chain % N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, qd = lane & 3;
  const int nw = K / 16;
  const int64_t r0 = static_cast<int64_t>(chain) * K + 16 * warp;  // first state row of this warp
  const uint16_t* Wn = W + static_cast<int64_t>(n) * kV * kV;
  const int64_t qkrow = static_cast<int64_t>(chain / N) * qk_heads(qkN, N) + qk_head(qkN, n);
  const uint16_t* kc = k + qkrow * K;
  const uint16_t* qc = q + qkrow * K;
  const uint16_t* vc = v + static_cast<int64_t>(chain) * kV;
  const float ft = bf16_bits_to_f32(f[chain]);
  const float omf = 1.f - ft;

  // H_{t-1} of rows g, g+8, columns 8nt + 2qd (+1), in the accumulator layout
  // (its loads are in flight while W is staged).
  float h[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const float2 x0 = *reinterpret_cast<const float2*>(H + (r0 + g) * kV + 8 * nt + 2 * qd);
    const float2 x1 = *reinterpret_cast<const float2*>(H + (r0 + g + 8) * kV + 8 * nt + 2 * qd);
    h[nt][0] = x0.x; h[nt][1] = x0.y; h[nt][2] = x1.x; h[nt][3] = x1.y;
  }
  for (int e = threadIdx.x; e < kV * kV / 8; e += blockDim.x) {  // 16-byte chunks of W
    const int row = e >> 3, col = (e & 7) * 8;
    const uint4 x = *reinterpret_cast<const uint4*>(Wn + row * kV + col);  // bf16, re-encoded as fp16
    *reinterpret_cast<uint4*>(wtile[row >> 4] + tile_off(row & 15, col)) =
        make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
  }
  __syncthreads();
  const float k0 = bf16_bits_to_f32(kc[16 * warp + g]), k1 = bf16_bits_to_f32(kc[16 * warp + g + 8]);
  float acc[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const uint32_t vv = *reinterpret_cast<const uint32_t*>(vc + 8 * nt + 2 * qd);
    const float v0 = bf16lo(vv), v1 = bf16hi(vv);
    acc[nt][0] = k0 * v0;
    acc[nt][1] = k0 * v1;
    acc[nt][2] = k1 * v0;
    acc[nt][3] = k1 * v1;
  }
#pragma unroll
  for (int kt = 0; kt < 4; ++kt) {
    // fp16 k-tile kt of H = n-tiles 2kt, 2kt+1 of the accumulator layout
    // (the scan kernels' operand precision).
    uint32_t a[4];
    a[0] = pack2_f16(h[2 * kt][0], h[2 * kt][1]);
    a[1] = pack2_f16(h[2 * kt][2], h[2 * kt][3]);
    a[2] = pack2_f16(h[2 * kt + 1][0], h[2 * kt + 1][1]);
    a[3] = pack2_f16(h[2 * kt + 1][2], h[2 * kt + 1][3]);
    const uint32_t wt = smem_u32(wtile[kt]);
#pragma unroll
    for (int nt2 = 0; nt2 < 4; ++nt2) {
      uint32_t bd[4];  // B fragments (k = W row, n = W column) of n-tiles 2nt2, 2nt2+1
      ldmatrix_x4_trans(bd, ldsm_addr_b_trans(wt, nt2, lane));
      mma_f16_16816(acc[2 * nt2], a, bd[0], bd[1]);
      mma_f16_16816(acc[2 * nt2 + 1], a, bd[2], bd[3]);
    }
  }
  const float q0 = bf16_bits_to_f32(qc[16 * warp + g]), q1 = bf16_bits_to_f32(qc[16 * warp + g + 8]);
  float yp[8][2];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) h[nt][e] = fmaf(omf, tanh_fast(acc[nt][e]) - h[nt][e], h[nt][e]);
    *reinterpret_cast<float2*>(H + (r0 + g) * kV + 8 * nt + 2 * qd) = make_float2(h[nt][0], h[nt][1]);
    *reinterpret_cast<float2*>(H + (r0 + g + 8) * kV + 8 * nt + 2 * qd) = make_float2(h[nt][2], h[nt][3]);
    yp[nt][0] = fmaf(q0, h[nt][0], q1 * h[nt][2]);
    yp[nt][1] = fmaf(q0, h[nt][1], q1 * h[nt][3]);
  }
  // Sum over the eight g lanes of each column (fixed tree), then over warps.
#pragma unroll
  for (int o = 4; o < 32; o <<= 1)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      yp[nt][0] += __shfl_xor_sync(0xffffffffu, yp[nt][0], o);
      yp[nt][1] += __shfl_xor_sync(0xffffffffu, yp[nt][1], o);
    }
  if (g == 0)
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
      *reinterpret_cast<float2*>(&ypart[warp][8 * nt + 2 * qd]) = make_float2(yp[nt][0], yp[nt][1]);
  __syncthreads();
  for (int j = threadIdx.x; j < kV; j += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += ypart[w][j];
    y[static_cast<int64_t>(chain) * kV + j] =
        fmaf(bf16_bits_to_f32(w_r[static_cast<int64_t>(n) * kV + j]), bf16_bits_to_f32(vc[j]), s);
  }
}

}  // namespace

bool decode_kernel_supported(int K, int V, m2rnn_dtype dtype) {
  return dtype == M2RNN_BF16 && V == kV && K % 16 == 0 && K >= 16 && K <= 16 * kMaxWarps;
}

cudaError_t launch_decode_step(float* H, const void* q, const void* k, const void* v, const void* f,
                               const void* W, const void* w_r, float* y, int B, int N, int K, int qkN,
                               StatusBlock* status, cudaStream_t stream) {
  decode_step_kernel<<<B * N, 32 * (K / 16), 0, stream>>>(
      H, static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
      static_cast<const uint16_t*>(f), static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(w_r), y, N, K, qkN, status);
  return cudaGetLastError();
}

}  // namespace m2rnn
