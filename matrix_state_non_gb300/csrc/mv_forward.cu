// Register-resident forward scan for small value heads, V = 16 (bf16
// inputs, fp32 state): the multi-value configuration of "M2RNN: Non-Linear
// RNNs with Matrix-Valued States for Scalable Language Modeling" (reading
// notes section 2.4: K = 64, V = 16, optionally one q/k shared by every
// head), Eq. 10-12 of section 2.1.
//
// One CTA per (b, n) head; compute warp w owns key rows 16w..16w+15 and all
// 16 value columns.  Rows never mix (section 1.2 of the notes), and a warp's
// 16 x 16 block of bf16(H_{t-1}) is exactly the A operand of its next
// m16n8k16 (the accumulator layout of its two n-tiles is the A layout of the
// one k-tile), so the recurrence of a warp needs nothing from the others:
// per step 2 warp MMAs with W (16 x 16) in registers, seeded with k v^T,
// then tanh and the gate blend on the fp32 state -- no shared-memory
// exchange and no barrier on the serial chain.  Only the readout sums over
// rows: the readout of step t-1 runs on the tensor core during step t (q
// replicated over the 16 A rows, H_{t-1} as B split into bf16 high and low
// parts, transposed from the accumulator layout with movmatrix), into a
// per-tile buffer whose row blocks the warps add in a fixed order once per
// tile of 32 steps.
// A producer warp streams q, k, v by TMA (and f by plain loads) into a
// 3-stage mbarrier ring.  Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 16;
constexpr int kRows = 16;
constexpr int kS = 32;   // steps per input tile
constexpr int kNS = 3;   // input stages
constexpr int kMaxRB = 8;  // K <= 128

struct MvFwdParams {
  FwdArgs a;
  int R;       // row blocks (compute warps)
  int ntiles;
  uint32_t stage_off, stage_bytes, q_off, k_off, v_off, f_off, y_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

// Compile-time modes: kY = readout y, kCk = checkpoints, kZ = the Z stash
// (no per-step branch on any of them).  The stash layout for V = 16: per
// (chain, step) the R row-block warps' 512 bytes each, lane l's 16 bytes
// holding its fp16 Z values in accumulator-fragment order, so a chunk of
// steps is one contiguous range.
template <bool kY, bool kCk, bool kZ>
__global__ void __launch_bounds__((kMaxRB + 1) * 32, 1)
    mv_forward_kernel(const __grid_constant__ MvFwdParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const FwdArgs& A = p.a;
  const int R = p.R, T = A.T, N = A.N, K = A.K;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  StatusBlock* status = A.status;
  uint8_t* sStage = smem + p.stage_off;
  float* sY = reinterpret_cast<float*>(smem + p.y_off);  // [2][kS][R][kV] per-warp readout partials
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + kNS;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* cabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  constexpr bool do_y = kY;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&full[i]), 32);  // producer lanes (+ TMA bytes)
      mbar_init(smem_u32(&empty[i]), R);  // one arrival per compute warp
    }
    *abort_flag = 0;
    *cabort = 0;
    fence_mbar_init_cluster();
  }
  __syncthreads();

  if (warp < R) {
    // ---------------- compute warps ----------------
    const int g = lane >> 2, qd = lane & 3, w = warp;
    const int CT = 32 * R;
    const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
    uint32_t bw[2][2];  // fp16 B[k][col] = W[k][8nt + col], k = 2qd.. and 2qd+8..
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = 8 * nt + g;
      bw[nt][0] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[(2 * qd) * kV + col]) |
                                  (static_cast<uint32_t>(Wg[(2 * qd + 1) * kV + col]) << 16));
      bw[nt][1] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[(2 * qd + 8) * kV + col]) |
                                  (static_cast<uint32_t>(Wg[(2 * qd + 9) * kV + col]) << 16));
      if (!f16x2_finite(bw[nt][0]) || !f16x2_finite(bw[nt][1]))
        report_device_error(status, kStatusCheck, kWhereWRange);
    }
    const int64_t row_g = static_cast<int64_t>(chain) * K + 16 * w + g;  // state row of lane g
    uint8_t* const zst = !kZ ? nullptr
                             : reinterpret_cast<uint8_t*>(A.zstash) + static_cast<int64_t>(chain) * T * R * 512 +
                                   w * 512 + lane * 16;
    float h[2][4];
    if (A.H0 != nullptr) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float2 x0 = *reinterpret_cast<const float2*>(A.H0 + row_g * kV + 8 * nt + 2 * qd);
        const float2 x1 = *reinterpret_cast<const float2*>(A.H0 + (row_g + 8) * kV + 8 * nt + 2 * qd);
        h[nt][0] = x0.x; h[nt][1] = x0.y; h[nt][2] = x1.x; h[nt][3] = x1.y;
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) h[nt][0] = h[nt][1] = h[nt][2] = h[nt][3] = 0.f;
    }
    // fp16 H_{t-1} of the warp's rows: its own A operand (see mma_common.cuh).
    uint32_t hown[4];
    auto split = [&]() {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        hown[2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
        hown[2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
      }
    };
    split();
    const uint16_t* wr = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    int ck_left = A.ckpt_every, ck_idx = 0;
    bool ok = true;
    for (int tile = 0; tile < p.ntiles; ++tile) {
      const int st = tile % kNS, yb = tile & 1;
      const bool mine = mbar_wait_timed(smem_u32(&full[st]), (tile / kNS) & 1, status, kWhereFwdFull);
      if (!mine) *cabort = 1;
      named_bar_sync(1, CT);
      if (*cabort) {
        ok = false;
        break;
      }
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(stage + p.q_off);
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(stage + p.k_off);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(stage + p.v_off);
      const float* fs = reinterpret_cast<const float*>(stage + p.f_off);
      float* yp = sY + yb * (kS * R * kV);
      const int t0 = tile * kS;
      const int nsteps = min(kS, T - t0);
      // Readout of y_{t-1} = H_{t-1}^T q_{t-1} over this warp's 16 rows, as
      // m16n8k16 MMAs: A[m][k] = q[k] for every m, B[k][n] = H[k][n].
      auto readout_mma = [&](uint32_t qlo, uint32_t qhi, float (&yd)[2][4]) {
        uint32_t qa[4];
        qa[0] = qa[1] = qlo;
        qa[2] = qa[3] = qhi;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {  // H_{t-1} as bf16 high and low parts (~16 bits)
          const uint32_t hi0 = pack2_bf16(h[nt][0], h[nt][1]);
          const uint32_t hi1 = pack2_bf16(h[nt][2], h[nt][3]);
          const uint32_t lo0 = pack2_bf16(h[nt][0] - bf16lo(hi0), h[nt][1] - bf16hi(hi0));
          const uint32_t lo1 = pack2_bf16(h[nt][2] - bf16lo(hi1), h[nt][3] - bf16hi(hi1));
          yd[nt][0] = yd[nt][1] = yd[nt][2] = yd[nt][3] = 0.f;
          mma_bf16_16816(yd[nt], qa, movmatrix_trans(hi0), movmatrix_trans(hi1));
          mma_bf16_16816(yd[nt], qa, movmatrix_trans(lo0), movmatrix_trans(lo1));
        }
      };
      auto store_y = [&](const float (&yd)[2][4], int sp) {
        if (g == 0) {  // row 0 of the (row-replicated) result: columns 8nt + 2qd (+1)
          float* dst = yp + (sp * R + w) * kV + 2 * qd;
          *reinterpret_cast<float2*>(dst) = make_float2(yd[0][0], yd[0][1]);
          *reinterpret_cast<float2*>(dst + 8) = make_float2(yd[1][0], yd[1][1]);
        }
      };
      // Steps run in segments that end where a checkpoint is due.
      for (int s = 0; s < nsteps;) {
        const int seg_end = kCk ? min(nsteps, s + ck_left) : nsteps;
        const int seg_len = seg_end - s;
        for (; s < seg_end; ++s) {
          const float k0 = bf16_bits_to_f32(ks[s * K + 16 * w + g]);
          const float k1 = bf16_bits_to_f32(ks[s * K + 16 * w + g + 8]);
          const float omf = 1.f - fs[s];
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * kV + 8 * nt + 2 * qd);
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            acc[nt][0] = k0 * v0;  // exact: products of bf16 values fit in fp32
            acc[nt][1] = k0 * v1;
            acc[nt][2] = k1 * v0;
            acc[nt][3] = k1 * v1;
            mma_f16_16816(acc[nt], hown, bw[nt][0], bw[nt][1]);  // + H_{t-1} W (Eq. 10)
          }
          float yd[2][4];
          if (do_y && s > 0) {
            const uint32_t qlo = *reinterpret_cast<const uint32_t*>(qs + (s - 1) * K + 16 * w + 2 * qd);
            const uint32_t qhi = *reinterpret_cast<const uint32_t*>(qs + (s - 1) * K + 16 * w + 2 * qd + 8);
            readout_mma(qlo, qhi, yd);
          }
          float zv[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              zv[nt][e] = tanh_fast(acc[nt][e]);
              h[nt][e] = fmaf(omf, zv[nt][e] - h[nt][e], h[nt][e]);  // Eq. 11
            }
          split();
          if constexpr (kZ)  // Z_t for the backward (a streaming store, off the chain)
            st_global_cs_v4(zst + static_cast<int64_t>(t0 + s) * R * 512,
                            make_uint4(pack2_f16(zv[0][0], zv[0][1]), pack2_f16(zv[0][2], zv[0][3]),
                                       pack2_f16(zv[1][0], zv[1][1]), pack2_f16(zv[1][2], zv[1][3])));
          if (do_y && s > 0) store_y(yd, s - 1);
        }
        if constexpr (kCk) {
          ck_left -= seg_len;
          if (ck_left == 0) {  // H after step t0 + s - 1 starts a chunk: checkpoint it
            ck_left = A.ckpt_every;
            ++ck_idx;
            if (t0 + s < T) {
              float* dst = A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + ck_idx - 1) * K + 16 * w + g) * kV;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) = make_float2(h[nt][0], h[nt][1]);
                *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt + 2 * qd) = make_float2(h[nt][2], h[nt][3]);
              }
            }
          }
        }
      }
      if (do_y && nsteps > 0) {  // the tile's last step
        const uint32_t qlo = *reinterpret_cast<const uint32_t*>(qs + (nsteps - 1) * K + 16 * w + 2 * qd);
        const uint32_t qhi = *reinterpret_cast<const uint32_t*>(qs + (nsteps - 1) * K + 16 * w + 2 * qd + 8);
        float yd[2][4];
        readout_mma(qlo, qhi, yd);
        store_y(yd, nsteps - 1);
      }
      // The tile's y: the row blocks summed in a fixed order, plus w_r * v.
      named_bar_sync(1, CT);
      if (do_y) {
        for (int idx = threadIdx.x; idx < nsteps * kV; idx += CT) {
          const int s = idx / kV, j = idx % kV;
          float sum = 0.f;
          for (int ww = 0; ww < R; ++ww) sum += yp[(s * R + ww) * kV + j];
          const int64_t row = (static_cast<int64_t>(b) * T + t0 + s) * N + n;
          A.y[row * kV + j] = fmaf(bf16_bits_to_f32(wr[j]), bf16_bits_to_f32(vs[s * kV + j]), sum);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));  // this warp is past its last read of the stage
    }
    if (ok && A.H_T != nullptr) {
      float* dst = A.H_T + row_g * kV;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) = make_float2(h[nt][0], h[nt][1]);
        *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt + 2 * qd) = make_float2(h[nt][2], h[nt][3]);
      }
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == R) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const GateSrc gs{A.f, A.gate_a, A.gate_alpha, A.gate_beta, true};
    int issued = 0;
    bool ok = true;
    for (int tile = 0; tile < p.ntiles; ++tile) {
      const int st = tile % kNS;
      if (tile >= kNS &&
          !mbar_wait(smem_u32(&empty[st]), ((tile / kNS) - 1) & 1, abort_flag, status, kWhereFwdEmpty)) {
        ok = false;
        break;
      }
      const int t0 = tile * kS;
      uint8_t* stage = sStage + st * p.stage_bytes;
      float fv = 0.f;
      if (t0 + lane < T) fv = gate_value(gs, (static_cast<int64_t>(b) * T + t0 + lane) * N + n, n);
      reinterpret_cast<float*>(stage + p.f_off)[lane] = fv;
      __syncwarp();
      const uint32_t fb = smem_u32(&full[st]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, p.tx_bytes);
        tma_load_4d(smem_u32(stage + p.q_off), &tm_q, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(stage + p.k_off), &tm_k, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(stage + p.v_off), &tm_v, fb, 0, n, t0, b);
      } else {
        mbar_arrive(fb);
      }
      issued = tile + 1;
    }
    if (!ok) {
      for (int tile = std::max(0, issued - kNS); tile < issued; ++tile)
        mbar_wait_timed(smem_u32(&full[tile % kNS]), (tile / kNS) & 1, nullptr, kWhereFwdDrain);
    }
  }
  __syncthreads();
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

}  // namespace

bool mv_forward_supported(int K, int V) { return V == kV && K % kRows == 0 && K >= kRows && K <= kRows * kMaxRB; }

cudaError_t launch_mv_forward(const FwdArgs& a, cudaStream_t stream) {
  if (mv_forward_pipe_supported(a.K, a.V, a.y != nullptr)) return launch_mv_forward_pipe(a, stream);
  MvFwdParams p{};
  p.a = a;
  p.R = a.K / kRows;
  p.ntiles = (a.T + kS - 1) / kS;
  p.stage_off = 0;
  p.q_off = 0;
  p.k_off = align_up(kS * a.K * 2, 128);
  p.v_off = p.k_off + align_up(kS * a.K * 2, 128);
  p.f_off = p.v_off + align_up(kS * kV * 2, 128);
  p.stage_bytes = align_up(p.f_off + kS * 4, 128);
  p.y_off = kNS * p.stage_bytes;
  p.bar_off = p.y_off + 2 * kS * p.R * kV * 4;
  p.misc_off = p.bar_off + 2 * kNS * 8;
  const uint32_t smem = align_up(p.misc_off + 16, 128);
  p.tx_bytes = 2 * kS * a.K * 2 + kS * kV * 2;

  CUtensorMap mq, mk, mv;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, a.K, a.K, kS) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, a.K, kS) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, kS))
    return cudaErrorInvalidValue;
  auto pick = [&](auto z) {
    constexpr bool Z = decltype(z)::value;
    return a.y != nullptr ? (a.ckpt != nullptr ? mv_forward_kernel<true, true, Z> : mv_forward_kernel<true, false, Z>)
                          : (a.ckpt != nullptr ? mv_forward_kernel<false, true, Z> : mv_forward_kernel<false, false, Z>);
  };
  auto kernel = a.zstash != nullptr ? pick(std::true_type{}) : pick(std::false_type{});
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<a.B * a.N, (p.R + 1) * 32, smem, stream>>>(p, mq, mk, mv);
  return cudaGetLastError();
}

}  // namespace m2rnn
