// Pipelined forward scan for small value heads, V = 16 (bf16 inputs, fp32
// state): the multi-value configuration of "M2RNN: Non-Linear RNNs with
// Matrix-Valued States for Scalable Language Modeling" (reading notes
// section 2.4), Eq. 10-12 of section 2.1, for up to 64 key rows per head.
//
// One CTA per (b, n) head.  Key rows never mix, so each block of 16 rows has
// a pair of warps on one scheduler and TMEM lane quadrant:
//   compute warp: the recurrence, as in the register-resident kernel (two
//     m16n8k16 MMAs per step with W in registers and the warp's own fp16 H
//     block as the A operand, seeded with k v^T, then tanh and the gate
//     blend); it leaves H_t (its fp16 A-operand pairs) in a double-buffered
//     tile of tensor memory, 4 columns per step, and writes checkpoints and
//     the Z stash;
//   readout warp: one tile of 32 steps behind, the block's share of
//     y_t = H_t^T q_t on the tensor core with fp16 operands (q replicated
//     over the A rows, H_t as B, transposed with movmatrix), stored one
//     step late so that no step waits for its own MMA; at the end of a tile
//     the readout warps add the row blocks' shares in a fixed order, plus
//     w_r * v_t, and write y.
// The compute warps never stop for the readout or for each other.  A
// producer warp streams k, v by TMA into a ring of input stages that the
// readout warps release; its lanes load f and q (q re-encoded as fp16, its
// range checked).  Every wait is bounded.
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
constexpr int kS = 32;       // steps per input tile
constexpr int kNS = 4;       // input stages: read out, computed, loading, spare
constexpr int kHCols = 4;    // TMEM columns per step (H_t as fp16 pairs, the A-fragment order)
constexpr int kThreads = 9 * 32;

struct MvFwdPipeParams {
  FwdArgs a;
  int R;
  int ntiles;
  uint32_t stage_off, stage_bytes, q_off, k_off, v_off, f_off, y_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

template <bool kCk, bool kZ>
__global__ void __launch_bounds__(kThreads, 1)
    mv_forward_pipe_kernel(const __grid_constant__ MvFwdPipeParams p, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const FwdArgs& A = p.a;
  const int R = p.R, T = A.T, N = A.N, K = A.K;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  StatusBlock* status = A.status;
  uint8_t* sStage = smem + p.stage_off;
  float* sY = reinterpret_cast<float*>(smem + p.y_off);  // [2][kS][R][kV] readout shares per row block
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + kNS;
  uint64_t* hfull = empty + kNS;  // [4 row blocks][2 tiles]: H of a tile is in tensor memory
  uint64_t* hempty = hfull + 8;   // [4][2]: it has been read out
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* rabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 8);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&full[i]), 32);  // producer lanes (+ TMA bytes)
      mbar_init(smem_u32(&empty[i]), R);  // one arrival per readout warp
    }
    for (int i = 0; i < 16; ++i) mbar_init(smem_u32(&hfull[i]), 1);
    *abort_flag = 0;
    *rabort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int g = lane >> 2, qd = lane & 3;

  if (warp < R) {
    // ---------------- compute warps ----------------
    const int w = warp;
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
    const uint32_t th = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
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
    uint32_t hown[4];  // fp16 H_{t-1} of the warp's rows: its own A operand
    auto split = [&]() {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        hown[2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
        hown[2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
      }
    };
    split();
    int ck_left = A.ckpt_every, ck_idx = 0;
    bool ok = true;
    for (int tile = 0; tile < p.ntiles; ++tile) {
      const int st = tile % kNS, hb = tile & 1;
      if (!mbar_wait(smem_u32(&full[st]), (tile / kNS) & 1, abort_flag, status, kWhereFwdFull) ||
          (tile >= 2 &&
           !mbar_wait(smem_u32(&hempty[2 * w + hb]), ((tile >> 1) - 1) & 1, abort_flag, status, kWhereFwdYEmpty))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint32_t ks = smem_u32(stage + p.k_off), vs = smem_u32(stage + p.v_off), fs = smem_u32(stage + p.f_off);
      const uint32_t tt = th + static_cast<uint32_t>(hb * kS * kHCols);
      const int t0 = tile * kS;
      const int nsteps = min(kS, T - t0);
      // The step's k (rows g, g + 8), v (columns 2qd.., 8 + 2qd..) and f,
      // loaded one step ahead (the tile's last step reloads itself).
      uint32_t kr0, kr1, vq0, vq1;
      float fo;
#define MV_FWD_LOAD_OPS(s_, kr0_, kr1_, vq0_, vq1_, fo_)          \
  {                                                               \
    const uint32_t krow = ks + 2 * ((s_) * K + 16 * w + g);       \
    kr0_ = ld_shared_u16(krow);                                   \
    kr1_ = ld_shared_u16(krow + 16);                              \
    vq0_ = ld_shared_b32(vs + 2 * ((s_) * kV + 2 * qd));          \
    vq1_ = ld_shared_b32(vs + 2 * ((s_) * kV + 8 + 2 * qd));      \
    fo_ = ld_shared_f32(fs + 4 * (s_));                           \
  }
      MV_FWD_LOAD_OPS(0, kr0, kr1, vq0, vq1, fo)
      // Steps run in segments that end where a checkpoint is due.
      for (int s = 0; s < nsteps;) {
        const int seg_end = kCk ? min(nsteps, s + ck_left) : nsteps;
        const int seg_len = seg_end - s;
#pragma unroll 2
        for (; s < seg_end; ++s) {
          const int sn = s + 1 < nsteps ? s + 1 : s;
          uint32_t nkr0, nkr1, nvq0, nvq1;
          float nfo;
          MV_FWD_LOAD_OPS(sn, nkr0, nkr1, nvq0, nvq1, nfo)
          const float k0 = bf16_bits_to_f32(static_cast<uint16_t>(kr0));
          const float k1 = bf16_bits_to_f32(static_cast<uint16_t>(kr1));
          const float omf = 1.f - fo;
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = nt == 0 ? vq0 : vq1;
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            acc[nt][0] = k0 * v0;  // exact: products of bf16 values fit in fp32
            acc[nt][1] = k0 * v1;
            acc[nt][2] = k1 * v0;
            acc[nt][3] = k1 * v1;
            mma_f16_16816(acc[nt], hown, bw[nt][0], bw[nt][1]);  // + H_{t-1} W (Eq. 10)
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
          // H_t for the readout warp: the fp16 pairs just packed as the next
          // step's A operand, which are also the readout's B operand.
          tmem_st_32x32b_x4(tt + kHCols * s, hown);
          if constexpr (kZ)  // Z_t for the backward (a streaming store, off the chain)
            st_global_cs_v4(zst + static_cast<int64_t>(t0 + s) * R * 512,
                            make_uint4(pack2_f16(zv[0][0], zv[0][1]), pack2_f16(zv[0][2], zv[0][3]),
                                       pack2_f16(zv[1][0], zv[1][1]), pack2_f16(zv[1][2], zv[1][3])));
          kr0 = nkr0; kr1 = nkr1; vq0 = nvq0; vq1 = nvq1; fo = nfo;
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
#undef MV_FWD_LOAD_OPS
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&hfull[2 * w + hb]));
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
  } else if (warp >= 4 && warp < 4 + R) {
    // ---------------- readout warps ----------------
    const int w = warp - 4;
    const int CT = 32 * R;
    const int rt = threadIdx.x - 128;  // 0 .. CT - 1
    const uint32_t th = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
    const uint16_t* wr = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    for (int tile = 0; tile < p.ntiles; ++tile) {
      const int st = tile % kNS, hb = tile & 1;
      const bool mine =
          mbar_wait(smem_u32(&full[st]), (tile / kNS) & 1, abort_flag, status, kWhereFwdFull) &&
          mbar_wait(smem_u32(&hfull[2 * w + hb]), (tile >> 1) & 1, abort_flag, status, kWhereFwdYFull);
      if (!mine) *rabort = 1;
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint32_t qs = smem_u32(stage + p.q_off);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(stage + p.v_off);
      float* yp = sY + hb * (kS * R * kV);
      const int t0 = tile * kS;
      const int nsteps = min(kS, T - t0);
      if (mine) {
        tc_fence_after_sync();
        const uint32_t tt = th + static_cast<uint32_t>(hb * kS * kHCols);
        uint32_t hr[4];
        tmem_ld_32x32b<4>(tt, hr);
        float yprev[4] = {0.f, 0.f, 0.f, 0.f};  // the previous step's share (stored one step late)
        // q of the block's rows 2qd.. and 2qd+8.. as bf16 pairs (A[m][k] =
        // q[k] for every m), loaded one step ahead.
        uint32_t qlo = ld_shared_b32(qs + 2 * (16 * w + 2 * qd));
        uint32_t qhi = ld_shared_b32(qs + 2 * (16 * w + 2 * qd + 8));
#pragma unroll 2
        for (int s = 0; s < nsteps; ++s) {
          const int sn = s + 1 < nsteps ? s + 1 : s;
          const uint32_t nqlo = ld_shared_b32(qs + 2 * (sn * K + 16 * w + 2 * qd));
          const uint32_t nqhi = ld_shared_b32(qs + 2 * (sn * K + 16 * w + 2 * qd + 8));
          tmem_ld_wait();
          tmem_ld_fence_regs(hr);
          const uint32_t hc[4] = {hr[0], hr[1], hr[2], hr[3]};  // H_t, fp16 pairs
          tmem_ld_32x32b<4>(tt + kHCols * (s + 1 < nsteps ? s + 1 : s), hr);
          // y in fp16 operands: H_t (|H| <= 1) to fp16 as in the state
          // transform; q as staged in fp16 by the producer.
          const uint32_t qa[4] = {qlo, qlo, qhi, qhi};
          float yd[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_f16_16816_zc(yd[nt], qa, movmatrix_trans(hc[2 * nt]), movmatrix_trans(hc[2 * nt + 1]));
          // The previous step's share (row 0 of the row-replicated result:
          // columns 8nt + 2qd, +1); its MMAs completed during this step.
          if (g == 0 && s > 0) {
            float* dst = yp + ((s - 1) * R + w) * kV + 2 * qd;
            *reinterpret_cast<float2*>(dst) = make_float2(yprev[0], yprev[1]);
            *reinterpret_cast<float2*>(dst + 8) = make_float2(yprev[2], yprev[3]);
          }
          yprev[0] = yd[0][0];
          yprev[1] = yd[0][1];
          yprev[2] = yd[1][0];
          yprev[3] = yd[1][1];
          qlo = nqlo;
          qhi = nqhi;
        }
        if (g == 0 && nsteps > 0) {
          float* dst = yp + ((nsteps - 1) * R + w) * kV + 2 * qd;
          *reinterpret_cast<float2*>(dst) = make_float2(yprev[0], yprev[1]);
          *reinterpret_cast<float2*>(dst + 8) = make_float2(yprev[2], yprev[3]);
        }
        // The tile's H is read (the last, repeated load included): the
        // compute warp may overwrite it.
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&hempty[2 * w + hb]));
      }
      named_bar_sync(1, CT);  // every row block's shares of the tile are written
      if (*rabort) break;
      // The tile's y: the row blocks summed in a fixed order, plus w_r * v.
      // (The share buffer alternates by tile, so no barrier is needed before
      // the next tile writes.)
      for (int idx = rt; idx < nsteps * kV; idx += CT) {
        const int s = idx / kV, j = idx % kV;
        float sum = 0.f;
        for (int ww = 0; ww < R; ++ww) sum += yp[(s * R + ww) * kV + j];
        const int64_t row = (static_cast<int64_t>(b) * T + t0 + s) * N + n;
        A.y[row * kV + j] = fmaf(bf16_bits_to_f32(wr[j]), bf16_bits_to_f32(vs[s * kV + j]), sum);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));  // past its last read of the stage
    }
    if (*rabort) *abort_flag = 1;
  } else if (warp == 8) {
    // ---------------- producer (k, v by TMA; q and f by its lanes) ----------------
    if (lane == 0) {
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
      {
        // q of step t0 + lane (all K rows), re-encoded as fp16 for the
        // readout's MMA once here instead of at every readout step; a
        // magnitude the fp16 operand cannot hold is reported.
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(A.q) +
            ((static_cast<int64_t>(b) * T + t0 + lane) * qk_heads(A.qkN, N) + qk_head(A.qkN, n)) * K);
        uint4* dst = reinterpret_cast<uint4*>(stage + p.q_off + lane * K * 2);
        uint32_t mag = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // K / 8 pieces of 16 bytes, K <= 64
          if (i < K / 8) {
            uint4 qv = t0 + lane < T ? src[i] : make_uint4(0u, 0u, 0u, 0u);
            mag = __vmaxu2(mag, __vmaxu2(qv.x & 0x7FFF7FFFu, qv.y & 0x7FFF7FFFu));
            mag = __vmaxu2(mag, __vmaxu2(qv.z & 0x7FFF7FFFu, qv.w & 0x7FFF7FFFu));
            qv = make_uint4(bf16x2_to_f16x2(qv.x), bf16x2_to_f16x2(qv.y), bf16x2_to_f16x2(qv.z),
                            bf16x2_to_f16x2(qv.w));
            dst[i] = qv;
          }
        }
        if ((mag & 0xFFFFu) >= 0x4780u || (mag >> 16) >= 0x4780u)  // |q| >= 65536 (or not finite)
          report_device_error(status, kStatusCheck, kWhereQRange);
      }
      __syncwarp();
      const uint32_t fb = smem_u32(&full[st]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, p.tx_bytes);
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
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <bool kCk, bool kZ>
cudaError_t launch_t(const MvFwdPipeParams& p, uint32_t smem, cudaStream_t stream, const CUtensorMap& mk,
                     const CUtensorMap& mv) {
  auto kernel = mv_forward_pipe_kernel<kCk, kZ>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<p.a.B * p.a.N, kThreads, smem, stream>>>(p, mk, mv);
  return cudaGetLastError();
}

}  // namespace

bool mv_forward_pipe_supported(int K, int V, bool readout) {
  return readout && V == kV && K % kRows == 0 && K >= kRows && K <= 4 * kRows;
}

cudaError_t launch_mv_forward_pipe(const FwdArgs& a, cudaStream_t stream) {
  if (!mv_forward_pipe_supported(a.K, a.V, a.y != nullptr)) return cudaErrorInvalidValue;
  MvFwdPipeParams p{};
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
  p.misc_off = p.bar_off + (2 * kNS + 16) * 8;
  const uint32_t smem = align_up(p.misc_off + 16, 128);
  p.tx_bytes = kS * a.K * 2 + kS * kV * 2;  // k and v by TMA (q is staged by the producer's lanes)

  CUtensorMap mk, mv;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, a.K, kS) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, kS))
    return cudaErrorInvalidValue;
  const bool ck = a.ckpt != nullptr, z = a.zstash != nullptr;
  if (z) return ck ? launch_t<true, true>(p, smem, stream, mk, mv) : launch_t<false, true>(p, smem, stream, mk, mv);
  return ck ? launch_t<true, false>(p, smem, stream, mk, mv) : launch_t<false, false>(p, smem, stream, mk, mv);
}

}  // namespace m2rnn
