// Pipelined backward-through-time for small value heads, V = 16 (bf16
// inputs, fp32 state and gradients): the multi-value configuration of
// "M2RNN: Non-Linear RNNs with Matrix-Valued States for Scalable Language
// Modeling" (reading notes section 2.4), with the chain rule of section 2.7;
// u_t = dy_t, C_T = dH_T:
//   R_t = C_t + q_t u_t^T,  D_t = ((1-f_t) R_t) * (1 - Z_t * Z_t),
//   C_{t-1} = f_t R_t + D_t W^T,
//   dq_t = H_t u_t, dk_t = D_t v_t, dv_t = D_t^T k_t + w_r * u_t,
//   df_t = <R_t, H_{t-1} - Z_t>,  dW += H_{t-1}^T D_t,  dw_r += u_t * v_t.
//
// One CTA per (b, n) head.  Key rows never mix, so each block of 16 rows is
// served by a pair of warps that share a TMEM lane quadrant:
//   rebuild warp: advances the block's state through a chunk from its start
//     state (the gate blend on the forward's Z stash, or the forward's step
//     with its MMA and tanh), keeps its dq_t = H_t u_t shares, and leaves per
//     step G = (1-f)(1-Z^2) and E = H_{t-1} - Z (fp16 pairs) and the bf16
//     H_{t-1}^T fragments of the dW product in a double-buffered chunk cache
//     in tensor memory, one chunk ahead of
//   chain warp: walks the chunk backwards with the state gradient in
//     registers: R, D = R * G, the chain MMA C_{t-1} = f R + D W^T (the bf16
//     D block is its A operand), and from the same block on the tensor core
//     dW += H_{t-1}^T D, dk = D v (v as column 0 of B) and the block's share
//     of dv = D^T k (k as row 0 of A); the df share <R, E> of every lane goes
//     to shared memory.  MMA results are stored one step late, so no step
//     waits for its own products.
// At the end of a chunk the chain warps add the dv and df shares over row
// blocks (and lanes) in a fixed order, and each rebuild warp adds its dq
// shares over the four lanes of a row.  The serial chain keeps only its own
// latency per step; the cross-lane sums run once per chunk with every load
// in flight.  A producer warp streams the chunk's q, k, v, dy (TMA), f, and
// the Z stash (bulk copy).  Every wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 16;
constexpr int kRows = 16;
constexpr int kCacheCols = 12;  // per step and thread: G (4 fp16 pairs), E (4), H^T fragments (4)
constexpr int kNS = 3;          // input slots (q, k, v, dy, f): chain chunk, rebuild chunk, next
constexpr int kNZ = 2;          // Z stash slots

struct PipeParams {
  BwdArgs a;
  int R, nq, nchunks;
  uint32_t set_cols;  // TMEM columns of one lane-quadrant set (two chunk buffers)
  uint32_t s_off, s_bytes, q_off, k_off, v_off, dy_off, f_off;  // input slots
  uint32_t z_off, z_bytes;                                      // Z stash slots
  uint32_t dvp_off, dv_step, dfp_off, df_step, qp_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

// Maximum chunk length: two chunk buffers of 12 columns per step in 512 TMEM
// columns per lane quadrant (one set for up to four row blocks, two sets for
// up to eight), and the shared-memory slots.
__host__ __device__ inline int pipe_max_chunk(int R) { return R <= 4 ? 20 : 10; }

template <bool kClip, bool kZ, bool kWide>
__global__ void __launch_bounds__(kWide ? 544 : 288, 1)
    mv_backward_pipe_kernel(const __grid_constant__ PipeParams p, const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_dy) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const BwdArgs& A = p.a;
  const int R = p.R, T = A.T, N = A.N, K = A.K, CL = A.ckpt_every;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  const int rb0 = 4 * p.nq, prod = 8 * p.nq;  // first rebuild warp, the producer warp
  StatusBlock* status = A.status;
  uint64_t* sfull = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* sempty = sfull + kNS;
  uint64_t* zfull = sempty + kNS;
  uint64_t* zempty = zfull + kNZ;
  uint64_t* cfull = zempty + kNZ;  // [8 row blocks][2 chunk buffers]
  uint64_t* cempty = cfull + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* cabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 8);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&sfull[i]), 32);  // producer lanes (+ TMA bytes)
      mbar_init(smem_u32(&sempty[i]), R);  // one arrival per chain warp
    }
    for (int i = 0; i < kNZ; ++i) {
      mbar_init(smem_u32(&zfull[i]), 1);
      mbar_init(smem_u32(&zempty[i]), R);  // one arrival per rebuild warp
    }
    for (int i = 0; i < 32; ++i) mbar_init(smem_u32(&cfull[i]), 1);
    *abort_flag = 0;
    *cabort = 0;
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
  const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;

  if (warp < R) {
    // ---------------- chain warps: the reverse walk ----------------
    const int w = warp;
    const int CT = 32 * R;
    uint32_t bt[2][2];  // B fragments of W^T (bf16): C_{t-1} = f R + D W^T
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = 8 * nt + g;
      bt[nt][0] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + 2 * qd);
      bt[nt][1] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + 2 * qd + 8);
    }
    const int64_t row_g = static_cast<int64_t>(chain) * K + 16 * w + g;  // state row of lane g
    float2 Ct[2], Cb[2];  // C_t: rows g (top) and g + 8 (bottom), columns 8nt + 2qd, +1
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (A.dH_T != nullptr) {
        Ct[nt] = *reinterpret_cast<const float2*>(A.dH_T + row_g * kV + 8 * nt + 2 * qd);
        Cb[nt] = *reinterpret_cast<const float2*>(A.dH_T + (row_g + 8) * kV + 8 * nt + 2 * qd);
      } else {
        Ct[nt] = Cb[nt] = make_float2(0.f, 0.f);
      }
    }
    float dWacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * (w & 3)) << 16) + (w >> 2) * p.set_cols;
    const uint16_t* wrg = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    // Per-step partials of the warp's rows: dv (lanes 0..3, four columns
    // each) and df.
    const uint32_t dvp = smem_u32(smem + p.dvp_off) + static_cast<uint32_t>((w * 4 + qd) * 16);
    const uint32_t dfp = smem_u32(smem + p.dfp_off) + static_cast<uint32_t>((w * 32 + lane) * 4);
    // The end-of-chunk dv task of this thread writes column tid % 16.
    const int jc = threadIdx.x & 15;
    const float wrc = bf16_bits_to_f32(wrg[jc]);
    bool ok = true;
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL, L = min(CL, T - s0);
      const int ss = ci % kNS, cb = ci & 1;
      const bool mine = mbar_wait(smem_u32(&sfull[ss]), (ci / kNS) & 1, abort_flag, status, kWhereBwdFull) &&
                        mbar_wait(smem_u32(&cfull[2 * w + cb]), (ci >> 1) & 1, abort_flag, status, kWhereBwdTReady);
      if (!mine) *cabort = 1;
      const uint8_t* sbuf = smem + p.s_off + ss * p.s_bytes;
      const uint32_t cq = smem_u32(sbuf + p.q_off), ck = smem_u32(sbuf + p.k_off), cv = smem_u32(sbuf + p.v_off);
      const uint32_t cdy = smem_u32(sbuf + p.dy_off), cf = smem_u32(sbuf + p.f_off);
      if (mine) {
        tc_fence_after_sync();
        const uint32_t tc = tq + static_cast<uint32_t>(cb * kCacheCols * CL);
        uint32_t ca[8], cx[4];
        tmem_ld_32x32b<8>(tc + kCacheCols * (L - 1), ca);
        tmem_ld_32x32b<4>(tc + kCacheCols * (L - 1) + 8, cx);
        // The step's operands from the chunk's input slot, loaded one step ahead.
        float q0, q1, ft;
        float2 u0, u1;
        uint32_t kp0, kp1, vb0, vb1;
#define MV_PIPE_LOAD_OPS(s_, q0_, q1_, ft_, u0_, u1_, kp0_, kp1_, vb0_, vb1_)                              \
  {                                                                                                        \
    const uint32_t qrow = cq + 2 * ((s_) * K + 16 * w + g);                                                \
    q0_ = bf16_bits_to_f32(ld_shared_u16(qrow));                                                           \
    q1_ = bf16_bits_to_f32(ld_shared_u16(qrow + 16));                                                      \
    ft_ = ld_shared_f32(cf + 4 * (s_));                                                                    \
    u0_ = ld_shared_f32x2(cdy + 4 * ((s_) * kV + 2 * qd));                                                 \
    u1_ = ld_shared_f32x2(cdy + 4 * ((s_) * kV + 8 + 2 * qd));                                             \
    const uint32_t kpair = ck + 2 * ((s_) * K + 16 * w + 2 * qd);                                          \
    kp0_ = ld_shared_b32(kpair);                                                                           \
    kp1_ = ld_shared_b32(kpair + 16);                                                                      \
    vb0_ = ld_shared_b32(cv + 2 * ((s_) * kV + 2 * qd));                                                   \
    vb1_ = ld_shared_b32(cv + 2 * ((s_) * kV + 8 + 2 * qd));                                               \
  }
        MV_PIPE_LOAD_OPS(L - 1, q0, q1, ft, u0, u1, kp0, kp1, vb0, vb1)
        // dk of step s + 1 (written one step late: the MMA result is not waited for in its own step).
        float* dkrow = A.dk + ((static_cast<int64_t>(b) * T + s0 + L) * N + n) * K + 16 * w + g;
        const int64_t dkstep = static_cast<int64_t>(N) * K;
        const bool row0 = (g == 0);
        float pdv[4] = {0.f, 0.f, 0.f, 0.f}, pdk0 = 0.f, pdk1 = 0.f;  // dv, dk of step s + 1
#pragma unroll 2
        for (int s = L - 1; s >= 0; --s) {
          const int sn = s > 0 ? s - 1 : 0;  // step 0 reloads itself (no branch in the loop)
          float nq0, nq1, nft;
          float2 nu0, nu1;
          uint32_t nkp0, nkp1, nvb0, nvb1;
          MV_PIPE_LOAD_OPS(sn, nq0, nq1, nft, nu0, nu1, nkp0, nkp1, nvb0, nvb1)
          tmem_ld_wait();
          tmem_ld_fence_regs(ca);
          tmem_ld_fence_regs(cx);
          uint32_t Gp[4], Ep[4], ha[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            Gp[i] = ca[i];
            Ep[i] = ca[4 + i];
            ha[i] = cx[i];
          }
          tmem_ld_32x32b<8>(tc + kCacheCols * sn, ca);
          tmem_ld_32x32b<4>(tc + kCacheCols * sn + 8, cx);
          const float2 u[2] = {u0, u1};
          const float2 q0v = make_float2(q0, q0), q1v = make_float2(q1, q1), fv = make_float2(ft, ft);
          float2 Rt[2], Rb[2];
          uint32_t da[4];  // bf16 D: the A operand of the chain, and of dk
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            Rt[nt] = __ffma2_rn(q0v, u[nt], Ct[nt]);  // R = C + q u^T
            Rb[nt] = __ffma2_rn(q1v, u[nt], Cb[nt]);
            const float2 Dt = __fmul2_rn(Rt[nt], f16x2_to_float2(Gp[2 * nt]));  // D = R (1-f)(1-Z^2)
            const float2 Db = __fmul2_rn(Rb[nt], f16x2_to_float2(Gp[2 * nt + 1]));
            da[2 * nt] = pack2_bf16(Dt.x, Dt.y);
            da[2 * nt + 1] = pack2_bf16(Db.x, Db.y);
            const float2 ft2 = __fmul2_rn(fv, Rt[nt]), fb2 = __fmul2_rn(fv, Rb[nt]);
            acc[nt][0] = ft2.x;
            acc[nt][1] = ft2.y;
            acc[nt][2] = fb2.x;
            acc[nt][3] = fb2.y;
          }
          // Chain: C_{t-1} = f R + D W^T (the bf16 D block of the warp's rows is the A operand).
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(acc[nt], da, bt[nt][0], bt[nt][1]);
          // D transposed by 8 x 8 blocks: the B operand of dW and dv (contraction over the rows).
          uint32_t dT[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) dT[i] = movmatrix_trans(da[i]);
          // dW += H_{t-1}^T D (A = H_{t-1}^T from the cache).
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(dWacc[nt], ha, dT[2 * nt], dT[2 * nt + 1]);
          // dv share of the warp's rows: k^T D (A = k of the rows in row 0), and
          // dk = D v (B = v in column 0; rows g, g + 8 in the lanes with qd == 0),
          // both from the bf16 D block with fp32 accumulation.
          const uint32_t ak[4] = {row0 ? kp0 : 0u, 0u, row0 ? kp1 : 0u, 0u};
          float dvs[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_bf16_16816_zc(dvs[nt], ak, dT[2 * nt], dT[2 * nt + 1]);
          float dks[4];
          mma_bf16_16816_zc(dks, da, row0 ? vb0 : 0u, row0 ? vb1 : 0u);
          // df share: <R, H_{t-1} - Z> over the thread's elements.
          float2 pe = __fmul2_rn(Rt[0], f16x2_to_float2(Ep[0]));
          pe = __ffma2_rn(Rb[0], f16x2_to_float2(Ep[1]), pe);
          pe = __ffma2_rn(Rt[1], f16x2_to_float2(Ep[2]), pe);
          pe = __ffma2_rn(Rb[1], f16x2_to_float2(Ep[3]), pe);
          st_shared_f32(dfp + static_cast<uint32_t>(s) * p.df_step, pe.x + pe.y);
          // The previous step's dv and dk (their MMAs completed during this step).
          const bool later = s + 1 < L;
          if (row0 && later)
            st_shared_f32x4(dvp + static_cast<uint32_t>(s + 1) * p.dv_step, make_float4(pdv[0], pdv[1], pdv[2], pdv[3]));
          if (qd == 0 && later) {
            dkrow[0] = pdk0;
            dkrow[8] = pdk1;
          }
          dkrow -= dkstep;
          pdv[0] = dvs[0][0]; pdv[1] = dvs[0][1]; pdv[2] = dvs[1][0]; pdv[3] = dvs[1][1];
          pdk0 = dks[0];
          pdk1 = dks[2];
          if constexpr (kClip) {  // per-step clipping of the state gradient
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[nt][e] = fminf(fmaxf(acc[nt][e], -A.clip), A.clip);
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            Ct[nt] = make_float2(acc[nt][0], acc[nt][1]);
            Cb[nt] = make_float2(acc[nt][2], acc[nt][3]);
          }
          q0 = nq0; q1 = nq1; ft = nft; u0 = nu0; u1 = nu1; kp0 = nkp0; kp1 = nkp1; vb0 = nvb0; vb1 = nvb1;
        }
#undef MV_PIPE_LOAD_OPS
        if (row0) st_shared_f32x4(dvp, make_float4(pdv[0], pdv[1], pdv[2], pdv[3]));  // step 0
        if (qd == 0) {
          dkrow[0] = pdk0;
          dkrow[8] = pdk1;
        }
        // The chunk buffer is read (the last, repeated load included): the
        // rebuild warp may refill it.
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cempty[2 * w + cb]));
      }
      named_bar_sync(1, CT);  // every chain warp's partials of the chunk are written
      if (*cabort) {
        ok = false;
        break;
      }
      // dv and df of the chunk: the row blocks (and for df the lanes) added in a fixed order.
      {
        const int tid = threadIdx.x;  // 0 .. CT - 1
        const uint32_t dvb = smem_u32(smem + p.dvp_off), dfb = smem_u32(smem + p.dfp_off);
        const uint32_t jq = static_cast<uint32_t>((jc & 7) >> 1), jcomp = static_cast<uint32_t>(((jc >> 3) << 1) | (jc & 1));
        for (int i = tid; i < 16 * L; i += CT) {
          const int sl = i >> 4;
          const uint32_t a = dvb + static_cast<uint32_t>(sl) * p.dv_step + jq * 16 + jcomp * 4;
          float x[8];
#pragma unroll
          for (int ww = 0; ww < 8; ++ww) x[ww] = ww < R ? ld_shared_f32(a + ww * 64) : 0.f;
          const float sum = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
          const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + sl) * N + n;
          const float uj = ld_shared_f32(cdy + 4 * (sl * kV + jc));
          A.dv[rowt * kV + jc] = fmaf(wrc, uj, sum);
        }
        // df: four threads per step, thread qq adding the lanes j = qq (mod 4) of
        // every row block, then the four in a fixed order.
        for (int base = 0; base < 4 * L; base += CT) {
          const int i = base + tid, sl = i >> 2, qq = i & 3;
          float f4[4] = {0.f, 0.f, 0.f, 0.f};
          if (sl < L) {
            const uint32_t a = dfb + static_cast<uint32_t>(sl) * p.df_step + qq * 4;
            for (int j = 0; j < 8 * R; j += 4) {
#pragma unroll
              for (int e = 0; e < 4; ++e) f4[e] += ld_shared_f32(a + (j + e) * 16);
            }
          }
          float fz = (f4[0] + f4[1]) + (f4[2] + f4[3]);
          fz += __shfl_xor_sync(0xffffffffu, fz, 1);
          fz += __shfl_xor_sync(0xffffffffu, fz, 2);
          if (sl < L && qq == 0) A.df[(static_cast<int64_t>(b) * T + s0 + sl) * N + n] = fz;
        }
      }
      named_bar_sync(1, CT);  // the partial buffers are free for the next chunk
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sempty[ss]));
    }
    if (ok) {
      // dW partial of this row block: rows m = g (+8), columns 8nt + 2qd (+1).
      float* dwp = A.dW_part + (static_cast<int64_t>(chain) * R + w) * kV * kV;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(dwp + g * kV + 8 * nt + 2 * qd) = make_float2(dWacc[nt][0], dWacc[nt][1]);
        *reinterpret_cast<float2*>(dwp + (g + 8) * kV + 8 * nt + 2 * qd) = make_float2(dWacc[nt][2], dWacc[nt][3]);
      }
      if (A.dH0 != nullptr) {  // C_0, the state gradient left after step 1
        float* dst = A.dH0 + row_g * kV;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) = Ct[nt];
          *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt + 2 * qd) = Cb[nt];
        }
      }
    } else {
      *abort_flag = 1;
    }
  } else if (warp >= rb0 && warp < rb0 + R) {
    // ---------------- rebuild warps: the chunk cache, one chunk ahead ----------------
    const int w = warp - rb0;
    uint32_t bw[2][2];  // B fragments of W (fp16): the forward's step
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
    const int64_t row_g = static_cast<int64_t>(chain) * K + 16 * w + g;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * (w & 3)) << 16) + (w >> 2) * p.set_cols;
    float2 dwl[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // dw_r: columns 8nt + 2qd, +1
    float2 ht[2], hb[2];  // H: rows g, g + 8
    // Start state of chunk c: H_0 (zero if not given) for c == 0, else checkpoint c - 1.
#define MV_PIPE_LOAD_START(c_)                                                                                 \
  {                                                                                                            \
    const float* src = ((c_) == 0) ? (A.H0 ? A.H0 + row_g * kV : nullptr)                                      \
                                   : A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + ((c_) - 1)) * K +     \
                                               16 * w + g) * kV;                                               \
    _Pragma("unroll") for (int nt = 0; nt < 2; ++nt) {                                                         \
      ht[nt] = src ? *reinterpret_cast<const float2*>(src + 8 * nt + 2 * qd) : make_float2(0.f, 0.f);          \
      hb[nt] = src ? *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt + 2 * qd) : make_float2(0.f, 0.f); \
    }                                                                                                          \
  }
    MV_PIPE_LOAD_START(p.nchunks - 1)
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL, L = min(CL, T - s0);
      const int ss = ci % kNS, zs = ci % kNZ, cb = ci & 1;
      if (!mbar_wait(smem_u32(&sfull[ss]), (ci / kNS) & 1, abort_flag, status, kWhereBwdFull)) break;
      if (kZ && !mbar_wait(smem_u32(&zfull[zs]), (ci / kNZ) & 1, abort_flag, status, kWhereBwdZFull)) break;
      if (ci >= 2 && !mbar_wait(smem_u32(&cempty[2 * w + cb]), ((ci >> 1) - 1) & 1, abort_flag, status, kWhereBwdTFree))
        break;
      tc_fence_after_sync();
      const uint8_t* sbuf = smem + p.s_off + ss * p.s_bytes;
      const uint32_t ck = smem_u32(sbuf + p.k_off), cv = smem_u32(sbuf + p.v_off);
      const uint32_t cdy = smem_u32(sbuf + p.dy_off), cf = smem_u32(sbuf + p.f_off);
      const uint32_t cz = smem_u32(smem + p.z_off + zs * p.z_bytes) + (w * 32 + lane) * 16;
      const uint32_t tc = tq + static_cast<uint32_t>(cb * kCacheCols * CL);
      const uint32_t qp = smem_u32(smem + p.qp_off) + static_cast<uint32_t>((w * CL * 32 + lane) * 8);
      // The step's operands, loaded one step ahead.
      float fo, k0 = 0.f, k1 = 0.f;
      uint4 zq = make_uint4(0u, 0u, 0u, 0u);
      float2 u0, u1;
      uint32_t vb0, vb1;
#define MV_PIPE_LOAD_RB(s_, fo_, zq_, k0_, k1_, u0_, u1_, vb0_, vb1_)                      \
  {                                                                                        \
    fo_ = ld_shared_f32(cf + 4 * (s_));                                                    \
    if constexpr (kZ) {                                                                    \
      zq_ = ld_shared_v4(cz + (s_) * R * 512);                                             \
    } else {                                                                               \
      const uint32_t krow = ck + 2 * ((s_) * K + 16 * w + g);                              \
      k0_ = bf16_bits_to_f32(ld_shared_u16(krow));                                         \
      k1_ = bf16_bits_to_f32(ld_shared_u16(krow + 16));                                    \
    }                                                                                      \
    u0_ = ld_shared_f32x2(cdy + 4 * ((s_) * kV + 2 * qd));                                 \
    u1_ = ld_shared_f32x2(cdy + 4 * ((s_) * kV + 8 + 2 * qd));                             \
    vb0_ = ld_shared_b32(cv + 2 * ((s_) * kV + 2 * qd));                                   \
    vb1_ = ld_shared_b32(cv + 2 * ((s_) * kV + 8 + 2 * qd));                               \
  }
      MV_PIPE_LOAD_RB(0, fo, zq, k0, k1, u0, u1, vb0, vb1)
#pragma unroll 2
      for (int s = 0; s < L; ++s) {
        const int sn = s + 1 < L ? s + 1 : s;  // the last step reloads itself (no branch in the loop)
        float nfo, nk0 = 0.f, nk1 = 0.f;
        uint4 nzq = make_uint4(0u, 0u, 0u, 0u);
        float2 nu0, nu1;
        uint32_t nvb0, nvb1;
        MV_PIPE_LOAD_RB(sn, nfo, nzq, nk0, nk1, nu0, nu1, nvb0, nvb1)
        const float omf = 1.f - fo;
        const float2 vv[2] = {make_float2(bf16lo(vb0), bf16hi(vb0)), make_float2(bf16lo(vb1), bf16hi(vb1))};
        const float2 u[2] = {u0, u1};
        float2 zt[2], zb[2];  // Z_s: rows g, g + 8
        if constexpr (kZ) {
          zt[0] = f16x2_to_float2(zq.x);
          zb[0] = f16x2_to_float2(zq.y);
          zt[1] = f16x2_to_float2(zq.z);
          zb[1] = f16x2_to_float2(zq.w);
        } else {
          uint32_t a[4];  // fp16 H_{s-1}, as in the forward
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            a[2 * nt] = pack2_f16(ht[nt].x, ht[nt].y);
            a[2 * nt + 1] = pack2_f16(hb[nt].x, hb[nt].y);
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            float acc[4] = {k0 * vv[nt].x, k0 * vv[nt].y, k1 * vv[nt].x, k1 * vv[nt].y};
            mma_f16_16816(acc, a, bw[nt][0], bw[nt][1]);
            zt[nt] = make_float2(tanh_fast(acc[0]), tanh_fast(acc[1]));
            zb[nt] = make_float2(tanh_fast(acc[2]), tanh_fast(acc[3]));
          }
        }
        uint32_t c8[8], c4[4];
        const float2 om2 = make_float2(omf, omf), nom2 = make_float2(-omf, -omf);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          // G = (1-f)(1 - Z^2), E = H_{s-1} - Z.
          const float2 gt = __ffma2_rn(nom2, __fmul2_rn(zt[nt], zt[nt]), om2);
          const float2 gb = __ffma2_rn(nom2, __fmul2_rn(zb[nt], zb[nt]), om2);
          c8[2 * nt] = pack2_f16(gt.x, gt.y);
          c8[2 * nt + 1] = pack2_f16(gb.x, gb.y);
          const float2 et = __fadd2_rn(ht[nt], make_float2(-zt[nt].x, -zt[nt].y));
          const float2 eb = __fadd2_rn(hb[nt], make_float2(-zb[nt].x, -zb[nt].y));
          c8[4 + 2 * nt] = pack2_f16(et.x, et.y);
          c8[4 + 2 * nt + 1] = pack2_f16(eb.x, eb.y);
        }
        // H_{s-1}^T as the A operand of dW += H_{s-1}^T D (8 x 8 blocks transposed).
        c4[0] = movmatrix_trans(pack2_bf16(ht[0].x, ht[0].y));
        c4[1] = movmatrix_trans(pack2_bf16(ht[1].x, ht[1].y));
        c4[2] = movmatrix_trans(pack2_bf16(hb[0].x, hb[0].y));
        c4[3] = movmatrix_trans(pack2_bf16(hb[1].x, hb[1].y));
        tmem_st_32x32b_x8(tc + kCacheCols * s, c8);
        tmem_st_32x32b_x4(tc + kCacheCols * s + 8, c4);
        // H_s = H_{s-1} + (1-f)(Z_s - H_{s-1}) (Eq. 11).
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          ht[nt] = __ffma2_rn(om2, __fadd2_rn(zt[nt], make_float2(-ht[nt].x, -ht[nt].y)), ht[nt]);
          hb[nt] = __ffma2_rn(om2, __fadd2_rn(zb[nt], make_float2(-hb[nt].x, -hb[nt].y)), hb[nt]);
        }
        // dq_s = H_s u_s: this thread's share of rows g, g + 8 (the four lanes of a
        // row are added at the end of the chunk).
        const float2 qt = __ffma2_rn(ht[1], u[1], __fmul2_rn(ht[0], u[0]));
        const float2 qb = __ffma2_rn(hb[1], u[1], __fmul2_rn(hb[0], u[0]));
        st_shared_f32x2(qp + s * 256, make_float2(qt.x + qt.y, qb.x + qb.y));
        // dw_r += u_s v_s (columns 8nt + 2qd, +1; the same in every lane of a column).
        dwl[0] = __ffma2_rn(u[0], vv[0], dwl[0]);
        dwl[1] = __ffma2_rn(u[1], vv[1], dwl[1]);
        fo = nfo; zq = nzq; k0 = nk0; k1 = nk1; u0 = nu0; u1 = nu1; vb0 = nvb0; vb1 = nvb1;
      }
#undef MV_PIPE_LOAD_RB
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&cfull[2 * w + cb]));
        if constexpr (kZ) mbar_arrive(smem_u32(&zempty[zs]));
      }
      // dq of the chunk: the four lanes of each row added in a fixed order.
      for (int i = lane; i < L * 8; i += 32) {
        const int sl = i >> 3, gg = i & 7;
        const uint32_t a = smem_u32(smem + p.qp_off) + static_cast<uint32_t>(((w * CL + sl) * 32 + 4 * gg) * 8);
        const float4 x0 = ld_shared_f32x4(a), x1 = ld_shared_f32x4(a + 16);
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + sl) * N + n;
        A.dq[rowt * K + 16 * w + gg] = (x0.x + x0.z) + (x1.x + x1.z);
        A.dq[rowt * K + 16 * w + gg + 8] = (x0.y + x0.w) + (x1.y + x1.w);
      }
      __syncwarp();  // the partials are read before the next chunk rewrites them
      if (ci + 1 < p.nchunks) MV_PIPE_LOAD_START(c - 1)  // in flight while the next waits run
    }
#undef MV_PIPE_LOAD_START
    if (w == 0 && g == 0 && !*abort_flag) {
      float* dst = A.dwr_part + static_cast<int64_t>(chain) * kV + 2 * qd;
      *reinterpret_cast<float2*>(dst) = dwl[0];
      *reinterpret_cast<float2*>(dst + 8) = dwl[1];
    }
  } else if (warp == prod) {
    // ---------------- producer: chunk inputs, last chunk first ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_dy);
    }
    const GateSrc gs{A.f, A.gate_a, A.gate_alpha, A.gate_beta, true};
    int s_issued = 0, z_issued = 0;  // chunks whose input / Z copies were issued
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int t0 = c * CL, L = min(CL, T - t0);
      const int ss = ci % kNS, zs = ci % kNZ;
      if (ci >= kNS &&
          !mbar_wait(smem_u32(&sempty[ss]), ((ci / kNS) - 1) & 1, abort_flag, status, kWhereBwdCEmpty))
        break;
      uint8_t* sbuf = smem + p.s_off + ss * p.s_bytes;
      const int t = t0 + lane;
      if (lane < CL)
        reinterpret_cast<float*>(sbuf + p.f_off)[lane] =
            (t < T) ? gate_value(gs, (static_cast<int64_t>(b) * T + t) * N + n, n) : 0.f;
      __syncwarp();
      const uint32_t fb = smem_u32(&sfull[ss]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, p.tx_bytes);
        tma_load_4d(smem_u32(sbuf + p.q_off), &tm_q, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(sbuf + p.k_off), &tm_k, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(sbuf + p.v_off), &tm_v, fb, 0, n, t0, b);
        tma_load_4d(smem_u32(sbuf + p.dy_off), &tm_dy, fb, 0, n, t0, b);
      } else {
        mbar_arrive(fb);
      }
      s_issued = ci + 1;
      if constexpr (kZ) {
        if (ci >= kNZ &&
            !mbar_wait(smem_u32(&zempty[zs]), ((ci / kNZ) - 1) & 1, abort_flag, status, kWhereBwdXEmpty))
          break;
        if (lane == 0) {
          const uint32_t zbytes = static_cast<uint32_t>(L * R * 512);
          const uint32_t zb = smem_u32(&zfull[zs]);
          mbar_arrive_expect_tx(zb, zbytes);
          bulk_load(smem_u32(smem + p.z_off + zs * p.z_bytes),
                    reinterpret_cast<const uint8_t*>(A.zstash) + (static_cast<int64_t>(chain) * T + t0) * R * 512,
                    zbytes, zb);
        }
        z_issued = ci + 1;
      }
    }
    if (*abort_flag) {
      // Let every copy that was issued land before the CTA exits.
      for (int ci = std::max(0, s_issued - kNS); ci < s_issued; ++ci)
        mbar_wait_timed(smem_u32(&sfull[ci % kNS]), (ci / kNS) & 1, nullptr, kWhereBwdDrain);
      for (int ci = std::max(0, z_issued - kNZ); ci < z_issued; ++ci)
        mbar_wait_timed(smem_u32(&zfull[ci % kNZ]), (ci / kNZ) & 1, nullptr, kWhereBwdDrain);
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

template <bool kClip, bool kZ>
cudaError_t launch_t(const PipeParams& p, uint32_t smem, bool wide, cudaStream_t stream, const CUtensorMap& mq,
                     const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdy) {
  auto kernel = wide ? mv_backward_pipe_kernel<kClip, kZ, true> : mv_backward_pipe_kernel<kClip, kZ, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<p.a.B * p.a.N, (8 * p.nq + 1) * 32, smem, stream>>>(p, mq, mk, mv, mdy);
  return cudaGetLastError();
}

}  // namespace

bool mv_backward_pipe_supported(int K, int V, int ckpt_every) {
  if (V != kV || K % kRows != 0 || K < kRows || K > 8 * kRows) return false;
  return ckpt_every >= 1 && ckpt_every <= pipe_max_chunk(K / kRows);
}

cudaError_t launch_mv_backward_pipe(const BwdArgs& a, cudaStream_t stream) {
  if (!mv_backward_pipe_supported(a.K, a.V, a.ckpt_every)) return cudaErrorInvalidValue;
  PipeParams p{};
  p.a = a;
  p.R = a.K / kRows;
  p.nq = (p.R + 3) / 4;
  const int C = a.ckpt_every;
  p.nchunks = (a.T + C - 1) / C;
  p.set_cols = 2u * kCacheCols * C;
  p.q_off = 0;
  p.k_off = align_up(C * a.K * 2, 128);
  p.v_off = p.k_off + align_up(C * a.K * 2, 128);
  p.dy_off = p.v_off + align_up(C * kV * 2, 128);
  p.f_off = p.dy_off + align_up(C * kV * 4, 128);
  p.s_bytes = align_up(p.f_off + C * 4, 128);
  p.s_off = 0;
  p.z_bytes = a.zstash != nullptr ? align_up(C * p.R * 512, 128) : 0u;
  p.z_off = p.s_off + kNS * p.s_bytes;
  // dv partials: [step][row block][4 lanes] x 16 bytes, the step stride padded
  // by 64 bytes (two steps read by one warp land on distinct banks); df
  // partials: [step][row block][32 lanes] x 4 bytes, the step stride padded by
  // 16 bytes (the end-of-chunk sum reads eight steps at once on distinct banks).
  p.dvp_off = p.z_off + kNZ * p.z_bytes;
  p.dv_step = static_cast<uint32_t>(p.R * 64 + 64);
  p.dfp_off = p.dvp_off + align_up(static_cast<uint32_t>(C) * p.dv_step, 128);
  p.df_step = static_cast<uint32_t>(p.R * 128 + 16);
  p.qp_off = p.dfp_off + align_up(static_cast<uint32_t>(C) * p.df_step, 128);
  p.bar_off = p.qp_off + static_cast<uint32_t>(C * p.R * 256);
  p.misc_off = p.bar_off + (2 * kNS + 2 * kNZ + 32) * 8;
  const uint32_t smem = align_up(p.misc_off + 16, 128);
  p.tx_bytes = 2 * C * a.K * 2 + C * kV * 2 + C * kV * 4;
  if (smem > 227u * 1024u) return cudaErrorInvalidValue;

  CUtensorMap mq, mk, mv, mdy;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, a.K, a.K, C) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, a.K, C) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, C) ||
      !make_tensor_map_btnx(&mdy, a.dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.N, kV, kV, C))
    return cudaErrorInvalidValue;
  const bool wide = p.nq > 1;
  if (a.zstash != nullptr)
    return a.clip > 0.f ? launch_t<true, true>(p, smem, wide, stream, mq, mk, mv, mdy)
                        : launch_t<false, true>(p, smem, wide, stream, mq, mk, mv, mdy);
  return a.clip > 0.f ? launch_t<true, false>(p, smem, wide, stream, mq, mk, mv, mdy)
                      : launch_t<false, false>(p, smem, wide, stream, mq, mk, mv, mdy);
}

}  // namespace m2rnn
