// Register-resident backward-through-time for small value heads, V = 16
// (bf16 inputs, fp32 state and gradients): the multi-value configuration of
// "M2RNN: Non-Linear RNNs with Matrix-Valued States for Scalable Language
// Modeling" (reading notes section 2.4), with the chain rule of section 2.7
// (value-residual terms restored); u_t = dy_t, C_T = dH_T:
//   R_t = C_t + q_t u_t^T,  D_t = ((1-f_t) R_t) * (1 - Z_t * Z_t),
//   C_{t-1} = f_t R_t + D_t W^T,
//   dq_t = H_t u_t, dk_t = D_t v_t, dv_t = D_t^T k_t + w_r * u_t,
//   df_t = <R_t, H_{t-1} - Z_t>,  dW += H_{t-1}^T D_t,  dw_r += u_t * v_t.
//
// One CTA per (b, n) head; compute warp w owns key rows 16w..16w+15 and all
// 16 value columns, so both serial chains stay inside the warp: the warp's
// bf16 16 x 16 blocks of H (forward rerun) and of D (C_{t-1} = f R + D W^T)
// are the A operands of its own m16n8k16 MMAs.  Chunks of C <= 32 steps run
// last first: the warp reruns its rows from the chunk's checkpoint, caching
// Z_t and H_{t-1} (fp32) in its own TMEM lanes, then walks the chunk back.
// dq_t and dk_t are row sums inside the warp; dv_t and df_t sum over rows:
// per-warp partials per step, added over the row blocks in a fixed order at
// the end of the chunk.  dW accumulates per warp in registers (H_{t-1}^T and
// D transposed with movmatrix) and leaves as one partial per row block.  A
// producer warp streams the chunk's q, k, v, dy by TMA (f by plain loads).
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
constexpr int kMaxRB = 8;       // K <= 128
constexpr int kMaxChunkMv = 32;  // one chunk cache: 16 TMEM columns per step
constexpr int kCBufs = 2;

struct MvBwdParams {
  BwdArgs a;
  int R, nchunks;
  uint32_t colset;  // TMEM column offset of warps 4..7 (they share lane quadrants with 0..3)
  uint32_t cbuf_off, cbuf_bytes, cq_off, ck_off, cv_off, cdy_off, cf_off, cz_off, part_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

// kClip: the state-gradient clamp as a compile-time switch (no per-step
// branch).  kZ: Z_t comes from the forward's stash (copied with the chunk's
// inputs), so the chunk rebuild is the gate blend alone.
template <bool kClip, bool kZ>
__global__ void __launch_bounds__((kMaxRB + 1) * 32, 1)
    mv_backward_kernel(const __grid_constant__ MvBwdParams p, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_dy) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const BwdArgs& A = p.a;
  const int R = p.R, T = A.T, N = A.N, K = A.K, CL = A.ckpt_every;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  StatusBlock* status = A.status;
  uint64_t* cfull = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* cempty = cfull + kCBufs;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* cabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 8);
  float* part_dv = reinterpret_cast<float*>(smem + p.part_off);  // [C][R][kV]
  float* part_df = part_dv + kMaxChunkMv * R * kV;                // [C][R]
  if (threadIdx.x == 0) {
    for (int i = 0; i < kCBufs; ++i) {
      mbar_init(smem_u32(&cfull[i]), 32);  // producer lanes (+ TMA bytes)
      mbar_init(smem_u32(&cempty[i]), R);  // one arrival per compute warp
    }
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

  if (warp < R) {
    // ---------------- compute warps ----------------
    const int g = lane >> 2, qd = lane & 3, w = warp;
    const int CT = 32 * R;
    const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
    uint32_t bw[2][2], bt[2][2];  // B fragments of W (rerun, fp16) and of W^T (C_{t-1} = f R + D W^T, bf16)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = 8 * nt + g;
      bw[nt][0] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[(2 * qd) * kV + col]) |
                                  (static_cast<uint32_t>(Wg[(2 * qd + 1) * kV + col]) << 16));
      bw[nt][1] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[(2 * qd + 8) * kV + col]) |
                                  (static_cast<uint32_t>(Wg[(2 * qd + 9) * kV + col]) << 16));
      if (!f16x2_finite(bw[nt][0]) || !f16x2_finite(bw[nt][1]))
        report_device_error(status, kStatusCheck, kWhereWRange);
      bt[nt][0] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + 2 * qd);
      bt[nt][1] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + 2 * qd + 8);
    }
    const int64_t row_g = static_cast<int64_t>(chain) * K + 16 * w + g;  // state row of lane g
    float Cg[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (A.dH_T != nullptr) {
        const float2 x0 = *reinterpret_cast<const float2*>(A.dH_T + row_g * kV + 8 * nt + 2 * qd);
        const float2 x1 = *reinterpret_cast<const float2*>(A.dH_T + (row_g + 8) * kV + 8 * nt + 2 * qd);
        Cg[nt][0] = x0.x; Cg[nt][1] = x0.y; Cg[nt][2] = x1.x; Cg[nt][3] = x1.y;
      } else {
        Cg[nt][0] = Cg[nt][1] = Cg[nt][2] = Cg[nt][3] = 0.f;
      }
    }
    float dWacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float dwr[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // warp 0, g == 0: columns 8nt + 2qd (+1)
    const uint32_t tcache = tmem_base + (static_cast<uint32_t>(32 * (w & 3)) << 16) + (w >> 2) * p.colset;
    const uint16_t* wrg = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    bool ok = true;
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL;
      const int L = min(CL, T - s0);
      const int cb = ci % kCBufs;
      const bool mine = mbar_wait_timed(smem_u32(&cfull[cb]), (ci / kCBufs) & 1, status, kWhereBwdFull);
      if (!mine) *cabort = 1;
      named_bar_sync(1, CT);
      if (*cabort) {
        ok = false;
        break;
      }
      const uint8_t* cbuf = smem + p.cbuf_off + cb * p.cbuf_bytes;
      const uint16_t* cq = reinterpret_cast<const uint16_t*>(cbuf + p.cq_off);
      const uint16_t* ck = reinterpret_cast<const uint16_t*>(cbuf + p.ck_off);
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(cbuf + p.cv_off);
      const float* cdy = reinterpret_cast<const float*>(cbuf + p.cdy_off);
      const float* cf = reinterpret_cast<const float*>(cbuf + p.cf_off);
      const uint32_t cz = smem_u32(cbuf + p.cz_off) + (w * 32 + lane) * 16;  // this thread's stashed Z, step 0
      // ---- rerun the chunk from its start state (Eq. 10-11), caching Z_s and H_{s-1} ----
      float h[2][4];
      {
        // Chunk 0 starts from H_0 (zero if not given), chunk c from checkpoint c - 1.
        const float* src =
            (c == 0) ? (A.H0 ? A.H0 + row_g * kV : nullptr)
                     : A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (c - 1)) * K + 16 * w + g) * kV;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if (src != nullptr) {
            const float2 x0 = *reinterpret_cast<const float2*>(src + 8 * nt + 2 * qd);
            const float2 x1 = *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt + 2 * qd);
            h[nt][0] = x0.x; h[nt][1] = x0.y; h[nt][2] = x1.x; h[nt][3] = x1.y;
          } else {
            h[nt][0] = h[nt][1] = h[nt][2] = h[nt][3] = 0.f;
          }
        }
      }
      if constexpr (kZ) {
        for (int s = 0; s < L; ++s) {
          const float omf = 1.f - cf[s];
          const uint4 zq = ld_shared_v4(cz + s * R * 512);
          const float z[2][4] = {{f16lo(zq.x), f16hi(zq.x), f16lo(zq.y), f16hi(zq.y)},
                                 {f16lo(zq.z), f16hi(zq.z), f16lo(zq.w), f16hi(zq.w)}};
          uint32_t cache[16];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              cache[4 * nt + e] = __float_as_uint(z[nt][e]);
              cache[8 + 4 * nt + e] = __float_as_uint(h[nt][e]);  // H_{s-1}
              h[nt][e] = fmaf(omf, z[nt][e] - h[nt][e], h[nt][e]);
            }
          tmem_st_32x32b_x16(tcache + 16 * s, cache);
        }
      } else {
      for (int s = 0; s < L; ++s) {
        uint32_t a[4];  // fp16 H_{s-1}, as in the forward
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          a[2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
          a[2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
        }
        const float k0 = bf16_bits_to_f32(ck[s * K + 16 * w + g]);
        const float k1 = bf16_bits_to_f32(ck[s * K + 16 * w + g + 8]);
        const float omf = 1.f - cf[s];
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint32_t vv = *reinterpret_cast<const uint32_t*>(cv + s * kV + 8 * nt + 2 * qd);
          acc[nt][0] = k0 * bf16lo(vv);
          acc[nt][1] = k0 * bf16hi(vv);
          acc[nt][2] = k1 * bf16lo(vv);
          acc[nt][3] = k1 * bf16hi(vv);
          mma_f16_16816(acc[nt], a, bw[nt][0], bw[nt][1]);
        }
        uint32_t cache[16];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float z = tanh_fast(acc[nt][e]);
            cache[4 * nt + e] = __float_as_uint(z);
            cache[8 + 4 * nt + e] = __float_as_uint(h[nt][e]);  // H_{s-1}
            h[nt][e] = fmaf(omf, z - h[nt][e], h[nt][e]);
          }
        tmem_st_32x32b_x16(tcache + 16 * s, cache);
      }
      }
      tmem_st_wait();
      // ---- reverse walk: h = H_t of the chunk's last step ----
      uint32_t slot[16];
      tmem_ld_32x32b<16>(tcache + 16 * (L - 1), slot);
      for (int s = L - 1; s >= 0; --s) {
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
        const float q0 = bf16_bits_to_f32(cq[s * K + 16 * w + g]);
        const float q1 = bf16_bits_to_f32(cq[s * K + 16 * w + g + 8]);
        const float k0 = bf16_bits_to_f32(ck[s * K + 16 * w + g]);
        const float k1 = bf16_bits_to_f32(ck[s * K + 16 * w + g + 8]);
        const float ft = cf[s], omf = 1.f - ft;
        float u[2][2], vv[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 uu = *reinterpret_cast<const float2*>(cdy + s * kV + 8 * nt + 2 * qd);
          u[nt][0] = uu.x;
          u[nt][1] = uu.y;
          const uint32_t vb = *reinterpret_cast<const uint32_t*>(cv + s * kV + 8 * nt + 2 * qd);
          vv[nt][0] = bf16lo(vb);
          vv[nt][1] = bf16hi(vb);
        }
        tmem_ld_wait();
        tmem_ld_fence_regs(slot);
        float Z[2][4], Hp[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            Z[nt][e] = __uint_as_float(slot[4 * nt + e]);
            Hp[nt][e] = __uint_as_float(slot[8 + 4 * nt + e]);
          }
        if (s > 0) tmem_ld_32x32b<16>(tcache + 16 * (s - 1), slot);
        float Rv[2][4], Dv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            Rv[nt][e] = fmaf(e < 2 ? q0 : q1, u[nt][e & 1], Cg[nt][e]);
            Dv[nt][e] = omf * Rv[nt][e] * fmaf(-Z[nt][e], Z[nt][e], 1.f);
          }
        // Chain: C_{t-1} = f R + D W^T (bf16(D) of the warp's rows is its own A operand).
        uint32_t da[4];
        da[0] = pack2_bf16(Dv[0][0], Dv[0][1]);
        da[1] = pack2_bf16(Dv[0][2], Dv[0][3]);
        da[2] = pack2_bf16(Dv[1][0], Dv[1][1]);
        da[3] = pack2_bf16(Dv[1][2], Dv[1][3]);
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = ft * Rv[nt][e];
          mma_bf16_16816(acc[nt], da, bt[nt][0], bt[nt][1]);
        }
        // dW += H_{t-1}^T D: A = H_{t-1}^T, B = D (both transposed 8 x 8 blocks).
        {
          uint32_t ha[4];
          ha[0] = movmatrix_trans(pack2_bf16(Hp[0][0], Hp[0][1]));
          ha[1] = movmatrix_trans(pack2_bf16(Hp[1][0], Hp[1][1]));
          ha[2] = movmatrix_trans(pack2_bf16(Hp[0][2], Hp[0][3]));
          ha[3] = movmatrix_trans(pack2_bf16(Hp[1][2], Hp[1][3]));
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_bf16_16816(dWacc[nt], ha, movmatrix_trans(da[2 * nt]), movmatrix_trans(da[2 * nt + 1]));
        }
        // Row sums inside the warp: dq = H_t u, dk = D v (rows g, g+8; fixed tree over qd).
        float pq0 = 0.f, pq1 = 0.f, pk0 = 0.f, pk1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pq0 = fmaf(h[nt][e], u[nt][e], pq0);
            pq1 = fmaf(h[nt][e + 2], u[nt][e], pq1);
            pk0 = fmaf(Dv[nt][e], vv[nt][e], pk0);
            pk1 = fmaf(Dv[nt][e + 2], vv[nt][e], pk1);
          }
        // Column sums over the warp's rows: dv partial = D^T k; df partial.
        float pv[4], pf = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pv[2 * nt] = fmaf(Dv[nt][0], k0, Dv[nt][2] * k1);
          pv[2 * nt + 1] = fmaf(Dv[nt][1], k0, Dv[nt][3] * k1);
#pragma unroll
          for (int e = 0; e < 4; ++e) pf = fmaf(Rv[nt][e], Hp[nt][e] - Z[nt][e], pf);
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
          pq0 += __shfl_xor_sync(0xffffffffu, pq0, o);
          pq1 += __shfl_xor_sync(0xffffffffu, pq1, o);
          pk0 += __shfl_xor_sync(0xffffffffu, pk0, o);
          pk1 += __shfl_xor_sync(0xffffffffu, pk1, o);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1)
#pragma unroll
          for (int i = 0; i < 4; ++i) pv[i] += __shfl_xor_sync(0xffffffffu, pv[i], o);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) pf += __shfl_xor_sync(0xffffffffu, pf, o);
        if (qd == 0) {
          A.dq[rowt * K + 16 * w + g] = pq0;
          A.dq[rowt * K + 16 * w + g + 8] = pq1;
          A.dk[rowt * K + 16 * w + g] = pk0;
          A.dk[rowt * K + 16 * w + g + 8] = pk1;
        }
        if (g == 0) {
          float* dst = part_dv + (s * R + w) * kV + 2 * qd;
          *reinterpret_cast<float2*>(dst) = make_float2(pv[0], pv[1]);
          *reinterpret_cast<float2*>(dst + 8) = make_float2(pv[2], pv[3]);
          if (w == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              dwr[nt][0] = fmaf(u[nt][0], vv[nt][0], dwr[nt][0]);
              dwr[nt][1] = fmaf(u[nt][1], vv[nt][1], dwr[nt][1]);
            }
          }
        }
        if (lane == 0) part_df[s * R + w] = pf;
        if constexpr (kClip) {  // per-step clipping of the state gradient
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = fminf(fmaxf(acc[nt][e], -A.clip), A.clip);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            Cg[nt][e] = acc[nt][e];
            h[nt][e] = Hp[nt][e];
          }
      }
      // dv_t, df_t of the chunk: the row blocks summed in a fixed order.
      named_bar_sync(1, CT);
      for (int idx = threadIdx.x; idx < L * (kV + 1); idx += CT) {
        const int s = idx / (kV + 1), j = idx % (kV + 1);
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
        float sum = 0.f;
        if (j < kV) {
          for (int ww = 0; ww < R; ++ww) sum += part_dv[(s * R + ww) * kV + j];
          A.dv[rowt * kV + j] = fmaf(bf16_bits_to_f32(wrg[j]), cdy[s * kV + j], sum);
        } else {
          for (int ww = 0; ww < R; ++ww) sum += part_df[s * R + ww];
          A.df[rowt] = sum;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&cempty[cb]));
      named_bar_sync(1, CT);  // the partial buffers are free for the next chunk
    }
    if (ok) {
      // dW partial of this row block: rows m = g (+8), columns 8nt + 2qd (+1).
      float* dwp = A.dW_part + (static_cast<int64_t>(chain) * R + w) * kV * kV;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(dwp + g * kV + 8 * nt + 2 * qd) = make_float2(dWacc[nt][0], dWacc[nt][1]);
        *reinterpret_cast<float2*>(dwp + (g + 8) * kV + 8 * nt + 2 * qd) = make_float2(dWacc[nt][2], dWacc[nt][3]);
      }
      if (w == 0 && g == 0) {
        float* dst = A.dwr_part + static_cast<int64_t>(chain) * kV + 2 * qd;
        *reinterpret_cast<float2*>(dst) = make_float2(dwr[0][0], dwr[0][1]);
        *reinterpret_cast<float2*>(dst + 8) = make_float2(dwr[1][0], dwr[1][1]);
      }
      if (A.dH0 != nullptr) {  // C_0, the state gradient left after step 1
        float* dst = A.dH0 + row_g * kV;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd) = make_float2(Cg[nt][0], Cg[nt][1]);
          *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt + 2 * qd) = make_float2(Cg[nt][2], Cg[nt][3]);
        }
      }
    } else {
      *abort_flag = 1;
    }
  } else if (warp == R) {
    // ---------------- TMA producer (chunks, last first) ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_dy);
    }
    const GateSrc gs{A.f, A.gate_a, A.gate_alpha, A.gate_beta, true};
    int issued = 0;
    bool ok = true;
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int cb = ci % kCBufs;
      if (ci >= kCBufs &&
          !mbar_wait(smem_u32(&cempty[cb]), ((ci / kCBufs) - 1) & 1, abort_flag, status, kWhereBwdCEmpty)) {
        ok = false;
        break;
      }
      const int t0 = c * CL;
      uint8_t* buf = smem + p.cbuf_off + cb * p.cbuf_bytes;
      const int t = t0 + lane;
      if (lane < CL)
        reinterpret_cast<float*>(buf + p.cf_off)[lane] =
            (t < T) ? gate_value(gs, (static_cast<int64_t>(b) * T + t) * N + n, n) : 0.f;
      __syncwarp();
      const uint32_t fb = smem_u32(&cfull[cb]);
      if (lane == 0) {
        const uint32_t zbytes = kZ ? static_cast<uint32_t>(min(CL, T - t0) * R * 512) : 0u;
        mbar_arrive_expect_tx(fb, p.tx_bytes + zbytes);
        if constexpr (kZ)  // the chunk's stashed Z: one contiguous range
          bulk_load(smem_u32(buf + p.cz_off),
                    reinterpret_cast<const uint8_t*>(A.zstash) + (static_cast<int64_t>(chain) * T + t0) * R * 512,
                    zbytes, fb);
        tma_load_4d(smem_u32(buf + p.cq_off), &tm_q, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.ck_off), &tm_k, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.cv_off), &tm_v, fb, 0, n, t0, b);
        tma_load_4d(smem_u32(buf + p.cdy_off), &tm_dy, fb, 0, n, t0, b);
      } else {
        mbar_arrive(fb);
      }
      issued = ci + 1;
    }
    if (!ok) {
      for (int ci = std::max(0, issued - kCBufs); ci < issued; ++ci)
        mbar_wait_timed(smem_u32(&cfull[ci % kCBufs]), (ci / kCBufs) & 1, nullptr, kWhereBwdDrain);
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

}  // namespace

bool mv_backward_supported(int K, int V, int ckpt_every) {
  if (V != kV || K % kRows != 0 || K < kRows || K > kRows * kMaxRB) return false;
  const int sets = (K / kRows > 4) ? 2 : 1;  // warps 4..7 share lane quadrants with 0..3
  return ckpt_every >= 1 && sets * 16 * ckpt_every <= 512;
}

cudaError_t launch_mv_backward(const BwdArgs& a, cudaStream_t stream) {
  if (!mv_backward_supported(a.K, a.V, a.ckpt_every)) return cudaErrorInvalidValue;
  if (mv_backward_pipe_supported(a.K, a.V, a.ckpt_every)) return launch_mv_backward_pipe(a, stream);
  MvBwdParams p{};
  p.a = a;
  p.R = a.K / kRows;
  const int C = a.ckpt_every;
  p.nchunks = (a.T + C - 1) / C;
  p.colset = 16u * C;
  p.cbuf_off = 0;
  p.cq_off = 0;
  p.ck_off = align_up(C * a.K * 2, 128);
  p.cv_off = p.ck_off + align_up(C * a.K * 2, 128);
  p.cdy_off = p.cv_off + align_up(C * kV * 2, 128);
  p.cf_off = p.cdy_off + align_up(C * kV * 4, 128);
  p.cz_off = align_up(p.cf_off + kMaxChunkMv * 4, 128);
  p.cbuf_bytes = align_up(p.cz_off + (a.zstash != nullptr ? C * p.R * 512 : 0), 128);
  p.part_off = kCBufs * p.cbuf_bytes;
  p.bar_off = p.part_off + align_up(kMaxChunkMv * p.R * (kV + 1) * 4, 128);
  p.misc_off = p.bar_off + 2 * kCBufs * 8;
  const uint32_t smem = align_up(p.misc_off + 16, 128);
  p.tx_bytes = 2 * C * a.K * 2 + C * kV * 2 + C * kV * 4;

  CUtensorMap mq, mk, mv, mdy;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, a.K, a.K, C) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, a.K, C) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, C) ||
      !make_tensor_map_btnx(&mdy, a.dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.N, kV, kV, C))
    return cudaErrorInvalidValue;
  auto kernel = a.zstash != nullptr ? (a.clip > 0.f ? mv_backward_kernel<true, true> : mv_backward_kernel<false, true>)
                                    : (a.clip > 0.f ? mv_backward_kernel<true, false> : mv_backward_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<a.B * a.N, (p.R + 1) * 32, smem, stream>>>(p, mq, mk, mv, mdy);
  return cudaGetLastError();
}

}  // namespace m2rnn
