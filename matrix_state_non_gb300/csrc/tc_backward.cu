// Tensor-core backward scan for V = 128 value columns (bf16 inputs, fp32
// state and gradients).
//
// Recurrence (reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued
// States for Scalable Language Modeling", section 2.1, Eq. 10-12) and its
// chain rule (section 2.7): with u_t = dy_t, C_T = dH_T,
//   R_t = C_t + q_t u_t^T,  D_t = (1 - f_t) R_t (1 - Z_t^2),
//   C_{t-1} = f_t R_t + D_t W^T,
//   dq_t = H_t u_t, dk_t = D_t v_t, dv_t = D_t^T k_t + w_r u_t,
//   df_t = <R_t, H_{t-1} - Z_t>, dW = sum_t H_{t-1}^T D_t, dw_r = sum_t u_t v_t.
//
// Work split.  Key rows never mix (notes section 1.2), in the backward too:
// row i of C_{t-1} depends on row i of D_t only.  One CTA per chain (b, n);
// compute warp w owns key rows 16w..16w+15 and all 128 value columns, so the
// chain needs no exchange between warps: per step a warp runs
//   C_{t-1}[rows] = f R + D[rows] W^T
// as 128 m16n8k16 warp MMAs (A = bf16 D of its own rows, from registers;
// B = W^T fragments by ldmatrix from a swizzled bf16 copy of W in shared
// memory).  Chunks of `ckpt_every` steps are walked in reverse: first the
// chunk's forward rerun from its checkpoint (the same warp-MMA step with an
// fp16 copy of W, as the forward computes it), which writes fp16 Z_t and
// H_{t-1} per thread to a global scratch cache and forms dq_t; then the
// reverse walk reads them back.  Per step each warp also writes bf16
// H_{t-1} and D_t tiles of its rows, and one thread issues the tcgen05 MMAs
// dW += H_{t-1}^T D_t (M = N = 128, K = 16 per warp) into a tensor-memory
// accumulator; the tiles are double-buffered behind the MMAs' commit.
// dk and dq are row sums (shuffles over the four lanes of a row), dv and df
// are summed over the rows in a fixed order (a reduce-scatter of shuffles for
// dv, a shuffle tree for df, then over the warps).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"
#include "ptx.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 128;
constexpr int kNT = kV / 8;    // n-tiles of 8 value columns per warp
constexpr int kKT = kV / 16;   // k-tiles of the contraction over value columns
constexpr int kStage = 16;     // steps of inputs staged in shared memory at a time
constexpr int kMinWarps = 4;   // the dW read-back needs all four TMEM lane quadrants

struct TcBwdParams {
  BwdArgs a;
  int nw;        // compute warps (K / 16)
  int nchunks;
  uint32_t wf_off, wb_off, in_off, q_off, k_off, v_off, u_off, f_off, tile_off, tile_bytes;
  uint32_t dvp_off, red_off, dwr_off, bar_off, misc_off;
};

// 128 x 128 16-bit tile, row-major with the 16-byte chunks of row r permuted
// by r mod 8, so that the eight rows of an ldmatrix block hit distinct banks.
__device__ __forceinline__ uint32_t wt_off(int r, int col) {
  return static_cast<uint32_t>(r * 256 + ((((col >> 3) ^ (r & 7))) << 4) + (col & 7) * 2);
}

// Canonical no-swizzle core-matrix layout of a 16-row x 128-column bf16 tile:
// the 8 x 8 block (rows 8i.., columns 8j..) is 128 contiguous bytes at
// 256 j + 128 i.  As tcgen05 operands (MN-major, the columns contiguous) the
// core matrices advance by 128 bytes along K (the 16 rows) and 256 along M / N.
__device__ __forceinline__ uint32_t cm16_off(int row, int col) {
  return static_cast<uint32_t>((col >> 3) * 256 + (row >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}

__device__ __forceinline__ uint32_t f16_to_bf16x2(uint32_t w) { return pack2_bf16(f16lo(w), f16hi(w)); }

// Bring `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

template <bool kClip>
__global__ void __launch_bounds__(256, 1) tc_backward_kernel(const __grid_constant__ TcBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const BwdArgs& A = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nw = p.nw, T = A.T, N = A.N, K = A.K, CL = A.ckpt_every;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  const int nthr = static_cast<int>(blockDim.x);
  const int CT = nw * 32;  // compute threads (named barrier 1)
  StatusBlock* status = A.status;
  const uint32_t wf = smem_u32(smem + p.wf_off), wb = smem_u32(smem + p.wb_off);
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + p.q_off);  // [kStage][K]
  uint16_t* ks = reinterpret_cast<uint16_t*>(smem + p.k_off);  // [kStage][K]
  uint16_t* vs = reinterpret_cast<uint16_t*>(smem + p.v_off);  // [kStage][kV]
  float* us = reinterpret_cast<float*>(smem + p.u_off);        // [kStage][kV]
  float* fs = reinterpret_cast<float*>(smem + p.f_off);        // [kStage]
  float* dvp = reinterpret_cast<float*>(smem + p.dvp_off);     // [2][nw][kV]
  float* red = reinterpret_cast<float*>(smem + p.red_off);     // [2][nw]
  float* dwr = reinterpret_cast<float*>(smem + p.dwr_off);     // [kV]
  uint64_t* dwfree = reinterpret_cast<uint64_t*>(smem + p.bar_off);  // [2] tile buffers
  uint64_t* dwdone = dwfree + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 8);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&dwfree[0]), 1);  // the dW MMAs' commit
    mbar_init(smem_u32(&dwfree[1]), 1);
    mbar_init(smem_u32(dwdone), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kV);  // dW accumulator: lane m, column j
    tmem_relinquish();
  }
  // W twice, swizzled row-major: fp16 for the rerun (as the forward computes
  // it; entries outside the fp16 range are reported), bf16 for D W^T.
  {
    const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
    for (int e = threadIdx.x; e < kV * kV / 2; e += nthr) {
      const int r = (2 * e) / kV, c = (2 * e) % kV;
      const uint32_t w2 = *reinterpret_cast<const uint32_t*>(Wg + r * kV + c);
      const uint32_t h2 = bf16x2_to_f16x2(w2);
      if (!f16x2_finite(h2)) report_device_error(status, kStatusCheck, kWhereWRange);
      *reinterpret_cast<uint32_t*>(smem + p.wf_off + wt_off(r, c)) = h2;
      *reinterpret_cast<uint32_t*>(smem + p.wb_off + wt_off(r, c)) = w2;
    }
    for (int j = threadIdx.x; j < kV; j += nthr) dwr[j] = 0.f;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  const bool comp = warp < nw;
  const int g = lane >> 2, qd = lane & 3;
  const int w = warp;
  const GateSrc gs{A.f, A.gate_a, A.gate_alpha, A.gate_beta, true};
  const uint16_t* qg = static_cast<const uint16_t*>(A.q);
  const uint16_t* kg = static_cast<const uint16_t*>(A.k);
  const uint16_t* vg = static_cast<const uint16_t*>(A.v);
  const uint16_t* wrg = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
  const int qkH = qk_heads(A.qkN, N), qkh = qk_head(A.qkN, n);
  // Per-thread scratch: the chunk cache [chain][step][warp][16 words][32
  // lanes] (words 0-7: fp16 Z_t, 8-15: fp16 H_{t-1}, k-tile order), then the
  // state gradient kept aside during the rerun [chain][warp][64][32 lanes].
  uint4* const cache = reinterpret_cast<uint4*>(A.scratch) +
                       (static_cast<int64_t>(chain) * CL * nw + w) * 16 * 32 + lane;
  float* const cg_save = reinterpret_cast<float*>(reinterpret_cast<uint4*>(A.scratch) +
                                                  static_cast<int64_t>(A.B) * N * CL * nw * 16 * 32) +
                         (static_cast<int64_t>(chain) * nw + w) * 64 * 32 + lane;
  const int64_t cstride = static_cast<int64_t>(nw) * 16 * 32;  // uint4 per step

  // State gradient C (accumulator layout: rows 16w + g (+8), columns 8nt + 2qd (+1)).
  float cg[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = 16 * w + g + 8 * (e >> 1), col = 8 * nt + 2 * qd + (e & 1);
      cg[nt][e] = (comp && A.dH_T != nullptr) ? A.dH_T[(static_cast<int64_t>(chain) * K + row) * kV + col] : 0.f;
    }
  }

  // Inputs of steps t0 .. t0 + cnt - 1 into the staging slots (all threads).
  auto stage = [&](int t0, int cnt) {
    __syncthreads();  // every reader of the previous slots is done
    for (int e = threadIdx.x; e < cnt * K; e += nthr) {
      const int s = e / K, i = e % K;
      const int64_t rq = ((static_cast<int64_t>(b) * T + t0 + s) * qkH + qkh) * K + i;
      qs[s * K + i] = qg[rq];
      ks[s * K + i] = kg[rq];
    }
    for (int e = threadIdx.x; e < cnt * kV; e += nthr) {
      const int s = e / kV, j = e % kV;
      const int64_t rv = ((static_cast<int64_t>(b) * T + t0 + s) * N + n) * kV + j;
      vs[s * kV + j] = vg[rv];
      us[s * kV + j] = A.dy[rv];
    }
    for (int s = threadIdx.x; s < cnt; s += nthr)
      fs[s] = gate_value(gs, (static_cast<int64_t>(b) * T + t0 + s) * N + n, n);
    __syncthreads();
  };

  const uint32_t idesc = idesc_bf16_f32(128, kV, /*a_mn_major=*/true, /*b_mn_major=*/true);
  int rs = 0;  // reverse steps done
  for (int ci = 0; ci < p.nchunks; ++ci) {
    const int c = p.nchunks - 1 - ci;
    const int s0 = c * CL, L = min(CL, T - s0);

    // ---------------- rerun of the chunk from its checkpoint (Eq. 10-11) ----------------
    float h[kNT][4];
    if (comp) {
      // The state gradient waits in scratch while the rerun needs the registers.
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) cg_save[(nt * 4 + e) * 32] = cg[nt][e];
      const float* hsrc = (c == 0) ? (A.H0 != nullptr ? A.H0 + static_cast<int64_t>(chain) * K * kV : nullptr)
                                   : A.ckpt + (static_cast<int64_t>(chain) * A.n_ckpt + (c - 1)) * K * kV;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = 16 * w + g + 8 * (e >> 1), col = 8 * nt + 2 * qd + (e & 1);
          h[nt][e] = hsrc != nullptr ? hsrc[row * kV + col] : 0.f;
        }
    }
    for (int sb = 0; sb < L; sb += kStage) {
      const int cnt = min(kStage, L - sb);
      stage(s0 + sb, cnt);
      if (!comp) continue;
      for (int s = 0; s < cnt; ++s) {
        const int sl = sb + s;
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + sl) * N + n;
        const float k0 = bf16_bits_to_f32(ks[s * K + 16 * w + g]);
        const float k1 = bf16_bits_to_f32(ks[s * K + 16 * w + g + 8]);
        const float omf = 1.f - fs[s];
        uint4* const cst = cache + sl * cstride;
        // fp16 H_{t-1} of this warp's rows as A fragments (k-tile kt = n-tiles
        // 2kt, 2kt + 1 of the accumulator layout); cached as they are.
        uint32_t a[kKT][4];
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt) {
          a[kt][0] = pack2_f16(h[2 * kt][0], h[2 * kt][1]);
          a[kt][1] = pack2_f16(h[2 * kt][2], h[2 * kt][3]);
          a[kt][2] = pack2_f16(h[2 * kt + 1][0], h[2 * kt + 1][1]);
          a[kt][3] = pack2_f16(h[2 * kt + 1][2], h[2 * kt + 1][3]);
          cst[(8 + kt) * 32] = make_uint4(a[kt][0], a[kt][1], a[kt][2], a[kt][3]);
        }
        // H_{t-1} W + k v^T: the rank-1 write seeds the accumulator (exact).
        float acc[kNT][4];
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * kV + 8 * nt + 2 * qd);
          const float v0 = bf16lo(vv), v1 = bf16hi(vv);
          acc[nt][0] = k0 * v0;
          acc[nt][1] = k0 * v1;
          acc[nt][2] = k1 * v0;
          acc[nt][3] = k1 * v1;
        }
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt)
#pragma unroll
          for (int ntp = 0; ntp < kNT / 2; ++ntp) {
            // B[k = m][n = j] = W[m][j]: four 8 x 8 blocks (m 16kt.. | 16kt+8..) x
            // (j 16ntp.. | 16ntp+8..), transposed on load.
            const int bi = lane >> 3;
            uint32_t bf[4];
            ldmatrix_x4_trans(bf, wf + wt_off(16 * kt + (bi & 1) * 8 + (lane & 7), 8 * (2 * ntp + (bi >> 1))));
            mma_f16_16816(acc[2 * ntp], a[kt], bf[0], bf[1]);
            mma_f16_16816(acc[2 * ntp + 1], a[kt], bf[2], bf[3]);
          }
        // Eq. 10-11; fp16 Z_t to the cache; dq_t = H_t u_t over the warp's rows.
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt) {
          float z[2][4];
#pragma unroll
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int nt = 2 * kt + m;
              z[m][e] = tanh_fast(acc[nt][e]);
              h[nt][e] = fmaf(omf, z[m][e] - h[nt][e], h[nt][e]);
            }
          cst[kt * 32] = make_uint4(pack2_f16(z[0][0], z[0][1]), pack2_f16(z[0][2], z[0][3]),
                                    pack2_f16(z[1][0], z[1][1]), pack2_f16(z[1][2], z[1][3]));
        }
        float pq0 = 0.f, pq1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const float2 uu = *reinterpret_cast<const float2*>(us + s * kV + 8 * nt + 2 * qd);
          pq0 = fmaf(h[nt][0], uu.x, fmaf(h[nt][1], uu.y, pq0));
          pq1 = fmaf(h[nt][2], uu.x, fmaf(h[nt][3], uu.y, pq1));
        }
        pq0 += __shfl_xor_sync(0xffffffffu, pq0, 1);
        pq1 += __shfl_xor_sync(0xffffffffu, pq1, 1);
        pq0 += __shfl_xor_sync(0xffffffffu, pq0, 2);
        pq1 += __shfl_xor_sync(0xffffffffu, pq1, 2);
        if (qd == 0) {
          A.dq[rowt * K + 16 * w + g] = pq0;
          A.dq[rowt * K + 16 * w + g + 8] = pq1;
        }
      }
    }
    if (comp) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) cg[nt][e] = cg_save[(nt * 4 + e) * 32];
    }

    // ---------------- reverse walk over the chunk ----------------
    for (int sb = ((L - 1) / kStage) * kStage; sb >= 0; sb -= kStage) {
      const int cnt = min(kStage, L - sb);
      stage(s0 + sb, cnt);
      if (!comp) continue;
      for (int s = cnt - 1; s >= 0; --s, ++rs) {
        const int sl = sb + s;
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + sl) * N + n;
        const int bsel = rs & 1;
        // This tile buffer was last read by the dW MMAs of step rs - 2.  (A
        // give-up raised the abort flag; the walk goes on so that every warp
        // reaches the same barriers, and the status block reports it.)
        if (rs >= 2) mbar_wait(smem_u32(&dwfree[bsel]), ((rs >> 1) - 1) & 1, abort_flag, status, kWhereBwdDW);
        const float q0 = bf16_bits_to_f32(qs[s * K + 16 * w + g]);
        const float q1 = bf16_bits_to_f32(qs[s * K + 16 * w + g + 8]);
        const float k0 = bf16_bits_to_f32(ks[s * K + 16 * w + g]);
        const float k1 = bf16_bits_to_f32(ks[s * K + 16 * w + g + 8]);
        const float ft = fs[s], omf = 1.f - ft;
        const uint4* const cst = cache + sl * cstride;
        // The step's cached Z_t and H_{t-1}, all loads issued before the first
        // use; the warp's 8 KB of the next step back are brought into L2.
        uint4 zq[kKT], hq[kKT];
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt) {
          zq[kt] = cst[kt * 32];
          hq[kt] = cst[(8 + kt) * 32];
        }
        if (sl > 0 && lane == 0) prefetch_l2(cst - cstride - lane, 16 * 32 * 16);
        const uint32_t tbh = smem_u32(smem + p.tile_off + bsel * p.tile_bytes + w * 8192), tbd = tbh + 4096;
        float* const dvw = dvp + (bsel * nw + w) * kV;
        uint32_t dA[kKT][4];  // bf16 D_t of the warp's rows (A fragments)
        float pk0 = 0.f, pk1 = 0.f, pf = 0.f;
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt) {
          const uint32_t zw[4] = {zq[kt].x, zq[kt].y, zq[kt].z, zq[kt].w};
          const uint32_t hw[4] = {hq[kt].x, hq[kt].y, hq[kt].z, hq[kt].w};
          // bf16 H_{t-1} into the dW tile (word positions as in the cache).
          st_shared_b32(tbh + cm16_off(g, 16 * kt + 2 * qd), f16_to_bf16x2(hw[0]));
          st_shared_b32(tbh + cm16_off(g + 8, 16 * kt + 2 * qd), f16_to_bf16x2(hw[1]));
          st_shared_b32(tbh + cm16_off(g, 16 * kt + 8 + 2 * qd), f16_to_bf16x2(hw[2]));
          st_shared_b32(tbh + cm16_off(g + 8, 16 * kt + 8 + 2 * qd), f16_to_bf16x2(hw[3]));
          float pv[2][2];  // dv shares: columns 8nt + 2qd (+1) over rows g, g+8
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int nt = 2 * kt + m;
            const float2 uu = *reinterpret_cast<const float2*>(us + s * kV + 8 * nt + 2 * qd);
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * kV + 8 * nt + 2 * qd);
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            float D[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float R = fmaf((e < 2) ? q0 : q1, (e & 1) ? uu.y : uu.x, cg[nt][e]);  // R = C + q u^T
              const uint32_t zword = zw[2 * m + (e >> 1)], hword = hw[2 * m + (e >> 1)];
              const float z = (e & 1) ? f16hi(zword) : f16lo(zword);
              const float hp = (e & 1) ? f16hi(hword) : f16lo(hword);
              D[e] = omf * R * fmaf(-z, z, 1.f);  // D = (1 - f) R (1 - Z^2)
              pf = fmaf(R, hp - z, pf);           // <R, H_{t-1} - Z>
              cg[nt][e] = ft * R;                 // the chain accumulator starts at f R
            }
            pk0 = fmaf(D[0], v0, fmaf(D[1], v1, pk0));  // D v, rows g, g+8
            pk1 = fmaf(D[2], v0, fmaf(D[3], v1, pk1));
            pv[m][0] = fmaf(D[0], k0, D[2] * k1);       // D^T k over the two rows
            pv[m][1] = fmaf(D[1], k0, D[3] * k1);
            dA[kt][2 * m] = pack2_bf16(D[0], D[1]);
            dA[kt][2 * m + 1] = pack2_bf16(D[2], D[3]);
          }
          st_shared_b32(tbd + cm16_off(g, 16 * kt + 2 * qd), dA[kt][0]);
          st_shared_b32(tbd + cm16_off(g + 8, 16 * kt + 2 * qd), dA[kt][1]);
          st_shared_b32(tbd + cm16_off(g, 16 * kt + 8 + 2 * qd), dA[kt][2]);
          st_shared_b32(tbd + cm16_off(g + 8, 16 * kt + 8 + 2 * qd), dA[kt][3]);
          // dv shares summed over the warp's rows (the eight lanes g of a
          // column), reduce-scatter in a fixed order: each exchange halves the
          // values a lane carries, so lane g ends with the full sum of value
          // (g >> 1) (column 16kt + 8 (g >> 2) + 2qd + ((g >> 1) & 1)).
          {
            const bool hi4 = (g & 4) != 0, hi2 = (g & 2) != 0;
            float k0 = hi4 ? pv[1][0] : pv[0][0], k1 = hi4 ? pv[1][1] : pv[0][1];
            k0 += __shfl_xor_sync(0xffffffffu, hi4 ? pv[0][0] : pv[1][0], 16);
            k1 += __shfl_xor_sync(0xffffffffu, hi4 ? pv[0][1] : pv[1][1], 16);
            float kk = hi2 ? k1 : k0;
            kk += __shfl_xor_sync(0xffffffffu, hi2 ? k0 : k1, 8);
            kk += __shfl_xor_sync(0xffffffffu, kk, 4);
            if ((g & 1) == 0) dvw[16 * kt + 8 * (g >> 2) + 2 * qd + ((g >> 1) & 1)] = kk;
          }
        }
        // Serial chain: C_{t-1} = f R + D W^T.  B[k = m][n = j] = W[j][m]:
        // blocks (j 16ntp.. | 16ntp+8..) x (m 16kt.. | 16kt+8..) of the bf16 W.
#pragma unroll
        for (int kt = 0; kt < kKT; ++kt)
#pragma unroll
          for (int ntp = 0; ntp < kNT / 2; ++ntp) {
            const int bi = lane >> 3;
            uint32_t bf[4];
            ldmatrix_x4(bf, wb + wt_off(8 * (2 * ntp + (bi >> 1)) + (lane & 7), 16 * kt + (bi & 1) * 8));
            mma_bf16_16816(cg[2 * ntp], dA[kt], bf[0], bf[1]);
            mma_bf16_16816(cg[2 * ntp + 1], dA[kt], bf[2], bf[3]);
          }
        if constexpr (kClip) {  // per-step clipping of the state gradient
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) cg[nt][e] = fminf(fmaxf(cg[nt][e], -A.clip), A.clip);
        }
        // dk_t: rows g, g+8 over the four lanes of a row.
        pk0 += __shfl_xor_sync(0xffffffffu, pk0, 1);
        pk1 += __shfl_xor_sync(0xffffffffu, pk1, 1);
        pk0 += __shfl_xor_sync(0xffffffffu, pk0, 2);
        pk1 += __shfl_xor_sync(0xffffffffu, pk1, 2);
        if (qd == 0) {
          A.dk[rowt * K + 16 * w + g] = pk0;
          A.dk[rowt * K + 16 * w + g + 8] = pk1;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) pf += __shfl_xor_sync(0xffffffffu, pf, o);
        if (lane == 0) red[bsel * nw + w] = pf;
        fence_proxy_async_smem();  // the tiles are read by the tensor core
        named_bar_sync(1, CT);
        if (warp == 0) {  // dW += H_{t-1}^T D_t, one K = 16 slice per warp's rows
          tc_fence_after_sync();
          if (elect_one()) {
            for (int w2 = 0; w2 < nw; ++w2) {
              const uint32_t t2 = smem_u32(smem + p.tile_off + bsel * p.tile_bytes + w2 * 8192);
              tc_mma_f16_ss(tmem_base, smem_desc_noswizzle(t2, 128, 256), smem_desc_noswizzle(t2 + 4096, 128, 256),
                            idesc, (rs > 0 || w2 > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&dwfree[bsel]));
          }
          __syncwarp();
        }
        // dv_t = the warps' shares in a fixed order + w_r u_t; dw_r += u_t v_t.
        for (int j = threadIdx.x; j < kV; j += CT) {
          float acc2 = 0.f;
          for (int w2 = 0; w2 < nw; ++w2) acc2 += dvp[(bsel * nw + w2) * kV + j];
          const float uj = us[s * kV + j];
          A.dv[rowt * kV + j] = fmaf(bf16_bits_to_f32(wrg[j]), uj, acc2);
          dwr[j] = fmaf(uj, bf16_bits_to_f32(vs[s * kV + j]), dwr[j]);
        }
        if (threadIdx.x == 0) {
          float d = 0.f;
          for (int w2 = 0; w2 < nw; ++w2) d += red[bsel * nw + w2];
          A.df[rowt] = d;
        }
      }
    }
  }

  if (comp && A.dH0 != nullptr) {  // C_0, the state gradient left after step 1
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * w + g + 8 * (e >> 1), col = 8 * nt + 2 * qd + (e & 1);
        A.dH0[(static_cast<int64_t>(chain) * K + row) * kV + col] = cg[nt][e];
      }
  }
  // dW partial of the chain from tensor memory once its last MMAs completed;
  // dw_r partial from shared memory.
  if (warp == 0) {
    if (elect_one()) tc_commit(smem_u32(dwdone));
    __syncwarp();
  }
  __syncthreads();
  for (int j = threadIdx.x; j < kV; j += nthr) A.dwr_part[static_cast<int64_t>(chain) * kV + j] = dwr[j];
  if (warp < kMinWarps) {
    mbar_wait(smem_u32(dwdone), 0, abort_flag, status, kWhereBwdDW);
    tc_fence_after_sync();
    float* dst = A.dW_part + static_cast<int64_t>(chain) * kV * kV + (32 * warp + lane) * kV;
#pragma unroll 1
    for (int c0 = 0; c0 < kV; c0 += 32) {
      uint32_t r[32];
      tmem_ld_32x32b<32>(tmem_base + (static_cast<uint32_t>(32 * warp) << 16) + c0, r);
      tmem_ld_wait();
      tmem_ld_fence_regs(r);
#pragma unroll
      for (int u = 0; u < 32; u += 4)
        *reinterpret_cast<float4*>(dst + c0 + u) = make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                                                               __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kV);
  }
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <bool kClip>
cudaError_t launch_t(const BwdArgs& a, cudaStream_t s) {
  TcBwdParams p{};
  p.a = a;
  p.nw = a.K / 16;
  p.nchunks = (a.T + a.ckpt_every - 1) / a.ckpt_every;
  uint32_t off = 0;
  p.wf_off = off;
  off += kV * kV * 2;
  p.wb_off = off;
  off += kV * kV * 2;
  p.q_off = off;
  off = align_up(off + kStage * a.K * 2, 16);
  p.k_off = off;
  off = align_up(off + kStage * a.K * 2, 16);
  p.v_off = off;
  off = align_up(off + kStage * kV * 2, 16);
  p.u_off = off;
  off = align_up(off + kStage * kV * 4, 16);
  p.f_off = off;
  off = align_up(off + kStage * 4, 128);
  p.tile_off = off;
  p.tile_bytes = static_cast<uint32_t>(p.nw) * 8192;
  off += 2 * p.tile_bytes;
  p.dvp_off = off;
  off += 2 * p.nw * kV * 4;
  p.red_off = off;
  off = align_up(off + 2 * p.nw * 4, 16);
  p.dwr_off = off;
  off += kV * 4;
  p.bar_off = off;
  off += 3 * 8;
  p.misc_off = off;
  off += 16;
  const uint32_t smem = align_up(off, 128) + 1024;  // + slack for the 1 KB alignment
  cudaError_t e = cudaFuncSetAttribute(tc_backward_kernel<kClip>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int threads = 32 * std::max(p.nw, kMinWarps);
  tc_backward_kernel<kClip><<<a.B * a.N, threads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool tc_backward_supported(int K, int V) { return V == kV && K >= 16 && K <= 128 && K % 16 == 0; }

int tc_backward_parts(int, int) { return 1; }

// The chunk cache (fp16 Z_t and H_{t-1} of every step of a chunk) and the
// state gradient kept aside during each rerun, per chain.
size_t tc_backward_scratch_bytes(int B, int N, int K, int V, int ckpt_every) {
  if (tc_backward128_supported(K, V, ckpt_every)) return tc_backward128_scratch_bytes(B, N, ckpt_every);
  const size_t chains = static_cast<size_t>(B) * N;
  return chains * static_cast<size_t>(ckpt_every) * K * V * 4 + chains * static_cast<size_t>(K) * V * 4;
}

cudaError_t launch_tc_backward(const BwdArgs& a, cudaStream_t s) {
  if (!tc_backward_supported(a.K, a.V) || a.dtype != M2RNN_BF16) return cudaErrorInvalidValue;
  // K = 128 with chunks of at most 16 steps: the all-tcgen05 kernel.
  if (tc_backward128_supported(a.K, a.V, a.ckpt_every)) return launch_tc_backward128(a, s);
  return a.clip > 0.f ? launch_t<true>(a, s) : launch_t<false>(a, s);
}

}  // namespace m2rnn
