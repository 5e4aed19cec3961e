// tcgen05 forward scan of the M2RNN recurrence for bf16 inputs, fp32 state.
//
// Recurrence (reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued
// States for Scalable Language Modeling", section 2.1, Eq. 10-12):
//   Z_t = tanh(H_{t-1} W + k_t v_t^T),  H_t = f_t H_{t-1} + (1-f_t) Z_t,
//   y_t = H_t^T q_t + w_r * v_t.
//
// Work split.  Key rows never mix (notes section 1.2): every row of H is its
// own vector recurrence sharing W.  A chain (b, n) is therefore split into R
// row blocks of G*NR rows, one CTA each, the R CTAs of a chain forming one
// thread-block cluster; only the readout y_t sums over rows, and that sum
// crosses CTAs through distributed shared memory, off the serial chain.
//
// Per step, per group of NR rows (one warpgroup), the transform runs on the
// tensor core in transposed form
//     D^T [V x NR] = W^T [V x V] * H_{t-1}^T [V x NR]      (M = 128, N = NR, K = V)
// with A = W^T written to tensor memory once (stacked 128/V times to fill
// M = 128, so the V = 64 case keeps all four TMEM lane quadrants busy), B =
// fp16(H_{t-1}) rewritten in shared memory every step (W re-encoded as fp16
// too: see mma_common.cuh), D in TMEM.  For V = 128 the rank-1 write v_t k_t^T
// is one more K slice of bf16 operands (A column [v_t, 0..], B row k_t: exact
// products) issued as its own MMA; for V = 64 the epilogue adds it.  TMEM lane
// L holds value column j = L mod V, so each thread owns a column j and ROWS
// rows of the state in fp32 registers: tanh, the gate blend and the readout
// over its rows are all thread-local.  The fp16 copy of H_t goes back to
// shared memory as the next MMA's B operand (MN-major: the thread's ROWS
// values are 16-byte runs).
//
// Warp roles: warps 0..4G-1 = G epilogue warpgroups; warp 4G = the MMA warp,
// which issues every group's MMAs from one elected lane of a converged warp,
// alternating between the groups so that one group's MMAs overlap the other
// group's tanh work (issued from an epilogue warp instead, the MMAs made that
// warp the one the next step waits for: 297 against 224 ns per step at
// V = 64, measured); warp 4G+1 = TMA producer for q/k/v tiles of S = 32
// steps (f through plain loads); warp 4G+2 = readout reducer, which sums the
// per-group/per-CTA partial readouts of a tile (one of them carries w_r * v)
// and stores y.  Checkpoints are written between segments of steps.  Every
// wait is bounded (see ptx.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"
#include "ptx.cuh"

namespace m2rnn {
namespace {

constexpr int kS = 32;   // steps per input tile (one f value per producer lane)
constexpr int kYS = 2;   // readout partial stages

template <int V_, int ROWS_>
struct FwdCfg {
  static constexpr int V = V_;
  static constexpr int ROWS = ROWS_;            // state rows per thread
  static constexpr int COPIES = 128 / V;        // W^T stacked to fill M = 128
  static constexpr int NR = ROWS * COPIES;      // rows per group = MMA N
  static constexpr int NS = (V == 64) ? 4 : 3;  // input pipeline stages
  static constexpr int KSTEPS = V / 16;         // MMAs per step (K = 16 each)
  // V = 128: the rank-1 write runs on the tensor core as one more K slice
  // (17 % faster on the T = 4096, K = V = 128 workload); at V = 64, with 8
  // rows per thread, writing the slice costs more than the FMAs it saves
  // (232 against 312 ns per step on the 16K workload), so it stays in the
  // epilogue there.
  static constexpr bool FOLD = (V == 128);
  // B = [H_{t-1}^T ; X]: V (+ 16) K-rows; the slice X carries the rank-1
  // write (first row k_t, the rest 0).
  static constexpr int KB = V + (FOLD ? 16 : 0);
  static constexpr uint32_t B_BYTES = NR * KB * 2u;
  static constexpr uint32_t SBO = KB * 16u;  // next 8 columns (B)
  static constexpr uint32_t LBO = 128u;     // next 8 K-elements
  static_assert(ROWS % 8 == 0, "rows per thread come in 16-byte runs");
  static_assert(NR % 16 == 0 && NR <= 256, "MMA N for M = 128");
};

struct TcFwdParams {
  FwdArgs a;
  int R, NRtot;
  int ntiles;
  uint32_t tmem_cols;
  uint32_t a_tcol;  // TMEM column of the A operand (W^T stacked), then (V = 128) G x 8 columns of [v_t, 0]
  uint32_t b_off, stage_off, stage_bytes, q_off, k_off, v_off, f_off;
  uint32_t y_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

// Store 32 data-path lanes x 32 bits x 1 column (thread i writes lane base + i).
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}

__device__ __forceinline__ void unpack8_bf16(const uint4 w, float (&o)[8]) {
  o[0] = __uint_as_float(w.x << 16);
  o[1] = __uint_as_float(w.x & 0xFFFF0000u);
  o[2] = __uint_as_float(w.y << 16);
  o[3] = __uint_as_float(w.y & 0xFFFF0000u);
  o[4] = __uint_as_float(w.z << 16);
  o[5] = __uint_as_float(w.z & 0xFFFF0000u);
  o[6] = __uint_as_float(w.w << 16);
  o[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

// Compile-time modes, no per-step test: G epilogue warpgroups, kY = readout
// y, kCk = checkpoints.  (G as a runtime value left the readout reducer's
// loops unrolled too little to keep up: 5.72 against 4.88 ms on the
// T = 4096, K = V = 128 workload, measured.)
template <int V, int ROWS, int G, bool kY, bool kCk>
__global__ void __launch_bounds__((4 * G + 3) * 32, 1)
    tc_forward_kernel(const __grid_constant__ TcFwdParams p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  using C = FwdCfg<V, ROWS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Align the working base to 1 KB (the launch reserves the slack).
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = p.R, NRtot = p.NRtot;
  const int T = p.a.T, N = p.a.N;
  const int cta_rank = static_cast<int>(blockIdx.x) % R;
  const int chain = static_cast<int>(blockIdx.x) / R;
  const int b = chain / N, n = chain % N;
  const int ntiles = p.ntiles;
  constexpr bool do_y = kY;
  constexpr int slots = G * C::COPIES;
  StatusBlock* status = p.a.status;

  uint8_t* sB = smem + p.b_off;
  uint8_t* sStage = smem + p.stage_off;
  float* sY = reinterpret_cast<float*>(smem + p.y_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::NS;
  uint64_t* dfull = bars + 2 * C::NS;
  uint64_t* hready = dfull + G;
  uint64_t* yfull = hready + G;
  uint64_t* ypeer = yfull + kYS;
  uint64_t* yempty = ypeer + kYS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(smem_u32(&full[i]), 32);
      mbar_init(smem_u32(&empty[i]), 4 * G);
    }
    for (int g = 0; g < G; ++g) {
      mbar_init(smem_u32(&dfull[g]), 1);
      mbar_init(smem_u32(&hready[g]), 4);
    }
    for (int i = 0; i < kYS; ++i) {
      mbar_init(smem_u32(&yfull[i]), 4 * G);
      mbar_init(smem_u32(&ypeer[i]), R);
      mbar_init(smem_u32(&yempty[i]), R);
    }
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (uint32_t e = threadIdx.x * 16; e < static_cast<uint32_t>(G) * C::B_BYTES; e += blockDim.x * 16)
      *reinterpret_cast<uint4*>(sB + e) = zero;  // H_0 = 0 and the rank-1 slice's zero rows
  }
  __syncthreads();
  if (p.a.H0 != nullptr && warp < 4 * G) {
    // fp16(H_0) as step 0's B operand: each epilogue thread writes the rows
    // and column it owns (the same mapping as below; together they cover
    // every element of each group's tile).
    const int g = warp / 4, L = 32 * (warp % 4) + lane;
    const int j = L % V, c = L / V;
    const int64_t row_global = static_cast<int64_t>(cta_rank) * NRtot + g * C::NR + c * ROWS;
    const float* src = p.a.H0 + (static_cast<int64_t>(chain) * p.a.K + row_global) * V + j;
    uint8_t* bslot = sB + g * C::B_BYTES + ((c * ROWS) / 8) * C::SBO + (j / 8) * C::LBO + (j % 8) * 16;
#pragma unroll
    for (int r0 = 0; r0 < ROWS; r0 += 8) {
      uint4 pk;
      pk.x = pack2_f16(src[(r0 + 0) * V], src[(r0 + 1) * V]);
      pk.y = pack2_f16(src[(r0 + 2) * V], src[(r0 + 3) * V]);
      pk.z = pack2_f16(src[(r0 + 4) * V], src[(r0 + 5) * V]);
      pk.w = pack2_f16(src[(r0 + 6) * V], src[(r0 + 7) * V]);
      *reinterpret_cast<uint4*>(bslot + (r0 / 8) * C::SBO) = pk;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // fp16 operands: W^T re-encoded, H_{t-1} rounded (see mma_common.cuh).
  const uint32_t idesc = idesc_f16_f32(128, C::NR, /*a_mn_major=*/false, /*b_mn_major=*/true);
  // The rank-1 slice multiplies the bf16 inputs as they are (exact products).
  const uint32_t idesc_x = idesc_bf16_f32(128, C::NR, /*a_mn_major=*/false, /*b_mn_major=*/true);
  const uint32_t a_tmem = tmem_base + p.a_tcol;
  if (warp < 4) {
    // A = [W^T; W^T; ...] in tensor memory (M = 128 lanes, K = V): lane L holds
    // row L, i.e. A[L][m] = W[m][L mod V], two fp16 per 32-bit column.  Warp w
    // writes lanes 32w..32w+31.
    const uint16_t* Wg = static_cast<const uint16_t*>(p.a.W) + static_cast<int64_t>(n) * V * V;
    const int jr = (32 * warp + lane) % V;
#pragma unroll
    for (int c0 = 0; c0 < V / 2; c0 += 32) {
      uint32_t regs[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int m = 2 * (c0 + u);
        regs[u] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[m * V + jr]) |
                                  (static_cast<uint32_t>(Wg[(m + 1) * V + jr]) << 16));
        if (!f16x2_finite(regs[u])) report_device_error(p.a.status, kStatusCheck, kWhereWRange);
      }
      tmem_st_32x32b_x32(a_tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, regs);
    }
    tmem_st_wait();
  }
  if (C::FOLD && warp < 4 * G) {
    // The rank-1 slice of group warp/4's A operand: [v_t, 0, ..., 0] per
    // lane, 8 columns; all but the first element stay zero.
    const uint32_t zeros[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st_32x32b_x8(a_tmem + (static_cast<uint32_t>(32 * (warp % 4)) << 16) + V / 2 + 8 * (warp / 4), zeros);
    tmem_st_wait();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  if (warp < 4 * G) {
    // ---------------- epilogue warpgroups ----------------
    const int g = warp / 4, wq = warp % 4;
    const int L = 32 * wq + lane;
    const int j = L % V, c = L / V;  // c is uniform within a warp
    const int row_in_cta = g * C::NR + c * ROWS;
    const int64_t row_global = static_cast<int64_t>(cta_rank) * NRtot + row_in_cta;
    const uint32_t dbar = smem_u32(&dfull[g]);
    const uint32_t hbar = smem_u32(&hready[g]);
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * wq) << 16) + g * C::NR + c * ROWS;
    uint8_t* bslot = sB + g * C::B_BYTES + ((c * ROWS) / 8) * C::SBO + (j / 8) * C::LBO + (j % 8) * 16;
    // V = 128: the rank-1 write of step x enters the MMA as one more K slice:
    // A column [v_x, 0..] in this thread's TMEM lane, B row k_x (the group's
    // rows, 16-byte runs copied by the first NR/8 threads).  Written once the
    // group's previous MMA has completed, before the group's arrival.  (A
    // second slice written while the MMA runs measured slower: 1094 against
    // 984 ns per step.)
    const uint32_t xaddr = a_tmem + (static_cast<uint32_t>(32 * wq) << 16) + V / 2 + 8 * g;
    auto put_x = [&](const uint8_t* stg, int sx) {
      const uint16_t* vx = reinterpret_cast<const uint16_t*>(stg + p.v_off);
      const uint16_t* kx = reinterpret_cast<const uint16_t*>(stg + p.k_off);
      tmem_st_32x32b_x1(xaddr, static_cast<uint32_t>(vx[sx * V + j]));
      if (L < C::NR / 8)
        *reinterpret_cast<uint4*>(sB + g * C::B_BYTES + L * C::SBO + V * 16) =
            *reinterpret_cast<const uint4*>(kx + sx * NRtot + g * C::NR + 8 * L);
    };
    float h[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      h[r] = p.a.H0 ? p.a.H0[(static_cast<int64_t>(chain) * p.a.K + row_global + r) * V + j] : 0.f;
    // The residual w_r * v_t of column j rides on the partial of the chain's
    // first rows (CTA 0, group 0, row run 0); the reducer only sums partials.
    const float wrv = (cta_rank == 0 && g == 0 && c == 0)
                          ? bf16_bits_to_f32(static_cast<const uint16_t*>(p.a.w_r)[static_cast<int64_t>(n) * V + j])
                          : 0.f;
    uint32_t dphase = 0;
    int ck_left = p.a.ckpt_every, ck_idx = 0;  // countdown to the next checkpoint
    bool ok = true;
    for (int tile = 0; tile < ntiles && ok; ++tile) {
      const int st = tile % C::NS;
      if (!mbar_wait(smem_u32(&full[st]), (tile / C::NS) & 1, abort_flag, status, kWhereFwdFull)) {
        ok = false;
        break;
      }
      const int ys = tile % kYS;
      if (do_y && tile >= kYS &&
          !mbar_wait<true>(smem_u32(&yempty[ys]), ((tile / kYS) - 1) & 1, abort_flag, status,
                           kWhereFwdYEmpty)) {
        ok = false;
        break;
      }
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(stage + p.q_off);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(stage + p.v_off);
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(stage + p.k_off);
      const float* fs = reinterpret_cast<const float*>(stage + p.f_off);
      float* yp = sY + ys * (kS * slots * V);
      const int nsteps = min(kS, T - tile * kS);
      if (C::FOLD && tile == 0) {  // step 0's rank-1 slice (its H_0 part is in place already)
        put_x(stage, 0);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(hbar);
      }
      // Steps run in segments that end where a checkpoint is due, so the step
      // itself carries no checkpoint test (the countdown inside the step cost
      // ~30 ns of a ~250 ns step, measured).
      for (int s = 0; s < nsteps && ok;) {
        const int seg_end = kCk ? min(nsteps, s + ck_left) : nsteps;
        const int seg_len = seg_end - s;
        for (; s < seg_end; ++s) {
          const int t = tile * kS + s;
          const float vj = bf16_bits_to_f32(vs[s * V + j]);
          const float omf = 1.f - fs[s];
          // V = 64: the rank-1 term k_i v_j of this thread's rows, formed while
          // the MMA is in flight (the product of two bf16 values is exact, so
          // adding it later rounds as a fused multiply-add would).
          float kv[C::FOLD ? 1 : ROWS];
          if constexpr (!C::FOLD) {
            const uint16_t* kr = ks + s * NRtot + row_in_cta;
  #pragma unroll
            for (int r0 = 0; r0 < ROWS; r0 += 8) {
              float kf[8];
              unpack8_bf16(*reinterpret_cast<const uint4*>(kr + r0), kf);
  #pragma unroll
              for (int u = 0; u < 8; ++u) kv[r0 + u] = kf[u] * vj;
            }
          }
          if (!mbar_wait(dbar, dphase, abort_flag, status, kWhereFwdD)) {
            ok = false;
            break;
          }
          dphase ^= 1u;
          tc_fence_after_sync();
          uint32_t acc[ROWS];
          tmem_ld_32x32b<ROWS>(taddr, acc);
          tmem_ld_wait();
          tmem_ld_fence_regs(acc);
  #pragma unroll
          for (int r0 = 0; r0 < ROWS; r0 += 8) {
  #pragma unroll
            for (int u = 0; u < 8; ++u) {
              // (H W)_ij + k_i v_j: from the MMA alone (V = 128), or + the rank-1 term here.
              float x = __uint_as_float(acc[r0 + u]);
              if constexpr (!C::FOLD) x += kv[r0 + u];
              const float z = tanh_fast(x);                     // Eq. 10
              h[r0 + u] = fmaf(omf, z - h[r0 + u], h[r0 + u]);  // Eq. 11
            }
            uint4 pk;
            pk.x = pack2_f16(h[r0 + 0], h[r0 + 1]);
            pk.y = pack2_f16(h[r0 + 2], h[r0 + 3]);
            pk.z = pack2_f16(h[r0 + 4], h[r0 + 5]);
            pk.w = pack2_f16(h[r0 + 6], h[r0 + 7]);
            *reinterpret_cast<uint4*>(bslot + (r0 / 8) * C::SBO) = pk;
          }
          // The next step's rank-1 slice (at a tile's end, from the next tile).
          if (C::FOLD && t + 1 < T) {
            if (s + 1 < nsteps) {
              put_x(stage, s + 1);
            } else {
              const int tn = tile + 1;
              if (!mbar_wait(smem_u32(&full[tn % C::NS]), (tn / C::NS) & 1, abort_flag, status, kWhereFwdFull)) {
                ok = false;
                break;
              }
              put_x(sStage + (tn % C::NS) * p.stage_bytes, 0);
            }
          }
          // Hand the operands to the tensor core: make the generic-proxy stores
          // visible to the async proxy, complete the tensor-memory store, then
          // one arrival per warp for the MMA warp.
          fence_proxy_async_smem();
          if (C::FOLD) tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(hbar);
          // ---- off the serial chain ----
          if (do_y) {
            const uint16_t* qr = qs + s * NRtot + row_in_cta;
            float ya = wrv * vj;  // w_r * v_t, carried by one partial of each column (wrv = 0 elsewhere)
  #pragma unroll
            for (int r0 = 0; r0 < ROWS; r0 += 8) {
              float qf[8];
              unpack8_bf16(*reinterpret_cast<const uint4*>(qr + r0), qf);
  #pragma unroll
              for (int u = 0; u < 8; ++u) ya = fmaf(qf[u], h[r0 + u], ya);  // Eq. 12, this thread's rows
            }
            yp[(s * slots + g * C::COPIES + c) * V + j] = ya;
          }
        }
        if (!ok) break;
        if constexpr (kCk) {
          ck_left -= seg_len;
          if (ck_left == 0) {  // H after step tile kS + s - 1 starts a chunk: checkpoint it
            ck_left = p.a.ckpt_every;
            ++ck_idx;
            if (tile * kS + s < T) {
              float* dst =
                  p.a.ckpt + ((static_cast<int64_t>(chain) * p.a.n_ckpt + ck_idx - 1) * p.a.K + row_global) * V + j;
  #pragma unroll
              for (int r = 0; r < ROWS; ++r) dst[static_cast<int64_t>(r) * V] = h[r];
            }
          }
        }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&empty[st]));
        if (do_y) mbar_arrive(smem_u32(&yfull[ys]));
      }
    }
    if (ok && p.a.H_T != nullptr) {
      float* dst = p.a.H_T + (static_cast<int64_t>(chain) * p.a.K + row_global) * V + j;
#pragma unroll
      for (int r = 0; r < ROWS; ++r) dst[static_cast<int64_t>(r) * V] = h[r];
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == 4 * G) {
    // ---------------- MMA warp: one converged warp issues every group's MMAs ----------------
    // Step t of group g needs fp16(H_{t-1}) and the rank-1 slice of step t
    // from that group's epilogue; the groups alternate, so one group's MMAs
    // run while the other group's epilogue uses the special-function units.
    // B descriptor of group g, K slice kk: the start-address field (bits 0-13,
    // in 16-byte units) advances by (g * B_BYTES + kk * 2 * LBO) / 16.
    const uint64_t bdesc0 = smem_desc_noswizzle(smem_u32(sB), C::LBO, C::SBO);
    uint32_t hph = 0u;  // bit g: phase of hready[g]
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      for (int g = 0; g < G; ++g) {
        if (C::FOLD || t > 0) {  // (without the fold, step 0 multiplies H_0 alone, in place at the start)
          if (!mbar_wait(smem_u32(&hready[g]), (hph >> g) & 1u, abort_flag, status, kWhereFwdH)) {
            ok = false;
            break;
          }
          hph ^= 1u << g;
        }
        if (elect_one()) {
          tc_fence_after_sync();
          const uint64_t bg = bdesc0 + ((static_cast<uint32_t>(g) * C::B_BYTES) >> 4);
          if (C::FOLD)  // v_t k_t^T first (it starts the accumulator)
            tc_mma_f16_ts(tmem_base + g * C::NR, a_tmem + V / 2 + 8 * g, bg + ((C::KSTEPS * 2 * C::LBO) >> 4),
                          idesc_x, 0u);
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS; ++kk)
            tc_mma_f16_ts(tmem_base + g * C::NR, a_tmem + kk * 8, bg + ((kk * 2 * C::LBO) >> 4), idesc,
                          (C::FOLD || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&dfull[g]));
        }
        __syncwarp();
      }
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == 4 * G + 1) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const GateSrc gs{p.a.f, p.a.gate_a, p.a.gate_alpha, p.a.gate_beta, true};
    int issued = 0;
    bool ok = true;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int st = tile % C::NS;
      if (tile >= C::NS &&
          !mbar_wait(smem_u32(&empty[st]), ((tile / C::NS) - 1) & 1, abort_flag, status, kWhereFwdEmpty)) {
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
        tma_load_4d(smem_u32(stage + p.q_off), &tm_q, fb, cta_rank * NRtot, qk_head(p.a.qkN, n), t0, b);
        tma_load_4d(smem_u32(stage + p.k_off), &tm_k, fb, cta_rank * NRtot, qk_head(p.a.qkN, n), t0, b);
        tma_load_4d(smem_u32(stage + p.v_off), &tm_v, fb, 0, n, t0, b);
      } else {
        mbar_arrive(fb);
      }
      issued = tile + 1;
    }
    if (!ok) {  // let every issued copy land before the CTA can exit
      for (int tile = std::max(0, issued - C::NS); tile < issued; ++tile) {
        volatile int never = 0;
        mbar_wait(smem_u32(&full[tile % C::NS]), (tile / C::NS) & 1, &never, nullptr, kWhereFwdDrain);
      }
    }
  } else if (warp == 4 * G + 2 && do_y) {
    // ---------------- readout reducer ----------------
    // The partials already carry w_r * v_t (see the epilogue): y_t is their
    // sum in a fixed order (CTAs, then slots), every load of a step issued
    // before the first add.
    bool ok = true;
    int done = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int ys = tile % kYS;
      const uint32_t par = (tile / kYS) & 1;
      if (!mbar_wait(smem_u32(&yfull[ys]), par, abort_flag, status, kWhereFwdYFull)) {
        ok = false;
        break;
      }
      fence_acq_rel_cluster();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&ypeer[ys]), lane));
      if (!mbar_wait<true>(smem_u32(&ypeer[ys]), par, abort_flag, status, kWhereFwdYPeer)) {
        ok = false;
        break;
      }
      const int t0 = tile * kS;
      const int nsteps = min(kS, T - t0);
      const uint32_t ybase = smem_u32(sY + ys * (kS * slots * V));
      for (int s = cta_rank; s < nsteps; s += R) {
        const int64_t row = (static_cast<int64_t>(b) * T + t0 + s) * N + n;
        float acc[V / 32];
#pragma unroll
        for (int u = 0; u < V / 32; ++u) acc[u] = 0.f;
        for (int pr = 0; pr < R; ++pr) {
          const uint32_t rb = mapa_shared(ybase, pr) + static_cast<uint32_t>((s * slots * V + lane) * 4);
          float x[slots][V / 32];
#pragma unroll
          for (int sl = 0; sl < slots; ++sl)
#pragma unroll
            for (int u = 0; u < V / 32; ++u) x[sl][u] = ld_shared_cluster_f32(rb + static_cast<uint32_t>((sl * V + 32 * u) * 4));
#pragma unroll
          for (int sl = 0; sl < slots; ++sl)
#pragma unroll
            for (int u = 0; u < V / 32; ++u) acc[u] += x[sl][u];
        }
#pragma unroll
        for (int u = 0; u < V / 32; ++u) p.a.y[row * V + lane + 32 * u] = acc[u];
      }
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&yempty[ys]), lane));
      done = tile + 1;
    }
    // Do not let this CTA exit while a peer may still read its partials.
    for (int tile = std::max(0, done - kYS); tile < done; ++tile) {
      if (!mbar_wait<true>(smem_u32(&yempty[tile % kYS]), (tile / kYS) & 1, abort_flag, status,
                           kWhereFwdExit))
        break;
    }
    if (!ok) *abort_flag = 1;
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int V, int ROWS, int G, bool kY, bool kCk>
cudaError_t launch_cfg_mode(const FwdArgs& a, int R, cudaStream_t stream) {
  using C = FwdCfg<V, ROWS>;
  TcFwdParams p{};
  p.a = a;
  p.R = R;
  p.NRtot = G * C::NR;
  p.ntiles = (a.T + kS - 1) / kS;
  // TMEM: D accumulators (G x NR columns) then A = W^T (V/2 columns).
  p.a_tcol = align_up(static_cast<uint32_t>(G * C::NR), 32);
  uint32_t cols = 32;
  while (cols < p.a_tcol + V / 2 + (C::FOLD ? 8 * G : 0)) cols *= 2;
  p.tmem_cols = cols;
  p.b_off = 0;
  p.stage_off = align_up(p.b_off + G * C::B_BYTES, 128);
  p.q_off = 0;
  p.k_off = align_up(p.q_off + kS * p.NRtot * 2, 128);
  p.v_off = align_up(p.k_off + kS * p.NRtot * 2, 128);
  p.f_off = align_up(p.v_off + kS * V * 2, 128);
  p.stage_bytes = align_up(p.f_off + kS * 4, 128);
  p.y_off = p.stage_off + C::NS * p.stage_bytes;
  const uint32_t slots = G * C::COPIES;
  p.bar_off = align_up(p.y_off + kYS * kS * slots * V * 4, 8);
  p.misc_off = p.bar_off + (2 * C::NS + 2 * G + 3 * kYS) * 8;
  uint32_t smem = align_up(p.misc_off + 16, 128) + 1024;
  // One CTA per SM: the per-step latency, not throughput, bounds this kernel,
  // so CTAs must not share an SM's special-function and tensor units.
  smem = std::max<uint32_t>(smem, 120 * 1024);
  p.tx_bytes = 2 * kS * p.NRtot * 2 + kS * V * 2;

  CUtensorMap mq, mk, mv;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, a.K, p.NRtot, kS) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, p.NRtot, kS) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, V, V, kS))
    return cudaErrorInvalidValue;

  auto kern = tc_forward_kernel<V, ROWS, G, kY, kCk>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (R > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.N * R));
  cfg.blockDim = dim3(static_cast<unsigned>((4 * G + 3) * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(R);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p, mq, mk, mv);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int V, int ROWS, int G>
cudaError_t launch_cfg(const FwdArgs& a, int R, cudaStream_t stream) {
  if (a.zstash != nullptr) return cudaErrorInvalidValue;  // the Z stash is written by the warp-MMA forwards
  const bool y = a.y != nullptr, ck = a.ckpt != nullptr;
  if (y) return ck ? launch_cfg_mode<V, ROWS, G, true, true>(a, R, stream)
                   : launch_cfg_mode<V, ROWS, G, true, false>(a, R, stream);
  return ck ? launch_cfg_mode<V, ROWS, G, false, true>(a, R, stream)
            : launch_cfg_mode<V, ROWS, G, false, false>(a, R, stream);
}

}  // namespace

bool tc_forward_supported(int K, int V) {
  if (V == 64) return K >= 16 && K <= 128 && K % 16 == 0;
  if (V == 128) return K == 32 || K == 64 || K == 128;
  return false;
}

cudaError_t launch_tc_forward(const FwdArgs& a, cudaStream_t s) {
  if (a.V == 64) return launch_cfg<64, 8, 1>(a, /*R=*/a.K / 16, s);
  if (a.V == 128) {
    // Two warpgroups ping-pong on the tensor core, each with half the rows.
    if (a.K == 128) return launch_cfg<128, 64, 2>(a, 1, s);
    if (a.K == 64) return launch_cfg<128, 32, 2>(a, 1, s);
    if (a.K == 32) return launch_cfg<128, 16, 2>(a, 1, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace m2rnn
