// tcgen05 backward scan for K = V = 128 (bf16 inputs, fp32 state and
// gradients): the wide-head training workload.
//
// Recurrence (reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued
// States for Scalable Language Modeling", section 2.1, Eq. 10-12) and its
// chain rule (section 2.7): with u_t = dy_t, C_T = dH_T,
//   R_t = C_t + q_t u_t^T,  D_t = (1 - f_t) R_t (1 - Z_t^2),
//   C_{t-1} = f_t R_t + D_t W^T,
//   dq_t = H_t u_t, dk_t = D_t v_t, dv_t = D_t^T k_t + w_r u_t,
//   df_t = <R_t, H_{t-1} - Z_t>, dW = sum_t H_{t-1}^T D_t, dw_r = sum_t u_t v_t.
//
// One CTA per chain (b, n); the 128 key rows form two groups of 64 (one
// epilogue warpgroup each), and epilogue thread L of a group owns value
// column j = L (TMEM lane L) of the group's 64 rows.  Every matrix product
// runs on the tensor core (one MMA warp issues them all):
//   rerun (per chunk, forward in time, from the chunk's checkpoint): the
//     forward's step, D^T = W^T H_{t-1}^T + v_t k_t^T (A = fp16 W^T and the
//     rank-1 column in TMEM, B = fp16 H^T tile in shared memory); the
//     epilogue applies tanh and the gate blend and writes fp16 Z_t and
//     H_{t-1} to a per-chain chunk cache in global memory (64 KB per step,
//     chunks short enough for the cache of every chain to stay in L2);
//   reverse walk (backward in time): the state gradient C lives in the
//     tensor-memory accumulator.  The epilogue reads C_t, forms R = C + q u^T,
//     D = R (1 - f)(1 - Z^2) and the df share <R, H_{t-1} - Z>, writes f R
//     back into the accumulator and bf16 D and H_{t-1} tiles into shared
//     memory; the tensor core then adds W D^T (A = bf16 W in TMEM) to form
//     C_{t-1}, and from the same tiles forms dW += H_{t-1}^T D (accumulated
//     in TMEM), dv = D^T k, dk = D v and dq_t = H_t u_t (u split into bf16
//     hi + lo parts), each a small MMA with N = 16 whose result lands in TMEM
//     lane = output index.
// The bf16 tiles use one core-matrix layout (thread j writes its column's
// rows as 16-byte runs); the operands read them as MN-major (rows
// contiguous) or K-major (the contraction over rows contiguous) as each
// product needs.  Every wait is bounded (ptx.cuh).
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
constexpr int kK = 128;
constexpr int kNR = 64;          // rows per group
constexpr int kMaxC = 16;        // chunk length limit (shared memory: the chunk input buffers)
constexpr int kThreads = 320;    // 8 epilogue warps, the MMA warp, the TMA producer
constexpr int kMmaWarp = 8;  // warp 9: the TMA producer

// Tensor memory columns (512 allocated).
constexpr uint32_t kAcc = 0;      // [2 groups][64]: rerun D^T, reverse C^T (lane = value column)
constexpr uint32_t kDW = 128;     // [128]: dW (lane m, column j)
constexpr uint32_t kARR = 256;    // [64]: A = fp16 W^T (lane L: W[m][L], two per column)
constexpr uint32_t kAX = 320;     // [2][8]: rerun rank-1 column [v_t, 0 ...] per group
constexpr uint32_t kACH = 336;    // [64]: A = bf16 W (lane L: W[L][j])
constexpr uint32_t kSmall = 400;  // [2 buffers][dk 16 | dv 16 | dq 16]
constexpr uint32_t kTmemCols = 512;

// Shared memory (offsets from the 1 KB aligned base).
constexpr uint32_t kKB = kV + 16;                      // rerun B: H^T K-rows + the rank-1 slice
constexpr uint32_t kRBBytes = kNR * kKB * 2;           // 18432 per group
constexpr uint32_t kRBSbo = kKB * 16;                  // 2304: next 8 rows (N)
constexpr uint32_t kTileBytes = kNR * kV * 2;          // 16384: a bf16 D or H tile of one group
constexpr uint32_t kTileSbo = kV * 16;                 // 2048: next 8 rows
constexpr uint32_t kRB = 0;                            // [2 groups]
constexpr uint32_t kDT = kRB + 2 * kRBBytes;           // [2 parities][2 groups]
constexpr uint32_t kHT = kDT + 4 * kTileBytes;         // [2 parities][2 groups]
constexpr uint32_t kKT = kHT + 4 * kTileBytes;         // [2 groups] k tiles: K = 64 rows x N = 16, K-major
constexpr uint32_t kVT = kKT + 2 * 2048;               // v tile: K = 128 x N = 16, K-major
constexpr uint32_t kUT = kVT + 4096;                   // u tile: K = 128 x N = 16, MN-major
constexpr uint32_t kCB = kUT + 4096;                   // chunk input buffers

struct Tc128Params {
  BwdArgs a;
  int nchunks;
  uint32_t cbuf_bytes, cq_off, ck_off, cv_off, cdy_off, cf_off;
  uint32_t red_off, bar_off, misc_off;
  uint32_t tx_bytes;
  uint4* cache;  // [chain][C steps][Z | H][2 groups][8 runs][128 threads] x 16 bytes
  float* csave;  // [chain][2 groups][64 rows][128 threads]: the state gradient across a rerun
};

// One core-matrix tile (K = value column j, N = row r of a group): element
// (j, r) at (r / 8) * 2048 + (j / 8) * 128 + (j % 8) * 16 + (r % 8) * 2.
__device__ __forceinline__ uint32_t tile_run(int j, int r8) {  // the 16-byte run of rows 8 r8 .. 8 r8 + 7
  return static_cast<uint32_t>(r8 * kTileSbo + (j >> 3) * 128 + (j & 7) * 16);
}

// Shared-memory matrix descriptor; lbo = byte step along K, sbo = byte step
// along M / N (both for K-major and MN-major operands, no swizzle).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return smem_desc_noswizzle(addr, lbo, sbo);
}

// x as bf16 hi + lo (hi in the low half).
__device__ __forceinline__ uint32_t bf16_hi_lo(float x) {
  const uint32_t hb = pack_bf16x2(x, 0.f) & 0xFFFFu;
  const float lo = x - __uint_as_float(hb << 16);
  return hb | (pack_bf16x2(lo, 0.f) << 16);
}

// Bring `bytes` (a multiple of 16) at a 16-byte aligned global address into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// Drop a 128-byte line from L2 without writing it back (its data is dead:
// the chunk cache is rewritten before it is read again).
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}

// Sum over the 32 lanes, in every lane, on the tensor core (see the V = 64
// backward): bf16 hi + lo of each lane's value against ones, twice.
__device__ __forceinline__ float warp_sum_tc(float x) {
  const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  mma_bf16_16816(d, ones, bf16_hi_lo(x), 0u);
  const uint32_t h0 = bf16_hi_lo(d[0]), h1 = bf16_hi_lo(d[1]);
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  mma_bf16_16816(e, ones, (h0 & 0xFFFFu) | (h1 << 16), (h0 >> 16) | (h1 & 0xFFFF0000u));
  return e[0];
}

template <bool kClip>
__global__ void __launch_bounds__(kThreads, 1) tc_backward128_kernel(const __grid_constant__ Tc128Params p,
                                                                     const __grid_constant__ CUtensorMap tm_q,
                                                                     const __grid_constant__ CUtensorMap tm_k,
                                                                     const __grid_constant__ CUtensorMap tm_v,
                                                                     const __grid_constant__ CUtensorMap tm_dy) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const BwdArgs& A = p.a;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int T = A.T, N = A.N, CL = A.ckpt_every;
  const int chain = blockIdx.x, b = chain / N, n = chain % N;
  StatusBlock* status = A.status;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* hready = bars;        // [2] rerun: epilogue group -> MMA warp (4 warps)
  uint64_t* dready = bars + 2;    // [2] reverse: epilogue group -> MMA warp (4 warps)
  uint64_t* dfull = bars + 4;     // [2] MMA warp -> epilogue group (commit)
  uint64_t* cfull = bars + 6;     // [2] chunk inputs landed (producer lanes + TMA bytes)
  uint64_t* cempty = bars + 8;    // [2] chunk inputs free (8 epilogue warps)
  uint64_t* dwdone = bars + 11;   // every MMA has completed (commit)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 8);
  unsigned int* done_ctr = reinterpret_cast<unsigned int*>(smem + p.misc_off + 12);  // warps done with a chunk
  float* red = reinterpret_cast<float*>(smem + p.red_off);  // [kMaxC][8]: df partials per warp

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&hready[i]), 4);
      mbar_init(smem_u32(&dready[i]), 4);
      mbar_init(smem_u32(&dfull[i]), 1);
      mbar_init(smem_u32(&cfull[i]), 32);
      mbar_init(smem_u32(&cempty[i]), 8);
    }
    mbar_init(smem_u32(dwdone), 1);
    *abort_flag = 0;
    *done_ctr = 0u;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // Zero every tile once (H_0 = 0 where no start state is given, the rank-1
  // slice's rows beyond the first, the unused columns of the k, v, u tiles).
  for (uint32_t e = threadIdx.x * 16; e < kCB; e += kThreads * 16)
    *reinterpret_cast<uint4*>(smem + e) = make_uint4(0u, 0u, 0u, 0u);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // A operands in tensor memory, written once: fp16 W^T (rerun) and bf16 W
  // (reverse chain); lane L of warp w's quadrant.  Range check of the fp16
  // re-encoding as in the forward.
  if (warp < 4) {
    const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
    const int L = 32 * warp + lane;
    const uint32_t lq = static_cast<uint32_t>(32 * warp) << 16;
#pragma unroll 1
    for (int c0 = 0; c0 < kV / 2; c0 += 32) {
      uint32_t rr[32], rc[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int m = 2 * (c0 + u);
        rr[u] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[m * kV + L]) |
                                (static_cast<uint32_t>(Wg[(m + 1) * kV + L]) << 16));
        if (!f16x2_finite(rr[u])) report_device_error(status, kStatusCheck, kWhereWRange);
        rc[u] = *reinterpret_cast<const uint32_t*>(Wg + L * kV + m);
      }
      tmem_st_32x32b_x32(tmem_base + lq + kARR + c0, rr);
      tmem_st_32x32b_x32(tmem_base + lq + kACH + c0, rc);
    }
    // The rank-1 columns of both groups: every element but the first of each
    // lane stays zero (the slice's B rows beyond the first are zero too, but
    // uninitialised tensor memory could hold non-finite values).
    const uint32_t zeros[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st_32x32b_x16(tmem_base + lq + kAX, zeros);
    tmem_st_wait();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  if (warp < 8) {
    // ======================= epilogue warpgroups =======================
    const int g = warp >> 2, wq = warp & 3;
    const int j = 32 * wq + lane;  // value column, TMEM lane
    const uint32_t lq = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t tacc = tmem_base + lq + kAcc + kNR * g;
    const uint32_t hbar = smem_u32(&hready[g]), dbar = smem_u32(&dready[g]), fbar = smem_u32(&dfull[g]);
    uint32_t fphase = 0;  // parity of dfull[g]
    const int64_t row0 = static_cast<int64_t>(chain) * kK + kNR * g;  // first state row of the group
    const uint16_t* wrg = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    const float wrj = bf16_bits_to_f32(wrg[j]);
    uint4* const cache_c = p.cache + static_cast<int64_t>(chain) * CL * 2 * 2 * 8 * 128;
    float* const save = p.csave + (static_cast<int64_t>(chain) * 2 + g) * kNR * 128 + j;
    float dwr = 0.f;
    bool ok = true;
    int rs = 0;          // reverse steps done
    int64_t prev_t = -1; // time index of the reverse step whose small products are pending (group 1 reads them)
    int prev_s = 0;      // its index in the chunk (its u_t is in the chunk's input buffer)
    const float* cdy_cur = nullptr;

    auto wait_mma = [&]() -> bool {
      const bool w_ok = mbar_wait(fbar, fphase, abort_flag, status, kWhereBwdDW);
      fphase ^= 1u;
      tc_fence_after_sync();
      return w_ok;
    };
    // Group 1 writes out the small products of reverse step prev_t (buffer
    // (rs - 1) & 1): dk (lane = row), dv (lane = column), dq (lane = row,
    // hi and lo parts).
    auto read_small = [&]() {
      if (g != 1 || prev_t < 0) return;
      const uint32_t sb = tmem_base + lq + kSmall + 48u * static_cast<uint32_t>((rs - 1) & 1);
      uint32_t dk2[2], dv2[2], dq2[2];
      tmem_ld_32x32b<2>(sb, dk2);
      tmem_ld_32x32b<2>(sb + 16, dv2);
      tmem_ld_32x32b<2>(sb + 32, dq2);
      tmem_ld_wait();
      tmem_ld_fence_regs(dk2);
      tmem_ld_fence_regs(dv2);
      tmem_ld_fence_regs(dq2);
      const int64_t rowt = (static_cast<int64_t>(b) * T + prev_t) * N + n;
      A.dk[rowt * kK + j] = __uint_as_float(dk2[0]);
      A.dq[rowt * kK + j] = __uint_as_float(dq2[0]) + __uint_as_float(dq2[1]);
      const float uj = cdy_cur[prev_s * kV + j];
      A.dv[rowt * kV + j] = fmaf(wrj, uj, __uint_as_float(dv2[0]));
      prev_t = -1;
    };

    for (int ci = 0; ci < p.nchunks && ok; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL, L = min(CL, T - s0);
      const int cb = ci & 1;
      if (!mbar_wait(smem_u32(&cfull[cb]), (ci >> 1) & 1, abort_flag, status, kWhereBwdFull)) {
        ok = false;
        break;
      }
      const uint8_t* cbuf = smem + kCB + cb * p.cbuf_bytes;
      const uint16_t* cq = reinterpret_cast<const uint16_t*>(cbuf + p.cq_off);  // [C][128]
      const uint16_t* ck = reinterpret_cast<const uint16_t*>(cbuf + p.ck_off);
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(cbuf + p.cv_off);
      const float* cdy = reinterpret_cast<const float*>(cbuf + p.cdy_off);
      const float* cf = reinterpret_cast<const float*>(cbuf + p.cf_off);
      cdy_cur = cdy;

      // ---------------- rerun of the chunk (Eq. 10-11) ----------------
      float h[kNR];
      {
        const float* src = (c == 0) ? (A.H0 != nullptr ? A.H0 + row0 * kV + j : nullptr)
                                    : A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (c - 1)) * kK + kNR * g) * kV + j;
#pragma unroll
        for (int r = 0; r < kNR; ++r) h[r] = src != nullptr ? src[static_cast<int64_t>(r) * kV] : 0.f;
      }
      uint8_t* const rb = smem + kRB + g * kRBBytes + (j >> 3) * 128 + (j & 7) * 16;  // thread j's K-row of B
      auto put_h = [&]() {  // fp16 H as the rerun's B operand
#pragma unroll
        for (int r8 = 0; r8 < kNR / 8; ++r8)
          *reinterpret_cast<uint4*>(rb + r8 * kRBSbo) =
              make_uint4(pack2_f16(h[8 * r8], h[8 * r8 + 1]), pack2_f16(h[8 * r8 + 2], h[8 * r8 + 3]),
                         pack2_f16(h[8 * r8 + 4], h[8 * r8 + 5]), pack2_f16(h[8 * r8 + 6], h[8 * r8 + 7]));
      };
      auto put_x = [&](int s) {  // rank-1 slice of step s: A column [v_s, 0..], B row k_s
        tmem_st_x1(tmem_base + lq + kAX + 8 * g, static_cast<uint32_t>(cv[s * kV + j]));
        if (j < kNR / 8)
          *reinterpret_cast<uint4*>(smem + kRB + g * kRBBytes + j * kRBSbo + kV * 16) =
              *reinterpret_cast<const uint4*>(ck + s * kK + kNR * g + 8 * j);
      };
      auto hand_over = [&](uint32_t bar) {
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
      };
      put_h();
      put_x(0);
      hand_over(hbar);
      for (int s = 0; s < L; ++s) {
        if (!wait_mma()) {
          ok = false;
          break;
        }
        uint4* const cz = cache_c + ((static_cast<int64_t>(s) * 2 + 0) * 2 + g) * 8 * 128 + j;
        uint4* const chh = cache_c + ((static_cast<int64_t>(s) * 2 + 1) * 2 + g) * 8 * 128 + j;
        const float omf = 1.f - cf[s];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t acc[32];
          tmem_ld_32x32b<32>(tacc + 32 * half, acc);
          tmem_ld_wait();
          tmem_ld_fence_regs(acc);
#pragma unroll
          for (int r8 = 0; r8 < 4; ++r8) {
            const int rr = 32 * half + 8 * r8;
            float z[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) z[u] = tanh_fast(__uint_as_float(acc[8 * r8 + u]));
            chh[(4 * half + r8) * 128] = make_uint4(pack2_f16(h[rr], h[rr + 1]), pack2_f16(h[rr + 2], h[rr + 3]),
                                                    pack2_f16(h[rr + 4], h[rr + 5]), pack2_f16(h[rr + 6], h[rr + 7]));
            cz[(4 * half + r8) * 128] = make_uint4(pack2_f16(z[0], z[1]), pack2_f16(z[2], z[3]),
                                                   pack2_f16(z[4], z[5]), pack2_f16(z[6], z[7]));
#pragma unroll
            for (int u = 0; u < 8; ++u) h[rr + u] = fmaf(omf, z[u] - h[rr + u], h[rr + u]);
          }
        }
        if (s + 1 < L) {
          put_h();
          put_x(s + 1);
          hand_over(hbar);
        }
      }
      if (!ok) break;
      // H_{L-1} (after the chunk's last step) as the bf16 H tile that the
      // reverse walk's first dq product reads (parity L & 1).  That product
      // is issued in group 0's turn, which no hand-over of group 1 precedes
      // in this chunk: group 1 signals its tile on hready (one arrival more
      // than its rerun steps) and the MMA warp waits for it.
      {
        uint8_t* ht = smem + kHT + ((L & 1) * 2 + g) * kTileBytes;
#pragma unroll
        for (int r8 = 0; r8 < kNR / 8; ++r8)
          *reinterpret_cast<uint4*>(ht + tile_run(j, r8)) =
              make_uint4(pack2_bf16(h[8 * r8], h[8 * r8 + 1]), pack2_bf16(h[8 * r8 + 2], h[8 * r8 + 3]),
                         pack2_bf16(h[8 * r8 + 4], h[8 * r8 + 5]), pack2_bf16(h[8 * r8 + 6], h[8 * r8 + 7]));
      }
      if (g == 1) hand_over(hbar);

      // ---------------- reverse walk over the chunk ----------------
      // The next chunk's start state (its group's 64 rows, 32 KB) into L2.
      if (c > 1 && wq == 0 && lane == 0)
        prefetch_l2(A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (c - 2)) * kK + kNR * g) * kV,
                    kNR * kV * 4);
      for (int s = L - 1; s >= 0; --s, ++rs) {
        const int64_t t = s0 + s;
        const int par = s & 1;
        // The step's cached Z_t and H_{t-1}: all sixteen loads issued first.
        const uint4* const cz = cache_c + ((static_cast<int64_t>(s) * 2 + 0) * 2 + g) * 8 * 128 + j;
        const uint4* const chh = cache_c + ((static_cast<int64_t>(s) * 2 + 1) * 2 + g) * 8 * 128 + j;
        uint4 zq[8], hq[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          zq[i] = cz[i * 128];
          hq[i] = chh[i * 128];
        }
        // The next step back's cache of this group (Z and H, 16 KB each) into L2.
        if (s > 0 && wq == 0 && lane == 0) {
          prefetch_l2(cz - 2 * 2 * 8 * 128 - j, 16384);
          prefetch_l2(chh - 2 * 2 * 8 * 128 - j, 16384);
        }
        // C_t: the accumulator after the previous reverse step, or (first
        // step of a chunk) the copy kept across the rerun / dH_T.
        const bool first = (s == L - 1);
        if (!first) {
          if (!wait_mma()) {
            ok = false;
            break;
          }
          read_small();
        }
        const float ft = cf[s], omf = 1.f - ft;
        const float uj = cdy[s * kV + j];
        const float2 u2 = make_float2(uj, uj);
        float dfs = 0.f;
        uint8_t* const dtile = smem + kDT + (par * 2 + g) * kTileBytes;
        uint8_t* const htile = smem + kHT + (par * 2 + g) * kTileBytes;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t cw[32];
          if (first) {
            if (ci == 0) {
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const int r = 32 * half + u;
                cw[u] = __float_as_uint(A.dH_T != nullptr ? A.dH_T[(row0 + r) * kV + j] : 0.f);
              }
            } else {
#pragma unroll
              for (int u = 0; u < 32; ++u) cw[u] = __float_as_uint(save[(32 * half + u) * 128]);
            }
          } else {
            tmem_ld_32x32b<32>(tacc + 32 * half, cw);
            tmem_ld_wait();
            tmem_ld_fence_regs(cw);
            if constexpr (kClip) {  // the newly formed C_t (the caller's dH_T is not clipped)
#pragma unroll
              for (int u = 0; u < 32; ++u) cw[u] = __float_as_uint(fminf(fmaxf(__uint_as_float(cw[u]), -A.clip), A.clip));
            }
          }
          uint32_t fr[32];
#pragma unroll
          for (int r8 = 0; r8 < 4; ++r8) {
            const int rr = 32 * half + 8 * r8;
            const uint4 zw = zq[4 * half + r8], hw = hq[4 * half + r8];
            const uint32_t zwa[4] = {zw.x, zw.y, zw.z, zw.w}, hwa[4] = {hw.x, hw.y, hw.z, hw.w};
            const uint4 qv = *reinterpret_cast<const uint4*>(cq + s * kK + kNR * g + rr);
            const uint32_t qwa[4] = {qv.x, qv.y, qv.z, qv.w};
            uint32_t dpk[4], hpk[4];
#pragma unroll
            for (int u2i = 0; u2i < 4; ++u2i) {
              const float2 C2 = make_float2(__uint_as_float(cw[8 * r8 + 2 * u2i]), __uint_as_float(cw[8 * r8 + 2 * u2i + 1]));
              const float2 q2 = make_float2(bf16lo(qwa[u2i]), bf16hi(qwa[u2i]));
              const float2 Rv = __ffma2_rn(q2, u2, C2);                        // R = C + q u^T
              const float2 z = f16x2_to_float2(zwa[u2i]), hp = f16x2_to_float2(hwa[u2i]);
              const float2 zz = __fmul2_rn(z, z);
              const float2 G = __ffma2_rn(make_float2(-omf, -omf), zz, make_float2(omf, omf));  // (1-f)(1-Z^2)
              const float2 D = __fmul2_rn(Rv, G);
              const float2 E = __ffma2_rn(z, make_float2(-1.f, -1.f), hp);     // H_{t-1} - Z
              const float2 pe = __fmul2_rn(Rv, E);
              dfs += pe.x + pe.y;
              const float2 fR = __fmul2_rn(make_float2(ft, ft), Rv);
              fr[8 * r8 + 2 * u2i] = __float_as_uint(fR.x);
              fr[8 * r8 + 2 * u2i + 1] = __float_as_uint(fR.y);
              dpk[u2i] = pack2_bf16(D.x, D.y);
              hpk[u2i] = pack2_bf16(hp.x, hp.y);
            }
            const int r8g = 4 * half + r8;
            *reinterpret_cast<uint4*>(dtile + tile_run(j, r8g)) = make_uint4(dpk[0], dpk[1], dpk[2], dpk[3]);
            *reinterpret_cast<uint4*>(htile + tile_run(j, r8g)) = make_uint4(hpk[0], hpk[1], hpk[2], hpk[3]);
          }
          tmem_st_32x32b_x32(tacc + 32 * half, fr);  // f R: the chain MMA accumulates D W^T on it
        }
        // The small products' B operands: k_t of the group's rows (K-major,
        // column 0), and (group 0) u_t as bf16 hi / lo (MN-major, columns
        // 0 and 1), (group 1) v_t (K-major, column 0).
        if (j < kNR / 8)
          *reinterpret_cast<uint4*>(smem + kKT + g * 2048 + j * 256) =
              *reinterpret_cast<const uint4*>(ck + s * kK + kNR * g + 8 * j);
        if (g == 0) {
          const uint32_t hl = bf16_hi_lo(uj);
          *reinterpret_cast<uint4*>(smem + kUT + (j >> 3) * 128 + (j & 7) * 16) = make_uint4(hl, 0u, 0u, 0u);
          dwr = fmaf(uj, bf16_bits_to_f32(cv[s * kV + j]), dwr);
        } else if (j < kV / 8) {
          *reinterpret_cast<uint4*>(smem + kVT + j * 256) = *reinterpret_cast<const uint4*>(cv + s * kV + 8 * j);
        }
        hand_over(dbar);
        // This warp's cache lines of the step (every lane's loads consumed
        // above) leave L2 without a write-back: lanes 0-7 take the Z lines,
        // 8-15 the H lines, two each.
        if (lane < 16) {
          const uint4* base = (lane < 8 ? cz : chh) - j + 32 * wq;
          const int i2 = lane & 7;
          discard_l2(base + i2 * 128);
          discard_l2(base + i2 * 128 + 8);
          discard_l2(base + i2 * 128 + 16);
          discard_l2(base + i2 * 128 + 24);
        }
        const float wsum = warp_sum_tc(dfs);
        if (lane == 0) red[s * 8 + warp] = wsum;
        prev_t = t;
        prev_s = s;
      }
      if (!ok) break;
      // End of the chunk's walk: C_{s0 - 1} is the start of the next chunk's
      // walk (kept in global memory across its rerun), or dH_0.
      if (!wait_mma()) {
        ok = false;
        break;
      }
      read_small();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t cw[32];
        tmem_ld_32x32b<32>(tacc + 32 * half, cw);
        tmem_ld_wait();
        tmem_ld_fence_regs(cw);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          float x = __uint_as_float(cw[u]);
          if constexpr (kClip) x = fminf(fmaxf(x, -A.clip), A.clip);
          const int r = 32 * half + u;
          if (c > 0)
            save[r * 128] = x;
          else if (A.dH0 != nullptr)
            A.dH0[(row0 + r) * kV + j] = x;
        }
      }
      // df_t of the chunk: the last warp to finish its walk sums the eight
      // warp partials in a fixed order (no warp waits for the others; none
      // can overwrite the partials before the sum: the next chunk's walk
      // follows a rerun whose MMAs wait for every group, the summing warp's
      // included, and that warp sums before it joins the rerun).
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(done_ctr, 1u) == 7u;
        if (last) {
          *done_ctr = 0u;
          __threadfence_block();
        }
        mbar_arrive(smem_u32(&cempty[cb]));
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        for (int s = lane; s < L; s += 32) {
          float d = 0.f;
#pragma unroll
          for (int w8 = 0; w8 < 8; ++w8) d += red[s * 8 + w8];
          A.df[(static_cast<int64_t>(b) * T + s0 + s) * N + n] = d;
        }
        __syncwarp();
      }
    }
    if (ok && g == 0) A.dwr_part[static_cast<int64_t>(chain) * kV + j] = dwr;
    if (!ok) *abort_flag = 1;
  } else if (warp == kMmaWarp) {
    // ======================= MMA warp =======================
    const uint32_t idesc_rr = idesc_f16_f32(128, kNR, /*a_mn_major=*/false, /*b_mn_major=*/true);
    const uint32_t idesc_x = idesc_bf16_f32(128, kNR, false, true);
    const uint32_t idesc_ch = idesc_bf16_f32(128, kNR, false, true);
    const uint32_t idesc_dw = idesc_bf16_f32(128, kV, false, false);
    const uint32_t idesc_dv = idesc_bf16_f32(128, 16, false, false);
    const uint32_t idesc_dk = idesc_bf16_f32(128, 16, true, false);
    const uint32_t idesc_dq = idesc_bf16_f32(128, 16, true, true);
    uint32_t hph = 0u, dph = 0u;  // bit g: phase of hready[g], dready[g]
    bool ok = true;
    int rs = 0;
    for (int ci = 0; ci < p.nchunks && ok; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int L = min(CL, T - c * CL);
      // rerun
      for (int s = 0; s < L && ok; ++s) {
        for (int g = 0; g < 2; ++g) {
          if (!mbar_wait(smem_u32(&hready[g]), (hph >> g) & 1u, abort_flag, status, kWhereBwdTReady)) {
            ok = false;
            break;
          }
          hph ^= 1u << g;
          if (elect_one()) {
            tc_fence_after_sync();
            const uint32_t bg = sbase + kRB + g * kRBBytes;
            const uint32_t acc = tmem_base + kAcc + kNR * g;
            tc_mma_f16_ts(acc, tmem_base + kAX + 8 * g, sdesc(bg + (kV / 8) * 128, 128, kRBSbo), idesc_x, 0u);
#pragma unroll
            for (int kk = 0; kk < kV / 16; ++kk)
              tc_mma_f16_ts(acc, tmem_base + kARR + 8 * kk, sdesc(bg + kk * 256, 128, kRBSbo), idesc_rr, 1u);
            tc_commit(smem_u32(&dfull[g]));
          }
          __syncwarp();
        }
      }
      // reverse
      for (int s = L - 1; s >= 0 && ok; --s, ++rs) {
        // Group 1's H_{L-1} tile is written (read by the first step's dq
        // product in group 0's turn; group 0's own is ordered by its hand-over).
        if (s == L - 1) {
          if (!mbar_wait(smem_u32(&hready[1]), (hph >> 1) & 1u, abort_flag, status, kWhereBwdTReady)) {
            ok = false;
            break;
          }
          hph ^= 2u;
        }
        const int par = s & 1;
        const uint32_t sb = tmem_base + kSmall + 48u * static_cast<uint32_t>(rs & 1);
        for (int g = 0; g < 2; ++g) {
          if (!mbar_wait(smem_u32(&dready[g]), (dph >> g) & 1u, abort_flag, status, kWhereBwdXFull)) {
            ok = false;
            break;
          }
          dph ^= 1u << g;
          if (elect_one()) {
            tc_fence_after_sync();
            const uint32_t dt = sbase + kDT + (par * 2 + g) * kTileBytes;
            const uint32_t ht = sbase + kHT + (par * 2 + g) * kTileBytes;
            // C_{t-1}^T (+)= W D^T: A = W (TMEM), B = D^T of the group (MN-major).
#pragma unroll
            for (int kk = 0; kk < kV / 16; ++kk)
              tc_mma_f16_ts(tmem_base + kAcc + kNR * g, tmem_base + kACH + 8 * kk, sdesc(dt + kk * 256, 128, kTileSbo),
                            idesc_ch, 1u);
            // dW += H_{t-1}^T D over the group's rows: both K-major (rows contiguous).
#pragma unroll
            for (int kk = 0; kk < kNR / 16; ++kk)
              tc_mma_f16_ss(tmem_base + kDW, sdesc(ht + kk * 2 * kTileSbo, kTileSbo, 128),
                            sdesc(dt + kk * 2 * kTileSbo, kTileSbo, 128), idesc_dw, (rs > 0 || g > 0 || kk > 0) ? 1u : 0u);
            // dv_t = D^T k_t: A = D^T (K-major), B = k_t of the group's rows (K-major, column 0).
#pragma unroll
            for (int kk = 0; kk < kNR / 16; ++kk)
              tc_mma_f16_ss(sb + 16, sdesc(dt + kk * 2 * kTileSbo, kTileSbo, 128),
                            sdesc(sbase + kKT + g * 2048 + kk * 512, 256, 128), idesc_dv, (g > 0 || kk > 0) ? 1u : 0u);
            if (g == 0) {
              // dq_t = H_t u_t: A = H_t of both groups (written one step later
              // in time, parity (s + 1) & 1; MN-major, M = 128 rows), B = u_t
              // hi / lo (MN-major, columns 0 and 1).
              const uint32_t hq = sbase + kHT + ((par ^ 1) * 2) * kTileBytes;
#pragma unroll
              for (int kk = 0; kk < kV / 16; ++kk)
                tc_mma_f16_ss(sb + 32, sdesc(hq + kk * 256, 128, kTileSbo), sdesc(sbase + kUT + kk * 256, 128, 2048),
                              idesc_dq, kk > 0 ? 1u : 0u);
            } else {
              // dk_t = D_t v_t: A = D of both groups (MN-major, M = 128 rows), B = v_t (K-major, column 0).
              const uint32_t d0 = sbase + kDT + (par * 2) * kTileBytes;
#pragma unroll
              for (int kk = 0; kk < kV / 16; ++kk)
                tc_mma_f16_ss(sb, sdesc(d0 + kk * 256, 128, kTileSbo), sdesc(sbase + kVT + kk * 512, 256, 128), idesc_dk,
                              kk > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&dfull[g]));
          }
          __syncwarp();
        }
      }
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ======================= TMA producer (chunks, last first) =======================
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
      const int cb = ci & 1;
      if (ci >= 2 && !mbar_wait(smem_u32(&cempty[cb]), ((ci >> 1) - 1) & 1, abort_flag, status, kWhereBwdCEmpty)) {
        ok = false;
        break;
      }
      uint8_t* buf = smem + kCB + cb * p.cbuf_bytes;
      const int t0 = c * CL;
      const int t = t0 + lane;
      const float fv = (lane < CL && t < T) ? gate_value(gs, (static_cast<int64_t>(b) * T + t) * N + n, n) : 0.f;
      if (lane < CL) reinterpret_cast<float*>(buf + p.cf_off)[lane] = fv;
      __syncwarp();
      const uint32_t fb = smem_u32(&cfull[cb]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, p.tx_bytes);
        tma_load_4d(smem_u32(buf + p.cq_off), &tm_q, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.ck_off), &tm_k, fb, 0, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.cv_off), &tm_v, fb, 0, n, t0, b);
        tma_load_4d(smem_u32(buf + p.cdy_off), &tm_dy, fb, 0, n, t0, b);
      } else {
        mbar_arrive(fb);
      }
      issued = ci + 1;
    }
    if (!ok) {  // every issued copy lands before the CTA can exit
      for (int ci = std::max(0, issued - 2); ci < issued; ++ci)
        mbar_wait_timed(smem_u32(&cfull[ci & 1]), (ci >> 1) & 1, nullptr, kWhereBwdDrain);
    }
  }

  // dW of the chain from tensor memory once every MMA has completed.
  if (warp == kMmaWarp) {
    if (elect_one()) tc_commit(smem_u32(dwdone));
    __syncwarp();
  }
  if (warp < 4) {
    const bool done = mbar_wait(smem_u32(dwdone), 0, abort_flag, status, kWhereBwdDW);
    tc_fence_after_sync();
    if (done && !*abort_flag) {
      float* dst = A.dW_part + static_cast<int64_t>(chain) * kV * kV + (32 * warp + lane) * kV;
#pragma unroll 1
      for (int c0 = 0; c0 < kV; c0 += 32) {
        uint32_t r[32];
        tmem_ld_32x32b<32>(tmem_base + (static_cast<uint32_t>(32 * warp) << 16) + kDW + c0, r);
        tmem_ld_wait();
        tmem_ld_fence_regs(r);
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(dst + c0 + u) = make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                                                                 __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <bool kClip>
cudaError_t launch_t(const BwdArgs& a, uint4* cache, float* csave, cudaStream_t s) {
  Tc128Params p{};
  p.a = a;
  const int C = a.ckpt_every;
  p.nchunks = (a.T + C - 1) / C;
  p.cq_off = 0;
  p.ck_off = align_up(C * kK * 2, 128);
  p.cv_off = p.ck_off + align_up(C * kK * 2, 128);
  p.cdy_off = p.cv_off + align_up(C * kV * 2, 128);
  p.cf_off = p.cdy_off + align_up(C * kV * 4, 128);
  p.cbuf_bytes = align_up(p.cf_off + 32 * 4, 128);
  p.red_off = kCB + 2 * p.cbuf_bytes;
  p.bar_off = align_up(p.red_off + kMaxC * 8 * 4, 8);
  p.misc_off = p.bar_off + 12 * 8;
  p.tx_bytes = 2 * C * kK * 2 + C * kV * 2 + C * kV * 4;
  p.cache = cache;
  p.csave = csave;
  const uint32_t smem = align_up(p.misc_off + 16, 128) + 1024;

  CUtensorMap mq, mk, mv, mdy;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, kK, kK, C) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, kK, kK, C) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, C) ||
      !make_tensor_map_btnx(&mdy, a.dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.N, kV, kV, C))
    return cudaErrorInvalidValue;
  auto kern = tc_backward128_kernel<kClip>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<a.B * a.N, kThreads, smem, s>>>(p, mq, mk, mv, mdy);
  return cudaGetLastError();
}

}  // namespace

bool tc_backward128_supported(int K, int V, int ckpt_every) {
  return K == kK && V == kV && ckpt_every >= 1 && ckpt_every <= kMaxC;
}

// The chunk cache (fp16 Z_t and H_{t-1} of every step of a chunk, 64 KB per
// step) and the state gradient kept across each rerun (64 KB), per chain.
size_t tc_backward128_scratch_bytes(int B, int N, int ckpt_every) {
  const size_t chains = static_cast<size_t>(B) * N;
  return chains * static_cast<size_t>(ckpt_every) * 2 * kK * kV * 2 + chains * kK * kV * 4;
}

cudaError_t launch_tc_backward128(const BwdArgs& a, cudaStream_t s) {
  if (!tc_backward128_supported(a.K, a.V, a.ckpt_every) || a.dtype != M2RNN_BF16) return cudaErrorInvalidValue;
  const size_t chains = static_cast<size_t>(a.B) * a.N;
  uint4* cache = reinterpret_cast<uint4*>(a.scratch);
  float* csave = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.scratch) +
                                          chains * static_cast<size_t>(a.ckpt_every) * 2 * kK * kV * 2);
  return a.clip > 0.f ? launch_t<true>(a, cache, csave, s) : launch_t<false>(a, cache, csave, s);
}

}  // namespace m2rnn
