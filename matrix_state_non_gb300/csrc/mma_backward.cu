// Register-resident backward-through-time for V = 64 value columns (bf16
// inputs, fp32 state and gradients).
//
// Chain rule for Eq. 10-12 as derived in section 2.7 of the reading notes on
// "M2RNN: Non-Linear RNNs with Matrix-Valued States for Scalable Language
// Modeling" (the notes' correction of the paper's Algorithm 2), with the
// value-residual terms restored; u_t = dy_t, C_T = dH_T:
//   R_t = C_t + q_t u_t^T,  D_t = ((1-f_t) R_t) * (1 - Z_t * Z_t),
//   C_{t-1} = f_t R_t + D_t W^T,
//   dq_t = H_t u_t, dk_t = D_t v_t, dv_t = D_t^T k_t + w_r * u_t,
//   df_t = <R_t, H_{t-1} - Z_t>,  dW += H_{t-1}^T D_t,  dw_r += u_t * v_t.
//
// Work split as in the forward: a chain's K rows in blocks of 16, one CTA per
// block (rows never mix; only dv_t, df_t, dW and dw_r sum over rows, and
// those are written as row-block partials and summed afterwards in a fixed
// order).  The time axis runs over chunks of C <= 20 steps, last chunk first;
// for each chunk the forward is rebuilt from its checkpoint (section 2.6 of
// the notes describes the paper's rerun-and-cache backward; here only two
// chunks are cached, on chip) and then walked backwards.  Three warpgroups:
//   reverse warps   (each owning 16 value columns) the serial chain:
//                   R -> D = R * G -> bf16(D) tile -> one named barrier -> 8
//                   warp MMAs seeded with f R -> C_{t-1}; besides it only the
//                   df share <R, E>, handed to the gradient warps with the D
//                   tile through a ring of shared-memory slots;
//   recompute warps (each owning 16 value columns) the rebuild of the next
//                   chunk: Eq. 10-11 rerun, or, when the forward left its Z_t
//                   in a stash (fp16), only H_t = H_{t-1} + (1-f_t)(Z_t -
//                   H_{t-1}) from the chunk's checkpoint with Z_t bulk-copied
//                   a chunk at a time.  Per step and thread they cache in
//                   their own tensor-memory lanes what the reverse walk needs,
//                   G = (1-f)(1-Z^2) and E = H_{t-1} - Z (fp16), and write
//                   bf16 H_{t-1} tiles for the dW MMA into a chunk buffer in
//                   shared memory; they also form dq_t = H_t u_t (per-thread
//                   shares summed at the chunk's end) and issue the chunk
//                   loads (TMA);
//   gradient warps  dW += H_{t-1}^T D_t as one tcgen05 MMA per step into a
//                   tensor-memory accumulator; every fourth step each warp
//                   forms dk_t = D_t v_t and the row block's D_t^T k_t as
//                   warp MMAs on the step's bf16 D tile (ldmatrix, plain and
//                   transposed), sums the df shares, and adds dw_r.
// Warp w of each warpgroup runs on scheduler w, so the three interleave.  The
// elementwise work is in packed fp32x2 arithmetic.  Two chunk caches (8
// tensor-memory columns per step) and two H tile buffers let the rebuild of
// chunk c-1 overlap the reverse walk of chunk c.  Shared memory is what
// bounds the chunk length (20 steps).
//
// Measured (timing-only copies, B=4 N=8 T=4096): the proxy fence before the
// reverse warps' hand-off cost 7.5 % of the kernel while it had the H tile and
// df stores of the same step to drain.  The H tiles are now written by the
// recompute warps, and the fence sits right after the exchange barrier (the
// D tile stores are complete, no ldmatrix or MMA is in flight yet) and
// before the df store (read only by the generic proxy).  A latency probe of
// the reverse step alone: fence after the chain MMAs 343 cycles per step,
// after the barrier 294, none 281.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 64;
constexpr int kRows = 16;
constexpr int kThreads = 384;     // reverse warps 0-3, recompute warps 4-7, gradient warps 8-11
// Tensor memory: columns [0, 320) hold two chunk caches, columns [448, 512)
// the dW accumulator.  Per step and thread, 8 columns: G = (1-f)(1-Z^2) as
// four fp16 pairs, then E = H_{t-1} - Z as four fp16 pairs, each in the order
// (column block 0, row g), (0, g+8), (1, g), (1, g+8).
constexpr int kDWCol = 448;
constexpr int kCacheCols = 8;
constexpr int kMaxChunk = 20;  // bounded by shared memory (the H tile and Z stash chunk buffers)
static_assert(2 * kMaxChunk * kCacheCols <= kDWCol, "chunk caches overlap the dW accumulator");
constexpr int kCBufs = 4;         // chunk input buffers (reverse, gradient, recompute, loading)
constexpr int kNX = 8;            // exchange ring slots, reverse -> gradient warps
// Exchange slot (reverse -> gradient warps), one per time step:
//   Dt  bf16 D tile: A operand of the reverse warps' chain MMAs (ldmatrix),
//       B operand of the dW MMA (tcgen05), and the operand of the gradient
//       warps' dk and dv MMAs (ldmatrix, plain and transposed)
//   Df  per-thread shares of df = <R, H_{t-1} - Z> over the thread's eight values: [128]
// The H tile buffer holds, per chunk and step, the bf16 H_{t-1} tile: the A
// operand of the dW MMA, H_{t-1}^T (M = 64).
// Both bf16 tiles use the canonical no-swizzle core-matrix layout: the 8 x 8
// block (rows 8i.., columns 8j..) is 128 contiguous bytes at 256 j + 128 i, so
// as tcgen05 operands (MN-major, the columns contiguous) the core matrices
// advance by 128 bytes along K (the 16 rows) and 256 bytes along M / N.
constexpr uint32_t kXDt = 0, kXDf = 2048, kXSlotBytes = 2560;
constexpr uint32_t kHTileBytes = 2048;
static_assert(kXDf + 128 * 4 <= kXSlotBytes, "exchange slot overflow");

__device__ __forceinline__ uint32_t cm_off(int row, int col) {
  return static_cast<uint32_t>((col >> 3) * 256 + (row >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}
// ldmatrix.x4 address for the A fragments of k-tile kt (columns 16kt..16kt+15)
// of a core-matrix tile: matrices (rows 0-7 | 8-15) x (columns 16kt.. | 16kt+8..).
__device__ __forceinline__ uint32_t cm_ldsm_a(uint32_t tile, int kt, int lane) {
  const int mi = lane >> 3;
  return tile + cm_off((lane & 7) + (mi & 1) * 8, 16 * kt + (mi >> 1) * 8);
}
// ldmatrix.x4.trans address for the A fragments of the transposed tile (rows =
// tile columns 16mt..16mt+15, k = the 16 tile rows): matrices (tile rows 0-7 |
// 8-15) x (columns 16mt.. | 16mt+8..), the column block varying fastest.
__device__ __forceinline__ uint32_t cm_ldsm_at(uint32_t tile, int mt, int lane) {
  const int mi = lane >> 3;
  return tile + cm_off((lane & 7) + (mi >> 1) * 8, 16 * mt + (mi & 1) * 8);
}

__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }

struct MmaBwdParams {
  BwdArgs a;
  int R;
  int nchunks;
  int nbuf;  // TMEM cache buffers (2)
  uint32_t htile_off, cbuf_off, cbuf_bytes, cq_off, ck_off, cv_off, cdy_off, cf_off;
  uint32_t xring_off, dqp_off, dwr_off, bar_off, misc_off, zbuf_off, hbuf_off;
  uint32_t tx_bytes;
  float* dvp;  // [B*T*N][R][V]: row-block partials of D^T k
  float* dfp;  // [B*T*N][R]:    row-block partials of df
};

// One rebuilt step for the reverse walk: from Z_s (fp32 pairs z), H_{s-1}
// (fp32 pairs h, advanced in place to H_s) and 1 - f_s, the 8 cache words of
// this thread and its four bf16 H_{s-1} pairs for the dW tile.  Pairs are
// indexed [column block nt][row half: 0 = g, 1 = g + 8].
__device__ __forceinline__ void rebuild_step(const float2 (&z)[2][2], float2 (&h)[2][2], float omf,
                                             uint32_t (&cache)[kCacheCols], uint32_t (&hb)[4]) {
  const float2 omf2 = splat2(omf), nomf2 = splat2(-omf), neg1 = splat2(-1.f);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float2 zz = __fmul2_rn(z[nt][hh], z[nt][hh]);
      const float2 G = __ffma2_rn(nomf2, zz, omf2);                 // (1-f)(1 - Z^2)
      const float2 E = __ffma2_rn(z[nt][hh], neg1, h[nt][hh]);      // H_{s-1} - Z_s
      cache[2 * nt + hh] = pack2_f16(G.x, G.y);
      cache[4 + 2 * nt + hh] = pack2_f16(E.x, E.y);
      hb[2 * nt + hh] = pack_bf16x2(h[nt][hh].x, h[nt][hh].y);
      h[nt][hh] = __ffma2_rn(nomf2, E, h[nt][hh]);                  // H_s = H_{s-1} + (1-f)(Z_s - H_{s-1})
    }
}

__device__ __forceinline__ void tmem_st_cache(uint32_t taddr, const uint32_t (&c)[kCacheCols]) {
  tmem_st_32x32b_x8(taddr, c);
}

__device__ __forceinline__ void tmem_ld_cache(uint32_t taddr, uint32_t (&c)[kCacheCols]) {
  tmem_ld_32x32b<8>(taddr, c);
}

// kClip: the state-gradient clamp, a compile-time switch (a per-step branch
// on it cost ~7% of the kernel, measured).
template <bool kClip>
__global__ void __launch_bounds__(kThreads, 1)
    mma_backward_kernel(const __grid_constant__ MmaBwdParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_dy) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const BwdArgs& A = p.a;
  const int R = p.R, T = A.T, N = A.N, CL = A.ckpt_every;
  const int cta_rank = static_cast<int>(blockIdx.x) % R;
  const int chain = static_cast<int>(blockIdx.x) / R;
  const int b = chain / N, n = chain % N;
  StatusBlock* status = A.status;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* cfull = bars;
  uint64_t* cempty = cfull + kCBufs;
  uint64_t* tready = cempty + kCBufs;
  uint64_t* tfree = tready + 2;
  uint64_t* xfull = tfree + 2;
  uint64_t* xempty = xfull + kNX;
  uint64_t* dwdone = xempty + kNX;
  uint64_t* zfull = dwdone + 1;  // [2]: Z stash chunk buffers
  uint64_t* hfree = zfull + 2;   // [2]: every dW MMA reading an H tile buffer is complete
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* vabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  volatile int* rabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 8);
  volatile int* gabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 12);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 16);

  if (threadIdx.x == 0) {
    // Warps arrive once each (lane 0 after __syncwarp), except the loading
    // warp, whose lanes each publish a value of f.
    for (int i = 0; i < kCBufs; ++i) {
      mbar_init(smem_u32(&cfull[i]), 32);    // the loading warp's lanes (+ TMA bytes)
      mbar_init(smem_u32(&cempty[i]), 4);    // the gradient warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tready[i]), 4);    // one lane per recompute warp
      mbar_init(smem_u32(&tfree[i]), 4);     // one lane per reverse warp
    }
    for (int i = 0; i < kNX; ++i) {
      mbar_init(smem_u32(&xfull[i]), 4);     // the reverse warps
      mbar_init(smem_u32(&xempty[i]), 2);    // the dW MMA's commit + the step's duty warp
    }
    mbar_init(smem_u32(dwdone), 1);          // every dW MMA complete
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&zfull[i]), 1);  // the loading lane (+ bulk bytes)
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&hfree[i]), 1);  // the dW MMAs' commit
    *abort_flag = 0;
    *vabort = 0;
    *rabort = 0;
    *gabort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {  // the whole tensor memory: chunk caches and the dW accumulator
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Warp w of the reverse and recompute warpgroups owns value columns
  // 16w..16w+15 (thread columns jcol0 + 8nt + {0,1}, rows g and g+8 of the
  // CTA's block).  Reverse warp w and recompute warp w + 4 share TMEM lanes
  // 32w.. and the same fragment positions, so each reverse thread reads
  // exactly what its recompute partner cached: buffer tb, slot s = columns
  // 12 (C tb + s) .. + 11.
  const int w = warp & 3;
  const int g = lane >> 2, qd = lane & 3;
  const int ctid = threadIdx.x & 127;
  const int jcol0 = 16 * w + 2 * qd;
  const int64_t row_g = static_cast<int64_t>(cta_rank) * kRows + g;
  const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
  const uint32_t tcache = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
  const uint32_t xring0 = smem_u32(smem + p.xring_off);
  const uint32_t hbuf0 = smem_u32(smem + p.hbuf_off);  // two buffers of C H tiles

  if (warp < 4) {
    // ======================= reverse warps =======================
    // Backward transform fragments: B[k = j][col = m] = W[16w + m][j] (D W^T),
    // k-tiles in the order w, w+1, w+2, w+3 (mod 4): the first is this warp's
    // own 16 columns of D, whose A fragments it already holds.
    uint32_t bt[2][4][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = 16 * w + 8 * nt + g;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k0 = 16 * ((w + i) & 3) + 2 * qd;
        bt[nt][i][0] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + k0);
        bt[nt][i][1] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + k0 + 8);
      }
    }
    // State gradient C as pairs [column block nt][row half], initialised with dH_T.
    float2 Cg[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (A.dH_T != nullptr) {
        const float* src = A.dH_T + (static_cast<int64_t>(chain) * A.K + row_g) * kV + jcol0 + 8 * nt;
        Cg[nt][0] = *reinterpret_cast<const float2*>(src);
        Cg[nt][1] = *reinterpret_cast<const float2*>(src + 8 * kV);
      } else {
        Cg[nt][0] = Cg[nt][1] = make_float2(0.f, 0.f);
      }
    }
    bool ok = true;
    bool xready = true;  // the slot of step rs is known to be free
    int rs = 0;          // reverse steps done (processing order)
    int xs = 0;          // exchange slot of step rs
    uint32_t xpar = 0;   // its phase parity, (rs / kNX) & 1
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int L = min(CL, T - c * CL);
      const int cb = ci % kCBufs, tb = ci % p.nbuf;
      bool mine = mbar_wait_timed(smem_u32(&cfull[cb]), (ci / kCBufs) & 1, status, kWhereBwdFull);
      if (mine)
        mine = mbar_wait_timed(smem_u32(&tready[tb]), (ci / p.nbuf) & 1, status, kWhereBwdTReady);
      if (!mine) *vabort = 1;
      named_bar_sync(1, 128);
      if (*vabort) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t cbuf = smem_u32(smem + p.cbuf_off + cb * p.cbuf_bytes);
      const uint32_t sq = cbuf + p.cq_off, sdy = cbuf + p.cdy_off, sf = cbuf + p.cf_off;
      const uint32_t tbuf = tcache + kCacheCols * CL * tb;
      // The next slot's TMEM load is issued one step ahead and waited for at
      // the top of the step.
      uint32_t sr[kCacheCols];
      tmem_ld_cache(tbuf + kCacheCols * (L - 1), sr);
      for (int s = L - 1; s >= 0; --s, ++rs) {
        // The slot is free once the gradient warps have consumed step rs - kNX
        // (tested at the end of the previous step, so that the test's latency
        // overlaps that step's tail; waited for here only if it failed).  A
        // give-up is acted on at the next chunk boundary (the wait raised the
        // CTA's abort flag, so the remaining waits end at once).
        if (!xready && !mbar_wait(smem_u32(&xempty[xs]), xpar ^ 1u, abort_flag, status, kWhereBwdXEmpty))
          *vabort = 1;
        const uint32_t xb = xring0 + xs * kXSlotBytes;
        const float2 q0 = splat2(__uint_as_float(ld_shared_u16(sq + 2 * (s * kRows + g)) << 16));
        const float2 q1 = splat2(__uint_as_float(ld_shared_u16(sq + 2 * (s * kRows + g + 8)) << 16));
        const float2 f2 = splat2(ld_shared_f32(sf + 4 * s));
        float2 u[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) u[nt] = ld_shared_f32x2(sdy + 4 * (s * kV + jcol0 + 8 * nt));
        tmem_ld_wait();
        tmem_ld_fence_regs(sr);
        float2 G[2][2];
        uint32_t ew[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          G[i >> 1][i & 1] = f16x2_to_float2(sr[i]);
          ew[i] = sr[4 + i];
        }
        if (s > 0) tmem_ld_cache(tbuf + kCacheCols * (s - 1), sr);
        // R = C + q u^T ; D = R * G with G = (1-f)(1 - Z^2)
        float2 Rv[2][2], Dv[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          Rv[nt][0] = __ffma2_rn(q0, u[nt], Cg[nt][0]);
          Rv[nt][1] = __ffma2_rn(q1, u[nt], Cg[nt][1]);
          Dv[nt][0] = __fmul2_rn(Rv[nt][0], G[nt][0]);
          Dv[nt][1] = __fmul2_rn(Rv[nt][1], G[nt][1]);
        }
        // Serial chain: C_{t-1} = f R + D W^T on the warp MMAs.  bf16(D) of
        // this warp's columns is its own k-tile (the accumulator layout of
        // two n-tiles is the A layout of one k-tile): those two MMAs run
        // while the other three k-tiles load from the tile.
        const uint32_t dt = xb + kXDt;
        uint32_t aown[4];
        aown[0] = pack2_bf16(Dv[0][0].x, Dv[0][0].y);
        aown[1] = pack2_bf16(Dv[0][1].x, Dv[0][1].y);
        aown[2] = pack2_bf16(Dv[1][0].x, Dv[1][0].y);
        aown[3] = pack2_bf16(Dv[1][1].x, Dv[1][1].y);
        st_shared_b32(dt + cm_off(g, jcol0), aown[0]);
        st_shared_b32(dt + cm_off(g + 8, jcol0), aown[1]);
        st_shared_b32(dt + cm_off(g, jcol0 + 8), aown[2]);
        st_shared_b32(dt + cm_off(g + 8, jcol0 + 8), aown[3]);
        named_bar_sync(1, 128);
        // The D tile is also read by the tensor core (dW), through the async
        // proxy: this thread's stores to it completed before the barrier, so
        // the fence has nothing to wait for here; placed after the chain
        // MMAs it stalled the step by ~50 cycles (measured).
        fence_proxy_async_smem();
        uint32_t af[3][4];
#pragma unroll
        for (int i = 0; i < 3; ++i) ldmatrix_x4(af[i], cm_ldsm_a(dt, (w + 1 + i) & 3, lane));
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 a0 = __fmul2_rn(f2, Rv[nt][0]), a1 = __fmul2_rn(f2, Rv[nt][1]);
          acc[nt][0] = a0.x; acc[nt][1] = a0.y; acc[nt][2] = a1.x; acc[nt][3] = a1.y;
          mma_bf16_16816(acc[nt], aown, bt[nt][0][0], bt[nt][0][1]);
        }
#pragma unroll
        for (int i = 0; i < 3; ++i)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(acc[nt], af[i], bt[nt][i + 1][0], bt[nt][i + 1][1]);
        // Off the chain: this thread's share of df = <R, H_{t-1} - Z>, read
        // by the gradient warps through the generic proxy only.
        {
          float2 pe2 = __fmul2_rn(Rv[0][0], f16x2_to_float2(ew[0]));
          pe2 = __ffma2_rn(Rv[0][1], f16x2_to_float2(ew[1]), pe2);
          pe2 = __ffma2_rn(Rv[1][0], f16x2_to_float2(ew[2]), pe2);
          pe2 = __ffma2_rn(Rv[1][1], f16x2_to_float2(ew[3]), pe2);
          st_shared_f32(xb + kXDf + 4 * ctid, pe2.x + pe2.y);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&xfull[xs]));
        if constexpr (kClip) {  // per-step clipping of the state gradient
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = fminf(fmaxf(acc[nt][e], -A.clip), A.clip);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          Cg[nt][0] = make_float2(acc[nt][0], acc[nt][1]);
          Cg[nt][1] = make_float2(acc[nt][2], acc[nt][3]);
        }
        if (++xs == kNX) {
          xs = 0;
          xpar ^= 1u;
        }
        xready = rs + 1 < kNX || mbar_test_wait(smem_u32(&xempty[xs]), xpar ^ 1u);
      }
      // Every slot of this cache buffer has been read (the last load was
      // waited for at s = 0): the recompute may refill it.
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tfree[tb]));
    }
    if (ok && A.dH0 != nullptr) {  // C_0, the state gradient left after step 1
      float* dst = A.dH0 + (static_cast<int64_t>(chain) * A.K + row_g) * kV + jcol0;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        *reinterpret_cast<float2*>(dst + 8 * nt) = Cg[nt][0];
        *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt) = Cg[nt][1];
      }
    }
    if (!ok) *abort_flag = 1;
  } else if (warp < 8) {
    // ======================= recompute warps (Eq. 10-11) =======================
    // Forward transform fragments (fp16): B[k][col] = W[k][16w + col], k-tiles in
    // the order w, w+1, w+2, w+3 (mod 4): the first is this warp's own 16
    // columns of H, whose A fragments it holds in registers.
    uint32_t bw[2][4][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = 16 * w + 8 * nt + g;
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const int k0 = 16 * ((w + kt) & 3) + 2 * qd;
        bw[nt][kt][0] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[k0 * kV + col]) |
                                        (static_cast<uint32_t>(Wg[(k0 + 1) * kV + col]) << 16));
        bw[nt][kt][1] = bf16x2_to_f16x2(static_cast<uint32_t>(Wg[(k0 + 8) * kV + col]) |
                                        (static_cast<uint32_t>(Wg[(k0 + 9) * kV + col]) << 16));
        if (!f16x2_finite(bw[nt][kt][0]) || !f16x2_finite(bw[nt][kt][1]))
          report_device_error(status, kStatusCheck, kWhereWRange);
      }
    }
    const uint32_t htile0 = smem_u32(smem + p.htile_off);
    const uint32_t dqp = smem_u32(smem + p.dqp_off);  // fp32 [C][4 warps][4 qd][8 g][row g, g+8]
    // Start state of a chunk: the checkpoint (H_0, zero if not given, for
    // chunk 0).  The next chunk's is loaded a chunk ahead, so its latency
    // stays off the path.
    auto load_start = [&](int cc, float2 (&hs)[2][2]) {
      if (cc == 0 && A.H0 == nullptr) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) hs[nt][0] = hs[nt][1] = make_float2(0.f, 0.f);
      } else {
        const float* src =
            (cc == 0 ? A.H0 + (static_cast<int64_t>(chain) * A.K + row_g) * kV
                     : A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (cc - 1)) * A.K + row_g) * kV) +
            jcol0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          hs[nt][0] = *reinterpret_cast<const float2*>(src + 8 * nt);
          hs[nt][1] = *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt);
        }
      }
    };
    float2 hnext[2][2];
    load_start(p.nchunks - 1, hnext);
    // Warp 4 also loads the chunk inputs, one chunk ahead of its own use:
    // q, k, v, dy by TMA, f gathered by the lanes (its global-load latency
    // hidden behind the chunk's recompute) and published at the chunk's end.
    const bool loader = (warp == 4);
    const GateSrc gs{A.f, A.gate_a, A.gate_alpha, A.gate_beta, true};
    auto issue_chunk = [&](int li) -> float {
      const int t0 = (p.nchunks - 1 - li) * CL;
      uint8_t* buf = smem + p.cbuf_off + (li % kCBufs) * p.cbuf_bytes;
      const uint32_t fb = smem_u32(&cfull[li % kCBufs]);
      if (lane == 0) {
        mbar_expect_tx(fb, p.tx_bytes);
        tma_load_4d(smem_u32(buf + p.cq_off), &tm_q, fb, cta_rank * kRows, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.ck_off), &tm_k, fb, cta_rank * kRows, qk_head(A.qkN, n), t0, b);
        tma_load_4d(smem_u32(buf + p.cv_off), &tm_v, fb, 0, n, t0, b);
        tma_load_4d(smem_u32(buf + p.cdy_off), &tm_dy, fb, 0, n, t0, b);
      }
      const int t = t0 + lane;
      return (lane < CL && t < T) ? gate_value(gs, (static_cast<int64_t>(b) * T + t) * N + n, n) : 0.f;
    };
    auto publish_chunk = [&](int li, float fv) {
      float* cfw = reinterpret_cast<float*>(smem + p.cbuf_off + (li % kCBufs) * p.cbuf_bytes + p.cf_off);
      if (lane < CL) cfw[lane] = fv;
      mbar_arrive(smem_u32(&cfull[li % kCBufs]));  // all 32 lanes: the phase's arrival count
    };
    // Z stash: chunk li's steps into the staging buffer (one bulk copy).
    const bool zs = A.zstash != nullptr;
    const uint8_t* zsrc = reinterpret_cast<const uint8_t*>(A.zstash) + static_cast<int64_t>(blockIdx.x) * T * kZStepBytes;
    // One staging buffer: chunk li + 1 is copied in once chunk li is rebuilt,
    // while the reverse warps still walk chunk li - 1.
    auto issue_z = [&](int li) {
      if (lane == 0) {
        const int t0 = (p.nchunks - 1 - li) * CL;
        const uint32_t bytes = static_cast<uint32_t>(min(CL, T - t0)) * kZStepBytes;
        const uint32_t zb = smem_u32(&zfull[0]);
        mbar_arrive_expect_tx(zb, bytes);
        bulk_load(smem_u32(smem + p.zbuf_off), zsrc + static_cast<int64_t>(t0) * kZStepBytes, bytes, zb);
      }
    };
    int zissued = 0;  // Z chunks whose copies have been issued
    if (loader) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_dy);
      }
      if (zs) issue_z(zissued++);
      publish_chunk(0, issue_chunk(0));
    }
    // The stash step (2 KB) holds, at (32 w + lane) * 16, the 16 bytes that
    // the forward's compute warp w, lane `lane`, wrote: {Z[g][j], Z[g][j+1]},
    // j = 16w + 8nt + 2qd, in the order (nt 0, row g), (0, g+8), (1, g),
    // (1, g+8) -- exactly this thread's values.
    const uint32_t zaddr = smem_u32(smem + p.zbuf_off) + static_cast<uint32_t>((32 * w + lane) * 16);
    bool ok = true;
    int issued = 1;  // chunks whose loads have been issued
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL;
      const int L = min(CL, T - s0);
      const int cb = ci % kCBufs, tb = ci % p.nbuf;
      bool mine = mbar_wait_timed(smem_u32(&cfull[cb]), (ci / kCBufs) & 1, status, kWhereBwdFull);
      // The cache buffer is free once the reverse warps have finished chunk
      // ci - nbuf.
      if (mine && ci >= p.nbuf)
        mine = mbar_wait_timed(smem_u32(&tfree[tb]), ((ci / p.nbuf) - 1) & 1, status, kWhereBwdTFree);
      // The input buffer chunk ci + 1 will use last held chunk ci - 3: free
      // once the gradient warps (the last to read it) are past it.
      if (mine && ci >= 3 && ci + 1 < p.nchunks)
        mine = mbar_wait_timed(smem_u32(&cempty[(ci + 1) % kCBufs]), ((ci - 3) / kCBufs) & 1, status,
                               kWhereBwdCEmpty);
      if (mine && zs) mine = mbar_wait_timed(smem_u32(&zfull[0]), ci & 1, status, kWhereBwdZFull);
      // The H tile buffer is free once every dW MMA of chunk ci - nbuf is done.
      if (mine && ci >= p.nbuf)
        mine = mbar_wait_timed(smem_u32(&hfree[tb]), ((ci / p.nbuf) - 1) & 1, status, kWhereBwdDW);
      if (!mine) *rabort = 1;
      named_bar_sync(2, 128);
      if (*rabort) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const bool more = loader && ci + 1 < p.nchunks;
      float fnext = 0.f;
      if (more) fnext = issue_chunk(ci + 1);
      const uint32_t cbuf = smem_u32(smem + p.cbuf_off + cb * p.cbuf_bytes);
      const uint32_t sk = cbuf + p.ck_off, sv = cbuf + p.cv_off, sdy = cbuf + p.cdy_off, sf = cbuf + p.cf_off;
      const uint32_t tbuf = tcache + kCacheCols * CL * tb;
      const uint32_t hbase = hbuf0 + static_cast<uint32_t>(tb * CL) * kHTileBytes;
      // This thread's four bf16 H_{s-1} pairs into step s's H tile.
      auto store_htile = [&](int s, const uint32_t (&hb)[4]) {
        const uint32_t ht = hbase + static_cast<uint32_t>(s) * kHTileBytes;
        st_shared_b32(ht + cm_off(g, jcol0), hb[0]);
        st_shared_b32(ht + cm_off(g + 8, jcol0), hb[1]);
        st_shared_b32(ht + cm_off(g, jcol0 + 8), hb[2]);
        st_shared_b32(ht + cm_off(g + 8, jcol0 + 8), hb[3]);
      };
      float2 h[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        h[nt][0] = hnext[nt][0];
        h[nt][1] = hnext[nt][1];
      }
      if (c > 0) load_start(c - 1, hnext);
      // dq_t = H_t u_t: this thread's share over its four columns (rows g
      // and g + 8), in fp32; the sixteen shares of a row are summed at the
      // chunk's end.
      auto dq_share = [&](int s) {
        const float2 u0 = ld_shared_f32x2(sdy + 4 * (s * kV + jcol0));
        const float2 u1 = ld_shared_f32x2(sdy + 4 * (s * kV + jcol0 + 8));
        const float2 pg = __ffma2_rn(h[1][0], u1, __fmul2_rn(h[0][0], u0));
        const float2 pg8 = __ffma2_rn(h[1][1], u1, __fmul2_rn(h[0][1], u0));
        st_shared_f32x2(dqp + 4 * ((s * 16 + w * 4 + qd) * kRows + 2 * g), make_float2(pg.x + pg.y, pg8.x + pg8.y));
      };
      auto pack_h = [&](uint32_t (&ha)[4]) {  // fp16 H as this warp's A fragment
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          ha[2 * nt] = pack2_f16(h[nt][0].x, h[nt][0].y);
          ha[2 * nt + 1] = pack2_f16(h[nt][1].x, h[nt][1].y);
        }
      };
      if (zs) {
        for (int s = 0; s < L; ++s) {
          const float omf = 1.f - ld_shared_f32(sf + 4 * s);
          const uint4 zv4 = ld_shared_v4(zaddr + s * kZStepBytes);
          const uint32_t zq[4] = {zv4.x, zv4.y, zv4.z, zv4.w};
          float2 z[2][2];
#pragma unroll
          for (int i = 0; i < 4; ++i) z[i >> 1][i & 1] = f16x2_to_float2(zq[i]);
          uint32_t cache[kCacheCols], hb[4];
          rebuild_step(z, h, omf, cache, hb);
          tmem_st_cache(tbuf + kCacheCols * s, cache);
          store_htile(s, hb);
          dq_share(s);
        }
        // Every read of this Z buffer and every dq share of the chunk is done.
        named_bar_sync(2, 128);
        if (loader && zissued < p.nchunks) issue_z(zissued++);
      } else {
        // Step s, as in the forward: acc = k_s v_s^T + fp16(H_{s-1}) W, the
        // own k-tile from registers while the other three load from the tile.
        uint32_t hh[4];
        auto store_tile = [&](uint32_t base) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int col = jcol0 + 8 * nt;
            st_shared_b32(base + tile_off(g, col), hh[2 * nt]);
            st_shared_b32(base + tile_off(g + 8, col), hh[2 * nt + 1]);
          }
        };
        pack_h(hh);
        store_tile(htile0);
        named_bar_sync(2, 128);
        for (int s = 0; s < L; ++s) {
          const float omf = 1.f - ld_shared_f32(sf + 4 * s);
          const uint32_t atile = htile0 + (s & 1) * 2048;
          uint32_t af[3][4];
#pragma unroll
          for (int i = 0; i < 3; ++i) ldmatrix_x4(af[i], ldsm_addr_a(atile, (w + 1 + i) & 3, lane));
          float acc[2][4];
          const float k0 = __uint_as_float(ld_shared_u16(sk + 2 * (s * kRows + g)) << 16);
          const float k1 = __uint_as_float(ld_shared_u16(sk + 2 * (s * kRows + g + 8)) << 16);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = ld_shared_b32(sv + 2 * (s * kV + jcol0 + 8 * nt));
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            acc[nt][0] = k0 * v0;
            acc[nt][1] = k0 * v1;
            acc[nt][2] = k1 * v0;
            acc[nt][3] = k1 * v1;
            mma_f16_16816(acc[nt], hh, bw[nt][0][0], bw[nt][0][1]);
          }
#pragma unroll
          for (int i = 0; i < 3; ++i)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_f16_16816(acc[nt], af[i], bw[nt][i + 1][0], bw[nt][i + 1][1]);
          float2 z[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            z[nt][0] = make_float2(tanh_fast(acc[nt][0]), tanh_fast(acc[nt][1]));
            z[nt][1] = make_float2(tanh_fast(acc[nt][2]), tanh_fast(acc[nt][3]));
          }
          uint32_t cache[kCacheCols], hb[4];
          rebuild_step(z, h, omf, cache, hb);
          pack_h(hh);
          store_tile(htile0 + ((s + 1) & 1) * 2048);
          tmem_st_cache(tbuf + kCacheCols * s, cache);
          store_htile(s, hb);
          dq_share(s);
          named_bar_sync(2, 128);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the chunk's H tiles are read by the tensor core
      if (more) publish_chunk(ci + 1, fnext);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tready[tb]));
      issued = ci + 2;
      // dq rows of the chunk (the last step's barrier ordered every share):
      // the sixteen shares of row r = g + 8 hi, warp by warp, in a fixed order.
      for (int idx = ctid; idx < L * kRows; idx += 128) {
        const int sp = idx >> 4, r = idx & 15;
        const uint32_t pp = dqp + 4 * (sp * 16 * kRows + 2 * (r & 7) + (r >> 3));
        float sum = 0.f;
#pragma unroll
        for (int sh = 0; sh < 16; ++sh) sum += ld_shared_f32(pp + 4 * sh * kRows);
        const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + sp) * N + n;
        A.dq[rowt * A.K + cta_rank * kRows + r] = sum;
      }
    }
    if (!ok) {
      *abort_flag = 1;
      // No TMA copy may still be writing when the CTA exits.
      if (loader) {
        for (int li = max(0, issued - 2); li < min(issued, p.nchunks); ++li)
          mbar_wait_timed(smem_u32(&cfull[li % kCBufs]), (li / kCBufs) & 1, nullptr, kWhereBwdDrain);
        if (zissued > 0) mbar_wait_timed(smem_u32(&zfull[0]), (zissued - 1) & 1, nullptr, kWhereBwdDrain);
      }
    }
  } else {
    // ======================= gradient warps =======================
    // Warp 8 issues the step's dW MMA (one elected lane, tcgen05, the
    // accumulator in TMEM columns 448..511; with M = 64, row 16q + r sits in
    // lane 32q + r):
    //   dW (+)= H_{t-1}^T (64 x 16) * D (16 x 64),
    // committed to the slot's empty barrier.  Every fourth step (rs % 4 == w)
    // warp 8 + w also forms that step's dk and dv partial on the tensor core
    // from the slot's bf16 D tile, sums the df shares (also on the tensor
    // core) and adds its columns' dw_r.  (Splitting that work over all four
    // warps every step was measured 46 % slower: four warps then poll the
    // step's barrier instead of two.)
    // dw_r: the chain's R row-block CTAs each sum a slice of the 32 column
    // pairs; this lane's pair is columns 2 dwr_pair, 2 dwr_pair + 1.
    float dwr0 = 0.f, dwr1 = 0.f;
    const int dwr_ppr = (kV / 2 + R - 1) / R;
    const int dwr_pair = cta_rank * dwr_ppr + lane;
    const bool dwr_lane = lane < dwr_ppr && dwr_pair < kV / 2;
    const uint32_t idesc = idesc_bf16_f32(64, kV, /*a_mn_major=*/true, /*b_mn_major=*/true);
    const uint32_t dw_tmem = tmem_base + kDWCol;
    bool ok = true;
    int rs = 0, xs = 0;
    uint32_t xpar = 0;
    for (int ci = 0; ci < p.nchunks; ++ci) {
      const int c = p.nchunks - 1 - ci;
      const int s0 = c * CL;
      const int L = min(CL, T - s0);
      const int cb = ci % kCBufs;
      const bool mine = mbar_wait_timed(smem_u32(&cfull[cb]), (ci / kCBufs) & 1, status, kWhereBwdFull);
      if (!mine) *gabort = 1;
      named_bar_sync(3, 128);
      if (*gabort) {
        ok = false;
        break;
      }
      const uint32_t cbuf = smem_u32(smem + p.cbuf_off + cb * p.cbuf_bytes);
      const uint32_t sk = cbuf + p.ck_off, sv = cbuf + p.cv_off, sdy = cbuf + p.cdy_off;
      const int tb = ci % p.nbuf;
      const uint32_t hbase = hbuf0 + static_cast<uint32_t>(tb * CL) * kHTileBytes;
      for (int s = L - 1; s >= 0; --s, ++rs) {
        const bool duty = (rs & 3) == w;
        const uint32_t xb = xring0 + xs * kXSlotBytes;
        // A give-up is acted on at the next chunk boundary.
        if ((w == 0 || duty) && !mbar_wait(smem_u32(&xfull[xs]), xpar, abort_flag, status, kWhereBwdXFull))
          *gabort = 1;
        if (w == 0) {
          tc_fence_after_sync();
          if (elect_one()) {
            tc_mma_f16_ss(dw_tmem, smem_desc_noswizzle(hbase + static_cast<uint32_t>(s) * kHTileBytes, 128, 256),
                          smem_desc_noswizzle(xb + kXDt, 128, 256), idesc, rs > 0 ? 1u : 0u);
            tc_commit(smem_u32(&xempty[xs]));  // arrives once the MMA has read the slot
          }
          __syncwarp();
        }
        if (duty) {
          const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
          const uint32_t dt = xb + kXDt;
          // dk_t = D_t v_t: A = D (four k-tiles), B = v_t pairs in every
          // column; row g's value is c0, row g + 8's c2 (in every lane).
          // The B fragments of all four k-tiles come from two ldmatrix.x4
          // whose eight row addresses per matrix all point at the same 8
          // values of v_t.
          {
            uint32_t vb[2][4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) ldmatrix_x4(vb[hf], sv + 2 * (s * kV + 32 * hf + 8 * (lane >> 3)));
            float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kt = 0; kt < 4; ++kt) {
              uint32_t a[4];
              ldmatrix_x4(a, cm_ldsm_a(dt, kt, lane));
              mma_bf16_16816(d4, a, vb[kt >> 1][2 * (kt & 1)], vb[kt >> 1][2 * (kt & 1) + 1]);
            }
            if (qd == 0) {
              A.dk[rowt * A.K + cta_rank * kRows + g] = d4[0];
              A.dk[rowt * A.K + cta_rank * kRows + g + 8] = d4[2];
            }
          }
          // Row-block partial of D_t^T k_t: A = D^T (ldmatrix.trans, four
          // 16-column m-tiles), B = k_t pairs of the block's rows in every
          // column; column 16 mt + g is c0 of m-tile mt, 16 mt + g + 8 its c2.
          // Lane (g, qd) stores m-tile qd's two values.
          {
            const uint32_t b0 = ld_shared_b32(sk + 2 * (s * kRows + 2 * qd));
            const uint32_t b1 = ld_shared_b32(sk + 2 * (s * kRows + 2 * qd + 8));
            float lo = 0.f, hi = 0.f;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
              uint32_t a[4];
              ldmatrix_x4_trans(a, cm_ldsm_at(dt, mt, lane));
              float d4[4] = {0.f, 0.f, 0.f, 0.f};
              mma_bf16_16816(d4, a, b0, b1);
              lo = (qd == mt) ? d4[0] : lo;
              hi = (qd == mt) ? d4[2] : hi;
            }
            float* dst = p.dvp + (rowt * R + cta_rank) * kV + 16 * qd + g;
            dst[0] = lo;
            dst[8] = hi;
          }
          // Row-block partial of df_t = <R_t, H_{t-1} - Z_t>: four shares
          // per lane, then the 32 lanes summed on the tensor core.
          {
            const float4 e4 = ld_shared_f32x4(xb + kXDf + 16 * lane);
            const float pf = warp_sum_mma((e4.x + e4.y) + (e4.z + e4.w));
            if (lane == 0) p.dfp[rowt * R + cta_rank] = pf;
          }
          if (dwr_lane) {  // dw_r += u_t * v_t over this CTA's columns
            const float2 uu = ld_shared_f32x2(sdy + 4 * (s * kV + 2 * dwr_pair));
            const uint32_t vv = ld_shared_b32(sv + 2 * (s * kV + 2 * dwr_pair));
            dwr0 = fmaf(uu.x, bf16lo(vv), dwr0);
            dwr1 = fmaf(uu.y, bf16hi(vv), dwr1);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&xempty[xs]));
        }
        if (++xs == kNX) {
          xs = 0;
          xpar ^= 1u;
        }
      }
      // The chunk's H tile buffer is free once its last dW MMA completes.
      if (w == 0) {
        if (elect_one()) tc_commit(smem_u32(&hfree[tb]));
        __syncwarp();
      }
      // The gradient warps are the last readers of the chunk's inputs.
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&cempty[cb]));
    }
    // No dW MMA may still be running when tensor memory is released.
    if (w == 0 && rs > 0) {
      if (elect_one()) tc_commit(smem_u32(dwdone));
      __syncwarp();
    }
    if (ok) {
      // dW partial of this row block from TMEM: accumulator row m = 16w + lane
      // in lane 32w + lane (lanes 16..31 of each quadrant unused), column
      // n = 448 + n.
      {
        if (!mbar_wait_timed(smem_u32(dwdone), 0, status, kWhereBwdDW)) *gabort = 1;
        tc_fence_after_sync();
        float* dwp = A.dW_part + static_cast<int64_t>(blockIdx.x) * kV * kV + (16 * w + (lane & 15)) * kV;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld_32x32b<32>(tmem_base + (static_cast<uint32_t>(32 * w) << 16) + kDWCol + 32 * half, r);
          tmem_ld_wait();
          tmem_ld_fence_regs(r);
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4)
            if (lane < 16) *reinterpret_cast<float4*>(dwp + 32 * half + c4) =
                make_float4(__uint_as_float(r[c4]), __uint_as_float(r[c4 + 1]), __uint_as_float(r[c4 + 2]),
                            __uint_as_float(r[c4 + 3]));
        }
      }
      // dw_r: the four warps' step subsets, summed in a fixed order.
      float* sd = reinterpret_cast<float*>(smem + p.dwr_off);
      *reinterpret_cast<float2*>(sd + w * kV + 2 * lane) = make_float2(dwr0, dwr1);
      named_bar_sync(3, 128);
      if (w == 0 && dwr_lane) {
        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) {
          const float2 x = *reinterpret_cast<const float2*>(sd + ww * kV + 2 * lane);
          acc2.x += x.x;
          acc2.y += x.y;
        }
        *reinterpret_cast<float2*>(A.dwr_part + static_cast<int64_t>(chain) * kV + 2 * dwr_pair) = acc2;
      }
    } else {
      *abort_flag = 1;
      if (w == 0 && rs > 0) mbar_wait_timed(smem_u32(dwdone), 0, nullptr, kWhereBwdDW);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// dv = sum over the chain's row blocks of D^T k (fixed order) + w_r * dy;
// df = sum of the RF row-block partials, in order.  One warp per (b, t, n).
__global__ void __launch_bounds__(256) mma_backward_rows_kernel(const float* __restrict__ dvp,
                                                                const float* __restrict__ dfp,
                                                                const float* __restrict__ dy,
                                                                const uint16_t* __restrict__ w_r,
                                                                float* __restrict__ dv, float* __restrict__ df,
                                                                int64_t rows, int N, int R, int RF) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += stride) {
    const int n = static_cast<int>(row % N);
    float a0 = 0.f, a1 = 0.f;
    for (int pr = 0; pr < R; ++pr) {
      const float2 x = *reinterpret_cast<const float2*>(dvp + (row * R + pr) * kV + 2 * lane);
      a0 += x.x;
      a1 += x.y;
    }
    const float2 u = *reinterpret_cast<const float2*>(dy + row * kV + 2 * lane);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(w_r + static_cast<int64_t>(n) * kV + 2 * lane);
    *reinterpret_cast<float2*>(dv + row * kV + 2 * lane) = make_float2(fmaf(bf16lo(wb), u.x, a0), fmaf(bf16hi(wb), u.y, a1));
    if (lane == 0) {
      float sf = 0.f;
      for (int pr = 0; pr < RF; ++pr) sf += dfp[row * RF + pr];
      df[row] = sf;
    }
  }
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }
inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

bool mma_backward_supported(int K, int V) { return V == kV && K % kRows == 0 && K >= kRows && K <= 128; }

size_t mma_backward_scratch_bytes(int B, int T, int N, int K, int, int) {
  const size_t rows = static_cast<size_t>(B) * T * N, R = static_cast<size_t>(K / kRows);
  return align256(sizeof(float) * rows * R * kV) + align256(sizeof(float) * rows * R);
}

int mma_backward_max_chunk() { return kMaxChunk; }

cudaError_t launch_mma_backward(const BwdArgs& a, cudaStream_t stream) {
  if (a.V != kV) return launch_mv_backward(a, stream);  // V = 16: the register-resident kernel
  if (a.ckpt_every > kMaxChunk) return cudaErrorInvalidValue;
  MmaBwdParams p{};
  p.a = a;
  p.R = a.K / kRows;
  const int C = a.ckpt_every;
  p.nchunks = (a.T + C - 1) / C;
  p.nbuf = 2;
  p.htile_off = 0;  // two 2 KB fp16 tiles for the rerun
  p.cbuf_off = 4096;
  p.cq_off = 0;
  p.ck_off = align_up(C * kRows * 2, 128);
  p.cv_off = p.ck_off + align_up(C * kRows * 2, 128);
  p.cdy_off = p.cv_off + align_up(C * kV * 2, 128);
  p.cf_off = p.cdy_off + align_up(C * kV * 4, 128);
  p.cbuf_bytes = align_up(p.cf_off + C * 4, 128);
  p.xring_off = align_up(p.cbuf_off + kCBufs * p.cbuf_bytes, 1024);
  p.hbuf_off = p.xring_off + kNX * kXSlotBytes;  // two buffers of C H tiles
  p.dqp_off = p.hbuf_off + 2 * C * kHTileBytes;
  p.dwr_off = p.dqp_off + C * 16 * kRows * 4;
  p.bar_off = p.dwr_off + 4 * kV * 4;
  p.misc_off = p.bar_off + (2 * kCBufs + 4 + 2 * kNX + 1 + 2 + 2) * 8;
  p.zbuf_off = align_up(p.misc_off + 32, 128);
  const uint32_t zbytes = a.zstash != nullptr ? static_cast<uint32_t>(C) * kZStepBytes : 0u;
  const uint32_t smem = p.zbuf_off + zbytes + 1024;
  p.tx_bytes = 2 * C * kRows * 2 + C * kV * 2 + C * kV * 4;
  const size_t rows = static_cast<size_t>(a.B) * a.T * a.N;
  p.dvp = a.scratch;
  p.dfp = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(a.scratch) +
                                   align256(sizeof(float) * rows * p.R * kV));

  CUtensorMap mq, mk, mv, mdy;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, qN, a.K, kRows, C) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, kRows, C) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, C) ||
      !make_tensor_map_btnx(&mdy, a.dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.N, kV, kV, C))
    return cudaErrorInvalidValue;
  auto kernel = a.clip > 0.f ? mma_backward_kernel<true> : mma_backward_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<static_cast<unsigned>(a.B * a.N * p.R), kThreads, smem, stream>>>(p, mq, mk, mv, mdy);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int blocks = static_cast<int>(std::min<size_t>((rows + 7) / 8, 152 * 16));
  mma_backward_rows_kernel<<<blocks, 256, 0, stream>>>(p.dvp, p.dfp, a.dy, static_cast<const uint16_t*>(a.w_r),
                                                       a.dv, a.df, static_cast<int64_t>(rows), a.N, p.R, p.R);
  return cudaGetLastError();
}

}  // namespace m2rnn
