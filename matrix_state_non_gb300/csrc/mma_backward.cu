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
// order).  The time axis runs over chunks of C <= 28 steps, last chunk first;
// for each chunk the forward is rerun from its checkpoint (section 2.6 of the
// notes describes the paper's rerun-and-cache backward; here only one or two
// chunks are cached) and then walked backwards.  Three warpgroups:
//   reverse warps   (each owning 16 value columns) the serial chain only:
//                   R -> D -> bf16(D) tile -> one named barrier -> 8 warp MMAs
//                   seeded with f R -> C_{t-1}; then their shares of dk, dv,
//                   df and the bf16 D and H_{t-1} tiles go to the gradient
//                   warps through a ring of shared-memory slots;
//   recompute warps (each owning 16 value columns) the forward rerun of the
//                   next chunk (Eq. 10-11), caching each thread's Z_t and
//                   H_{t-1} values (fp32) in its own lane of tensor memory, so
//                   the cache never touches DRAM; also dq_t = H_t u_t and the
//                   chunk loads (TMA).  When the forward left its Z_t in a
//                   stash (fp16), the rerun is only H_t = H_{t-1} + (1-f_t)
//                   (Z_t - H_{t-1}) from the chunk's checkpoint, with Z_t
//                   bulk-copied a chunk at a time: no MMA, no tanh, no
//                   exchange between the warps;
//   gradient warps  dW += H_{t-1}^T D_t as one tcgen05 MMA per step into a
//                   tensor-memory accumulator, and the fixed-order sums of
//                   the dk, dv, df shares and dw_r.
// Warp w of each warpgroup runs on scheduler w, so the three interleave.  The
// chunk caches hold each thread's Z_t and H_{t-1} as fp16 pairs, 8 TMEM
// columns per step; with the 64-column dW accumulator two caches of up to 28
// steps fit, and the rebuild of chunk c-1 overlaps the reverse walk of chunk
// c.
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
// Tensor memory: columns [0, 448) hold two chunk caches (8 columns per step:
// Z_t and H_{t-1} as fp16 pairs), columns [448, 512) the dW accumulator.
constexpr int kDWCol = 448;
constexpr int kCacheCols = 8;
constexpr int kMaxChunk = kDWCol / (2 * kCacheCols);  // 28: two caches, the recompute runs a chunk ahead
constexpr int kCBufs = 4;         // chunk input buffers (reverse, gradient, recompute, loading)
constexpr int kNX = 8;            // exchange ring slots, reverse -> gradient warps
// Exchange slot (reverse -> gradient warps), one per time step:
//   Dt  bf16 D tile: A operand of the reverse warps' chain MMAs (ldmatrix) and
//       B operand of the dW MMA (tcgen05)
//   Ht  bf16 H_{t-1} tile, followed by 2 KB of zeros: A operand of the dW MMA,
//       H_{t-1}^T padded from 64 to 128 rows
//   Dv  per-thread sums of D k over the thread's two rows: [g][64 columns], rows padded to 72 floats
//   Dk  per-thread sums of D v over the thread's four columns: [warp][qd][g][row g, g+8], groups padded to 18
//   Df  per-thread sums of R (H_{t-1} - Z) over the thread's eight values: [128]
// (strides chosen so that both the writers' and the readers' accesses are free of bank conflicts).
// Both bf16 tiles use the canonical no-swizzle core-matrix layout: the 8 x 8
// block (rows 8i.., columns 8j..) is 128 contiguous bytes at 256 j + 128 i, so
// as tcgen05 operands (MN-major, the columns contiguous) the core matrices
// advance by 128 bytes along K (the 16 rows) and 256 bytes along M / N.
constexpr int kDvStride = 72, kDkGroup = 18;
constexpr uint32_t kXDt = 0, kXHt = 2048, kXZero = 4096, kXDv = 6144, kXDk = kXDv + 8 * kDvStride * 4,
                   kXDf = kXDk + 16 * kDkGroup * 4, kXSlotBytes = 10240;
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

struct MmaBwdParams {
  BwdArgs a;
  int R;
  int nchunks;
  int nbuf;  // TMEM cache buffers (2)
  uint32_t htile_off, cbuf_off, cbuf_bytes, cq_off, ck_off, cv_off, cdy_off, cf_off;
  uint32_t xring_off, dqp_off, dwr_off, bar_off, misc_off, zbuf_off;
  uint32_t tx_bytes;
  float* dvp;  // [B*T*N][R][V]: row-block partials of D^T k
  float* dfp;  // [B*T*N][R]:    row-block partials of df
};

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
  // The zero halves of the dW MMA's A operand, written once.
  for (uint32_t i = threadIdx.x; i < kNX * 128u; i += kThreads) {
    const uint32_t slot = i >> 7, part = i & 127u;
    *reinterpret_cast<uint4*>(smem + p.xring_off + slot * kXSlotBytes + kXZero + part * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Warp w of every warpgroup owns value columns 16w..16w+15 (thread columns
  // jcol0 + 8nt + {0,1}, rows g and g+8 of the CTA's block).  Reverse warp w
  // and recompute warp w + 4 share TMEM lanes 32w.. and the same fragment
  // positions, so each reverse thread reads exactly what its recompute
  // partner cached: buffer tb, slot s = columns 16 (C tb + s) .. + 15 holding
  // {Z_s (8 values), H_{s-1} (8 values)}.
  const int w = warp & 3;
  const int g = lane >> 2, qd = lane & 3;
  const int ctid = threadIdx.x & 127;
  const int jcol0 = 16 * w + 2 * qd;
  const int64_t row_g = static_cast<int64_t>(cta_rank) * kRows + g;
  const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
  const uint32_t tcache = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
  const uint32_t xring0 = smem_u32(smem + p.xring_off);

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
    // State gradient C (C-fragment layout), initialised with dH_T.
    float Cg[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (A.dH_T != nullptr) {
        const float* src = A.dH_T + (static_cast<int64_t>(chain) * A.K + row_g) * kV + jcol0 + 8 * nt;
        const float2 x0 = *reinterpret_cast<const float2*>(src);
        const float2 x1 = *reinterpret_cast<const float2*>(src + 8 * kV);
        Cg[nt][0] = x0.x; Cg[nt][1] = x0.y; Cg[nt][2] = x1.x; Cg[nt][3] = x1.y;
      } else {
        Cg[nt][0] = Cg[nt][1] = Cg[nt][2] = Cg[nt][3] = 0.f;
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
      const uint8_t* cbuf = smem + p.cbuf_off + cb * p.cbuf_bytes;
      const uint16_t* cq = reinterpret_cast<const uint16_t*>(cbuf + p.cq_off);
      const uint16_t* ck = reinterpret_cast<const uint16_t*>(cbuf + p.ck_off);
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(cbuf + p.cv_off);
      const float* cdy = reinterpret_cast<const float*>(cbuf + p.cdy_off);
      const float* cf = reinterpret_cast<const float*>(cbuf + p.cf_off);
      const uint32_t tbuf = tcache + kCacheCols * CL * tb;
      // The next slot's TMEM load is issued one step ahead and waited for at
      // the top of the step.
      uint32_t slot_regs[kCacheCols];
      tmem_ld_32x32b<kCacheCols>(tbuf + kCacheCols * (L - 1), slot_regs);
      for (int s = L - 1; s >= 0; --s, ++rs) {
        // The slot is free once the gradient warps have consumed step rs - kNX
        // (tested at the end of the previous step, so that the test's latency
        // overlaps that step's tail; waited for here only if it failed).  A
        // give-up is acted on at the next chunk boundary (the wait raised the
        // CTA's abort flag, so the remaining waits end at once).
        if (!xready && !mbar_wait(smem_u32(&xempty[xs]), xpar ^ 1u, abort_flag, status, kWhereBwdXEmpty))
          *vabort = 1;
        const uint32_t xb = xring0 + xs * kXSlotBytes;
        float* xg = reinterpret_cast<float*>(smem + p.xring_off + xs * kXSlotBytes);
        const float q0 = bf16_bits_to_f32(cq[s * kRows + g]);
        const float q1 = bf16_bits_to_f32(cq[s * kRows + g + 8]);
        const float ft = cf[s];
        const float omf = 1.f - ft;
        float u[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 uu = *reinterpret_cast<const float2*>(cdy + s * kV + jcol0 + 8 * nt);
          u[nt][0] = uu.x;
          u[nt][1] = uu.y;
        }
        tmem_ld_wait();
        tmem_ld_fence_regs(slot_regs);
        float Z[2][4], Hp[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const uint32_t zw = slot_regs[2 * nt + e / 2], hw = slot_regs[4 + 2 * nt + e / 2];
            Z[nt][e] = f16lo(zw);
            Z[nt][e + 1] = f16hi(zw);
            Hp[nt][e] = f16lo(hw);
            Hp[nt][e + 1] = f16hi(hw);
          }
        if (s > 0) tmem_ld_32x32b<kCacheCols>(tbuf + kCacheCols * (s - 1), slot_regs);
        // R = C + q u^T ; D = (1-f) R (1 - Z^2)
        float Rv[2][4], Dv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float qq = (e < 2) ? q0 : q1;
            Rv[nt][e] = fmaf(qq, u[nt][e & 1], Cg[nt][e]);
            const float zz = Z[nt][e];
            Dv[nt][e] = omf * Rv[nt][e] * fmaf(-zz, zz, 1.f);
          }
        }
        // Serial chain: C_{t-1} = f R + D W^T on the warp MMAs.  bf16(D) of
        // this warp's columns is its own k-tile (the accumulator layout of
        // two n-tiles is the A layout of one k-tile): those two MMAs run
        // while the other three k-tiles load from the tile.
        const uint32_t dt = xb + kXDt;
        uint32_t aown[4];
        aown[0] = pack2_bf16(Dv[0][0], Dv[0][1]);
        aown[1] = pack2_bf16(Dv[0][2], Dv[0][3]);
        aown[2] = pack2_bf16(Dv[1][0], Dv[1][1]);
        aown[3] = pack2_bf16(Dv[1][2], Dv[1][3]);
        st_shared_b32(dt + cm_off(g, jcol0), aown[0]);
        st_shared_b32(dt + cm_off(g + 8, jcol0), aown[1]);
        st_shared_b32(dt + cm_off(g, jcol0 + 8), aown[2]);
        st_shared_b32(dt + cm_off(g + 8, jcol0 + 8), aown[3]);
        named_bar_sync(1, 128);
        uint32_t af[3][4];
#pragma unroll
        for (int i = 0; i < 3; ++i) ldmatrix_x4(af[i], cm_ldsm_a(dt, (w + 1 + i) & 3, lane));
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = ft * Rv[nt][e];
          mma_bf16_16816(acc[nt], aown, bt[nt][0][0], bt[nt][0][1]);
        }
#pragma unroll
        for (int i = 0; i < 3; ++i)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(acc[nt], af[i], bt[nt][i + 1][0], bt[nt][i + 1][1]);
        // Off the chain: this thread's shares of dk, dv, df, and bf16 H_{t-1}
        // for dW, handed to the gradient warps.
        {
          const float k0 = bf16_bits_to_f32(ck[s * kRows + g]);
          const float k1 = bf16_bits_to_f32(ck[s * kRows + g + 8]);
          float pk0 = 0.f, pk1 = 0.f, pe = 0.f;
          float* xdv = xg + kXDv / 4;
          const uint32_t ht = xb + kXHt;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int col = jcol0 + 8 * nt;
            const uint32_t vb = *reinterpret_cast<const uint32_t*>(cv + s * kV + col);
            const float v0 = bf16lo(vb), v1 = bf16hi(vb);
            pk0 = fmaf(Dv[nt][0], v0, pk0);
            pk0 = fmaf(Dv[nt][1], v1, pk0);
            pk1 = fmaf(Dv[nt][2], v0, pk1);
            pk1 = fmaf(Dv[nt][3], v1, pk1);
#pragma unroll
            for (int e = 0; e < 4; ++e) pe = fmaf(Rv[nt][e], Hp[nt][e] - Z[nt][e], pe);
            *reinterpret_cast<float2*>(xdv + g * kDvStride + col) =
                make_float2(fmaf(Dv[nt][0], k0, Dv[nt][2] * k1), fmaf(Dv[nt][1], k0, Dv[nt][3] * k1));
            st_shared_b32(ht + cm_off(g, col), pack2_bf16(Hp[nt][0], Hp[nt][1]));
            st_shared_b32(ht + cm_off(g + 8, col), pack2_bf16(Hp[nt][2], Hp[nt][3]));
          }
          *reinterpret_cast<float2*>(xg + kXDk / 4 + (w * 4 + qd) * kDkGroup + 2 * g) = make_float2(pk0, pk1);
          xg[kXDf / 4 + ctid] = pe;
        }
        fence_proxy_async_smem();  // the tiles are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&xfull[xs]));
        if constexpr (kClip) {  // per-step clipping of the state gradient
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = fminf(fmaxf(acc[nt][e], -A.clip), A.clip);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) Cg[nt][e] = acc[nt][e];
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
        *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(Cg[nt][0], Cg[nt][1]);
        *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt) = make_float2(Cg[nt][2], Cg[nt][3]);
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
    float* dqp = reinterpret_cast<float*>(smem + p.dqp_off);  // [C][4 warps][4 qd][8 g][row g, g+8]
    // Start state of a chunk: the checkpoint (H_0, zero if not given, for
    // chunk 0).  The next
    // chunk's is loaded a chunk ahead, so its latency stays off the path.
    auto load_start = [&](int cc, float (&hs)[2][4]) {
      if (cc == 0 && A.H0 == nullptr) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) hs[nt][0] = hs[nt][1] = hs[nt][2] = hs[nt][3] = 0.f;
      } else {
        const float* src =
            (cc == 0 ? A.H0 + (static_cast<int64_t>(chain) * A.K + row_g) * kV
                     : A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (cc - 1)) * A.K + row_g) * kV) +
            jcol0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 x0 = *reinterpret_cast<const float2*>(src + 8 * nt);
          const float2 x1 = *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt);
          hs[nt][0] = x0.x; hs[nt][1] = x0.y; hs[nt][2] = x1.x; hs[nt][3] = x1.y;
        }
      }
    };
    float hnext[2][4];
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
    // Z stash: chunk li's steps into buffer li % nbuf (one bulk copy).
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
      const uint8_t* cbuf = smem + p.cbuf_off + cb * p.cbuf_bytes;
      const uint16_t* ck = reinterpret_cast<const uint16_t*>(cbuf + p.ck_off);
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(cbuf + p.cv_off);
      const float* cdy = reinterpret_cast<const float*>(cbuf + p.cdy_off);
      const float* cf = reinterpret_cast<const float*>(cbuf + p.cf_off);
      const uint32_t tbuf = tcache + kCacheCols * CL * tb;
      float h[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) h[nt][e] = hnext[nt][e];
      if (c > 0) load_start(c - 1, hnext);
      auto dq_share = [&](int s, const float (&h)[2][4]) {
        // dq_t = H_t u_t: this thread's share (its four columns, rows g and
        // g + 8); the sixteen shares of a row are summed at the chunk's end.
        {
          const float2 u0 = *reinterpret_cast<const float2*>(cdy + s * kV + jcol0);
          const float2 u1 = *reinterpret_cast<const float2*>(cdy + s * kV + jcol0 + 8);
          float p0 = h[0][0] * u0.x;
          p0 = fmaf(h[0][1], u0.y, p0);
          p0 = fmaf(h[1][0], u1.x, p0);
          p0 = fmaf(h[1][1], u1.y, p0);
          float p1 = h[0][2] * u0.x;
          p1 = fmaf(h[0][3], u0.y, p1);
          p1 = fmaf(h[1][2], u1.x, p1);
          p1 = fmaf(h[1][3], u1.y, p1);
          *reinterpret_cast<float2*>(dqp + (s * 16 + w * 4 + qd) * kRows + 2 * g) = make_float2(p0, p1);
        }
      };
      if (zs) {
        // Z_t from the stash (written by the tcgen05 forward: per step and
        // row block, Z[8c .. 8c+7][j] as 16 bytes at (c, j)); the state
        // advances by the gate blend alone.  This thread's pairs: rows g, g+8
        // (row runs 0, 1) and columns m0, m0+1, m0+8, m0+9 (m0 = 16w + 2qd).
        const uint16_t* zb = reinterpret_cast<const uint16_t*>(smem + p.zbuf_off) + (16 * w + 2 * qd) * 8 + g;
        for (int s = 0; s < L; ++s) {
          const float omf = 1.f - cf[s];
          const uint16_t* zs_ = zb + s * (kZStepBytes / 2);
          auto pair = [&](int run, int dm) {  // {Z[8 run + g][m0 + dm], Z[8 run + g][m0 + dm + 1]}
            const uint16_t* e = zs_ + (run * kV + dm) * 8;
            return static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[8]) << 16);
          };
          const uint4 zq = make_uint4(pair(0, 0), pair(1, 0), pair(0, 8), pair(1, 8));
          const float z[2][4] = {{f16lo(zq.x), f16hi(zq.x), f16lo(zq.y), f16hi(zq.y)},
                                 {f16lo(zq.z), f16hi(zq.z), f16lo(zq.w), f16hi(zq.w)}};
          // The cache takes Z_s as stashed (already fp16 pairs) and H_{s-1}.
          const uint32_t cache[kCacheCols] = {zq.x, zq.y, zq.z, zq.w,
                                              pack2_f16(h[0][0], h[0][1]), pack2_f16(h[0][2], h[0][3]),
                                              pack2_f16(h[1][0], h[1][1]), pack2_f16(h[1][2], h[1][3])};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) h[nt][e] = fmaf(omf, z[nt][e] - h[nt][e], h[nt][e]);
          tmem_st_32x32b_x8(tbuf + kCacheCols * s, cache);
          dq_share(s, h);
        }
        // Every read of this Z buffer and every dq share of the chunk is done.
        named_bar_sync(2, 128);
        if (loader && zissued < p.nchunks) issue_z(zissued++);
      } else {
        // Step s, as in the forward: acc = k_s v_s^T + fp16(H_{s-1}) W, the
        // own k-tile from registers while the other three load from the tile.
        uint32_t hh[4];
        auto split = [&]() {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            hh[2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
            hh[2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
          }
        };
        auto store_tile = [&](uint32_t base) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int col = jcol0 + 8 * nt;
            st_shared_b32(base + tile_off(g, col), hh[2 * nt]);
            st_shared_b32(base + tile_off(g + 8, col), hh[2 * nt + 1]);
          }
        };
        split();
        store_tile(htile0);
        named_bar_sync(2, 128);
        for (int s = 0; s < L; ++s) {
          const float omf = 1.f - cf[s];
          const uint32_t atile = htile0 + (s & 1) * 2048;
          uint32_t af[3][4];
#pragma unroll
          for (int i = 0; i < 3; ++i) ldmatrix_x4(af[i], ldsm_addr_a(atile, (w + 1 + i) & 3, lane));
          float acc[2][4];
          const float k0 = bf16_bits_to_f32(ck[s * kRows + g]);
          const float k1 = bf16_bits_to_f32(ck[s * kRows + g + 8]);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(cv + s * kV + jcol0 + 8 * nt);
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
          uint32_t cache[kCacheCols];  // Z_s and H_{s-1} as fp16 pairs
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            float z[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) z[e] = tanh_fast(acc[nt][e]);
            cache[2 * nt] = pack2_f16(z[0], z[1]);
            cache[2 * nt + 1] = pack2_f16(z[2], z[3]);
            cache[4 + 2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
            cache[4 + 2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[nt][e] = fmaf(omf, z[e] - h[nt][e], h[nt][e]);
          }
          split();
          store_tile(htile0 + ((s + 1) & 1) * 2048);
          tmem_st_32x32b_x8(tbuf + kCacheCols * s, cache);
          dq_share(s, h);
          named_bar_sync(2, 128);
        }
      }
      tmem_st_wait();
      if (more) publish_chunk(ci + 1, fnext);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tready[tb]));
      issued = ci + 2;
      // dq rows of the chunk (the last step's barrier ordered every share):
      // the sixteen shares of row r = g + 8 hi, warp by warp, in a fixed order.
      for (int idx = ctid; idx < L * kRows; idx += 128) {
        const int sp = idx >> 4, r = idx & 15;
        const float* pp = dqp + sp * 16 * kRows + 2 * (r & 7) + (r >> 3);
        float sum = 0.f;
#pragma unroll
        for (int sh = 0; sh < 16; ++sh) sum += pp[sh * kRows];
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
    // accumulator in TMEM columns 448..511):
    //   dW (+)= [H_{t-1}^T ; 0] (128 x 16) * D (16 x 64),
    // committed to the slot's empty barrier.  Every fourth step (rs % 4 == w)
    // warp 8 + w also sums that step's dk, dv and df shares.
    float dwr0 = 0.f, dwr1 = 0.f;  // dw_r columns 2 lane, 2 lane + 1 (row block 0 only)
    const int r16 = lane & 15, hh = lane >> 4;
    const uint32_t idesc = idesc_bf16_f32(128, kV, /*a_mn_major=*/true, /*b_mn_major=*/true);
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
      const uint8_t* cbuf = smem + p.cbuf_off + cb * p.cbuf_bytes;
      const uint16_t* cv = reinterpret_cast<const uint16_t*>(cbuf + p.cv_off);
      const float* cdy = reinterpret_cast<const float*>(cbuf + p.cdy_off);
      for (int s = L - 1; s >= 0; --s, ++rs) {
        const bool duty = (rs & 3) == w;
        const uint32_t xb = xring0 + xs * kXSlotBytes;
        const float* xg = reinterpret_cast<const float*>(smem + p.xring_off + xs * kXSlotBytes);
        // A give-up is acted on at the next chunk boundary.
        if ((w == 0 || duty) && !mbar_wait(smem_u32(&xfull[xs]), xpar, abort_flag, status, kWhereBwdXFull))
          *gabort = 1;
        if (w == 0) {
          tc_fence_after_sync();
          if (elect_one()) {
            tc_mma_f16_ss(dw_tmem, smem_desc_noswizzle(xb + kXHt, 128, 256),
                          smem_desc_noswizzle(xb + kXDt, 128, 256), idesc, rs > 0 ? 1u : 0u);
            tc_commit(smem_u32(&xempty[xs]));  // arrives once the MMA has read the slot
          }
          __syncwarp();
        }
        if (duty) {
          const int64_t rowt = (static_cast<int64_t>(b) * T + s0 + s) * N + n;
          // dk_t = D_t v_t: lane -> row r16 = g + 8 hi; warps 2 hh, 2 hh + 1 and
          // their four qd shares, then the two halves (fixed order).
          {
            const int gg = r16 & 7, hi = r16 >> 3;
            const float* xk = xg + kXDk / 4 + 2 * gg + hi;
            float pk = 0.f;
#pragma unroll
            for (int ww = 0; ww < 2; ++ww)
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) pk += xk[((2 * hh + ww) * 4 + qq) * kDkGroup];
            pk += __shfl_xor_sync(0xffffffffu, pk, 16);
            if (lane < 16) A.dk[rowt * A.K + cta_rank * kRows + r16] = pk;
          }
          // Row-block partial of D_t^T k_t: lane -> columns 2 lane, 2 lane + 1.
          {
            const float* xdv = xg + kXDv / 4 + 2 * lane;
            float2 a2 = *reinterpret_cast<const float2*>(xdv);
#pragma unroll
            for (int gg = 1; gg < 8; ++gg) {
              const float2 x = *reinterpret_cast<const float2*>(xdv + gg * kDvStride);
              a2.x += x.x;
              a2.y += x.y;
            }
            *reinterpret_cast<float2*>(p.dvp + (rowt * R + cta_rank) * kV + 2 * lane) = a2;
          }
          // Row-block partial of df_t = <R_t, H_{t-1} - Z_t>.
          {
            const float4 e4 = *reinterpret_cast<const float4*>(xg + kXDf / 4 + 4 * lane);
            float pf = (e4.x + e4.y) + (e4.z + e4.w);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) pf += __shfl_xor_sync(0xffffffffu, pf, o);  // fixed tree
            if (lane == 0) p.dfp[rowt * R + cta_rank] = pf;
          }
          if (cta_rank == 0) {  // dw_r += u_t * v_t, once per chain
            const float2 uu = *reinterpret_cast<const float2*>(cdy + s * kV + 2 * lane);
            const uint32_t vb = *reinterpret_cast<const uint32_t*>(cv + s * kV + 2 * lane);
            dwr0 = fmaf(uu.x, bf16lo(vb), dwr0);
            dwr1 = fmaf(uu.y, bf16hi(vb), dwr1);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&xempty[xs]));
        }
        if (++xs == kNX) {
          xs = 0;
          xpar ^= 1u;
        }
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
      // dW partial of this row block from TMEM: accumulator row m = lane 32w + lane
      // (rows 64..127 are the zero padding), column n = 448 + n.
      if (w < 2) {
        if (!mbar_wait_timed(smem_u32(dwdone), 0, status, kWhereBwdDW)) *gabort = 1;
        tc_fence_after_sync();
        float* dwp = A.dW_part + static_cast<int64_t>(blockIdx.x) * kV * kV + (32 * w + lane) * kV;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld_32x32b<32>(tmem_base + (static_cast<uint32_t>(32 * w) << 16) + kDWCol + 32 * half, r);
          tmem_ld_wait();
          tmem_ld_fence_regs(r);
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4)
            *reinterpret_cast<float4*>(dwp + 32 * half + c4) =
                make_float4(__uint_as_float(r[c4]), __uint_as_float(r[c4 + 1]), __uint_as_float(r[c4 + 2]),
                            __uint_as_float(r[c4 + 3]));
        }
      }
      // dw_r: the four warps' step subsets, summed in a fixed order.
      float* sd = reinterpret_cast<float*>(smem + p.dwr_off);
      *reinterpret_cast<float2*>(sd + w * kV + 2 * lane) = make_float2(dwr0, dwr1);
      named_bar_sync(3, 128);
      if (cta_rank == 0 && w == 0) {
        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) {
          const float2 x = *reinterpret_cast<const float2*>(sd + ww * kV + 2 * lane);
          acc2.x += x.x;
          acc2.y += x.y;
        }
        *reinterpret_cast<float2*>(A.dwr_part + static_cast<int64_t>(chain) * kV + 2 * lane) = acc2;
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
// df = sum over the row blocks.  One warp per (b, t, n).
__global__ void __launch_bounds__(256) mma_backward_rows_kernel(const float* __restrict__ dvp,
                                                                const float* __restrict__ dfp,
                                                                const float* __restrict__ dy,
                                                                const uint16_t* __restrict__ w_r,
                                                                float* __restrict__ dv, float* __restrict__ df,
                                                                int64_t rows, int N, int R) {
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
      for (int pr = 0; pr < R; ++pr) sf += dfp[row * R + pr];
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
  p.dqp_off = p.xring_off + kNX * kXSlotBytes;
  p.dwr_off = p.dqp_off + kMaxChunk * 16 * kRows * 4;
  p.bar_off = p.dwr_off + 4 * kV * 4;
  p.misc_off = p.bar_off + (2 * kCBufs + 4 + 2 * kNX + 1 + 2) * 8;
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
                                                       a.dv, a.df, static_cast<int64_t>(rows), a.N, p.R);
  return cudaGetLastError();
}

}  // namespace m2rnn
