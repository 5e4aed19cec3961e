// Register-resident forward scan for V = 64 value columns (bf16 inputs, fp32
// state): the latency-optimised kernel for small-state, long-sequence work.
//
// Recurrence (reading notes on "M2RNN: Non-Linear RNNs with Matrix-Valued
// States for Scalable Language Modeling", section 2.1, Eq. 10-12):
//   Z_t = tanh(H_{t-1} W + k_t v_t^T),  H_t = f_t H_{t-1} + (1-f_t) Z_t,
//   y_t = H_t^T q_t + w_r * v_t.
//
// Each chain (b, n) is split into K/16 row blocks (key rows never mix, notes
// section 1.2), one CTA each; the CTAs of a chain form a cluster and sum the
// readout through distributed shared memory, as in the tensor-memory kernel.
// Inside a CTA four compute warps own 16 value columns each of the 16 x 64
// state.  Per step a warp runs D = H_{t-1} * W[:, its 16 columns] + k v^T as
// eight m16n8k16 warp MMAs with fp16 operands (H_{t-1} rounded to fp16, W
// re-encoded as fp16 and held in registers for the whole scan; the rank-1
// write seeds the accumulator exactly), applies tanh and the gate blend to
// its 8 fp32 state values per thread, and writes fp16(H_t) to a swizzled
// shared tile that the four warps read back with ldmatrix after one named
// barrier.  The readout runs on four readout warps, one per compute warp on
// the same scheduler and tensor-memory lane quadrant: the compute warp leaves
// H_t (its fp16 A-operand pairs, 4 columns per step) in a double-buffered
// tile of tensor memory,
// and the readout warp, one tile of 32 steps behind, forms y^T = q^T H_t as
// one m16n8k16 per column tile with fp16 operands: q replicated over the A
// rows (staged in fp16 by the producer warp, which checks its range) and
// those H_t pairs, transposed into B fragments with movmatrix, as B, so the sum
// over rows needs no shuffles; it stores each step's share one step late,
// so that no step waits for its own MMAs.  A
// dependent m16n8k16 takes ~21 cycles, while a 4-instruction tcgen05 step
// costs several hundred cycles from issue to completion (measured on GB300).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "internal.h"
#include "gate.cuh"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 64;
constexpr int kRows = 16;   // key rows per CTA
constexpr int kS = 32;      // steps per input tile
constexpr int kNS = 4;      // input stages
constexpr int kYS = 2;      // readout partial stages
// Warps: 0-3 compute (8 / NT of them, each owning 8*NT of the 64 value
// columns), 4-7 readout, 8 the producer (k, v by TMA; q and f by its
// lanes), 9 the readout reducer.
template <int NT>
constexpr int kThreadsFor() { return 10 * 32; }
constexpr int kReadoutWarp0 = 4, kProducerWarp = 8, kReducerWarp = 9;
constexpr int kHCols = 4;  // tensor-memory columns per step of H_t (fp16 pairs, the exchange's A-fragment order)

struct MmaFwdParams {
  FwdArgs a;
  int R;
  int ntiles;
  int stall_tile;  // test hook: the producer never completes this tile (-1: off)
  uint32_t abuf_off, stage_off, stage_bytes, q_off, k_off, v_off, f_off, y_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

// Compile-time modes (a per-step branch costs ~20-30 ns of a ~250 ns step,
// measured): kY = readout y, kCk = checkpoints, kZ = the Z stash for the
// backward.  The V = 64 stash: per (chain, row block) and step 2 KB, compute
// warp w's lane L writing its 16 bytes at (32 w + L) * 16, its fp16 Z values
// in accumulator-fragment order (column block 0, row g), (0, g+8), (1, g),
// (1, g+8) -- the order in which the backward's recompute warps hold them --
// so a chunk of steps is one contiguous range.
template <int NT, bool kY, bool kCk, bool kZ>
__global__ void __launch_bounds__(kThreadsFor<NT>(), 1)
    mma_forward_kernel(const __grid_constant__ MmaFwdParams p, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int R = p.R;
  const int T = p.a.T, N = p.a.N;
  const int cta_rank = static_cast<int>(blockIdx.x) % R;
  const int chain = static_cast<int>(blockIdx.x) / R;
  const int b = chain / N, n = chain % N;
  const int ntiles = p.ntiles;
  constexpr bool do_y = kY;
  StatusBlock* status = p.a.status;
  constexpr int CW = 8 / NT;        // compute warps
  constexpr int NCOL = 8 * NT;      // value columns per compute warp
  constexpr int CT = CW * 32;       // compute threads (named barrier 1)

  uint8_t* sStage = smem + p.stage_off;
  float* sY = reinterpret_cast<float*>(smem + p.y_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* full = bars;
  uint64_t* empty = full + kNS;
  uint64_t* yfull = empty + kNS;
  uint64_t* ypeer = yfull + kYS;
  uint64_t* yempty = ypeer + kYS;
  uint64_t* hfull = yempty + kYS;  // [4 compute warps][2 tiles]: a tile's H_t is in tensor memory
  uint64_t* hempty = hfull + 8;    // [4][2]: it has been read out
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* cabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  volatile int* rabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 12);
  const uint32_t abuf0 = smem_u32(smem + p.abuf_off);  // two 2 KB fp16 tiles

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&full[i]), 32);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kYS; ++i) {
      mbar_init(smem_u32(&yfull[i]), 1);
      mbar_init(smem_u32(&ypeer[i]), R);
      mbar_init(smem_u32(&yempty[i]), R);
    }
    for (int i = 0; i < 16; ++i) mbar_init(smem_u32(&hfull[i]), 1);
    *abort_flag = 0;
    *cabort = 0;
    *rabort = 0;
    fence_mbar_init_cluster();
  }
  if (do_y && warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  for (int e = threadIdx.x; e < 2 * 2048 / 16; e += static_cast<int>(blockDim.x))
    reinterpret_cast<uint4*>(smem + p.abuf_off)[e] = make_uint4(0, 0, 0, 0);  // H_0 = 0
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = do_y ? *tmem_slot : 0u;

  if (warp < CW) {
    // ---------------- compute warps ----------------
    static_assert(NT == 2, "four compute warps of 16 value columns");
    const int g = lane >> 2, qd = lane & 3;
    const int w = warp;
    // W fragments for this warp's output columns: B[k][n] = W[k][16 w + n].
    // A warp's 16 columns of H are one k-tile, whose A fragments it holds in
    // registers: the k-tiles are stored in the order w, w+1, w+2, w+3 (mod 4)
    // so that the first is its own.
    const uint16_t* Wg = static_cast<const uint16_t*>(p.a.W) + static_cast<int64_t>(n) * kV * kV;
    uint32_t bw[2][4][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = NCOL * w + 8 * nt + g;
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
    // State: h[nt][0..3] = H[g][j], H[g][j+1], H[g+8][j], H[g+8][j+1], j = 16 w + 8nt + 2qd.
    float h[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) h[nt][c] = 0.f;
    const int jcol0 = NCOL * w + 2 * qd;
    const int64_t row_g = static_cast<int64_t>(cta_rank) * kRows + g;
    // fp16 H_{t-1} as the MMA operand (see mma_common.cuh).  hh: this warp's
    // own k-tile (accumulator layout = A layout); the exchange tile holds
    // all four k-tiles.
    uint32_t hh[4] = {0u, 0u, 0u, 0u};
    auto split = [&]() {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        hh[2 * nt] = pack2_f16(h[nt][0], h[nt][1]);
        hh[2 * nt + 1] = pack2_f16(h[nt][2], h[nt][3]);
      }
    };
    auto store_tiles = [&](uint32_t base) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = jcol0 + 8 * nt;
        st_shared_b32(base + tile_off(g, col), hh[2 * nt]);
        st_shared_b32(base + tile_off(g + 8, col), hh[2 * nt + 1]);
      }
    };
    if (p.a.H0 != nullptr) {
      // Start from the given state: fp32 into the registers, fp16 into the
      // operand tile of step 0 (ordered by the first tile's barrier).
      const float* src = p.a.H0 + (static_cast<int64_t>(chain) * p.a.K + row_g) * kV + jcol0;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float2 x0 = *reinterpret_cast<const float2*>(src + 8 * nt);
        const float2 x1 = *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt);
        h[nt][0] = x0.x; h[nt][1] = x0.y; h[nt][2] = x1.x; h[nt][3] = x1.y;
      }
      split();
      store_tiles(abuf0);
    }
    int ck_left = p.a.ckpt_every, ck_idx = 0;  // countdown to the next checkpoint (no division per step)
    const uint32_t th = tmem_base + (static_cast<uint32_t>(32 * w) << 16);  // this warp's lane quadrant
    uint8_t* const zst = !kZ ? nullptr
                             : reinterpret_cast<uint8_t*>(p.a.zstash) +
                                   (static_cast<int64_t>(chain) * R + cta_rank) * T * kZStepBytes + (32 * w + lane) * 16;
    bool ok = true;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int st = tile % kNS, hb = tile & 1;
      bool mine = mbar_wait_timed(smem_u32(&full[st]), (tile / kNS) & 1, status, kWhereFwdFull);
      if (mine && do_y && tile >= 2)  // the tensor-memory tile has been read out
        mine = mbar_wait(smem_u32(&hempty[2 * w + hb]), ((tile >> 1) - 1) & 1, abort_flag, status, kWhereFwdYEmpty);
      if (!mine) *cabort = 1;
      named_bar_sync(1, CT);
      if (*cabort) {  // every compute warp reads the flag after the same barrier
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(stage + p.k_off);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(stage + p.v_off);
      const float* fs = reinterpret_cast<const float*>(stage + p.f_off);
      const uint32_t tt = th + static_cast<uint32_t>(hb * kS * kHCols);
      const int nsteps = min(kS, T - tile * kS);
      // Steps run in segments that end where a checkpoint is due, so the
      // step itself carries no checkpoint test.
      for (int s = 0; s < nsteps;) {
        const int seg_end = kCk ? min(nsteps, s + ck_left) : nsteps;
        const int seg_len = seg_end - s;
        for (; s < seg_end; ++s) {
          const int t = tile * kS + s;
          // Inputs of step t.
          const float k0 = bf16_bits_to_f32(ks[s * kRows + g]);
          const float k1 = bf16_bits_to_f32(ks[s * kRows + g + 8]);
          const float omf = 1.f - fs[s];
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(vs + s * kV + jcol0 + 8 * nt);
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            acc[nt][0] = k0 * v0;  // exact: products of bf16 values fit in fp32
            acc[nt][1] = k0 * v1;
            acc[nt][2] = k1 * v0;
            acc[nt][3] = k1 * v1;
          }
          // H_{t-1} as the A operand: the own k-tile from registers, issued
          // while the other three load from the tile.
          const uint32_t atile = abuf0 + (t & 1) * 2048;
          uint32_t af[3][4];
#pragma unroll
          for (int i = 0; i < 3; ++i) ldmatrix_x4(af[i], ldsm_addr_a(atile, (w + 1 + i) & 3, lane));
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) mma_f16_16816(acc[nt], hh, bw[nt][0][0], bw[nt][0][1]);
          // Two accumulation chains (f16 products, fp32 sums) for the other
          // three k-tiles: two dependent MMAs after the tile loads, not three.
          float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            mma_f16_16816(acc[nt], af[0], bw[nt][1][0], bw[nt][1][1]);
            mma_f16_16816(acc2[nt], af[1], bw[nt][2][0], bw[nt][2][1]);
          }
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            mma_f16_16816(acc2[nt], af[2], bw[nt][3][0], bw[nt][3][1]);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] += acc2[nt][e];
          }
          // Eq. 10-11 on this thread's 8 state values; fp16 H_t to the other tile.
          float zv[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              zv[nt][c] = tanh_fast(acc[nt][c]);
              h[nt][c] = fmaf(omf, zv[nt][c] - h[nt][c], h[nt][c]);
            }
          split();
          store_tiles(abuf0 + ((t + 1) & 1) * 2048);
          if constexpr (kZ)  // Z_t for the backward (a streaming store, off the chain)
            st_global_cs_v4(zst + static_cast<int64_t>(t) * kZStepBytes,
                            make_uint4(pack2_f16(zv[0][0], zv[0][1]), pack2_f16(zv[0][2], zv[0][3]),
                                       pack2_f16(zv[1][0], zv[1][1]), pack2_f16(zv[1][2], zv[1][3])));
          // H_t for the readout warp: the fp16 pairs just packed as the next
          // step's A operand, which are also the readout's B operand.
          if constexpr (kY) tmem_st_32x32b_x4(tt + kHCols * s, hh);
          named_bar_sync(1, CT);
        }
        if constexpr (kCk) {
          ck_left -= seg_len;
          if (ck_left == 0) {  // H after step t = tile kS + s - 1 starts a chunk: checkpoint it
            ck_left = p.a.ckpt_every;
            ++ck_idx;
            if (tile * kS + s < T) {
              float* dst = p.a.ckpt +
                           ((static_cast<int64_t>(chain) * p.a.n_ckpt + ck_idx - 1) * p.a.K + row_g) * kV + jcol0;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(h[nt][0], h[nt][1]);
                *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt) = make_float2(h[nt][2], h[nt][3]);
              }
            }
          }
        }
      }
      if constexpr (kY) {  // the tile's H_t for the readout warp, which also releases the stage
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&hfull[2 * w + hb]));
      } else {
        // Every compute warp is past its last read of this stage.
        if (threadIdx.x == 0) mbar_arrive(smem_u32(&empty[st]));
      }
    }
    if (ok) {
      if (p.a.H_T != nullptr) {
        float* dst = p.a.H_T + (static_cast<int64_t>(chain) * p.a.K + row_g) * kV + jcol0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(h[nt][0], h[nt][1]);
          *reinterpret_cast<float2*>(dst + 8 * kV + 8 * nt) = make_float2(h[nt][2], h[nt][3]);
        }
      }
    } else {
      *abort_flag = 1;
    }
  } else if (do_y && warp >= kReadoutWarp0 && warp < kReadoutWarp0 + CW) {
    // ---------------- readout warps ----------------
    // y_t share of this CTA's 16 rows for compute warp w's 16 columns, one
    // tile behind: y^T = q^T H_t with q replicated over the A rows and H_t
    // (bf16 high and low parts, transposed with movmatrix) as B.
    const int g = lane >> 2, qd = lane & 3;
    const int w = warp - kReadoutWarp0;
    const int jcol0 = NCOL * w + 2 * qd;
    const uint32_t th = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
    for (int tile = 0; tile < ntiles; ++tile) {
      const int st = tile % kNS, ys = tile % kYS, hb = tile & 1;
      bool mine = mbar_wait(smem_u32(&full[st]), (tile / kNS) & 1, abort_flag, status, kWhereFwdFull) &&
                  mbar_wait(smem_u32(&hfull[2 * w + hb]), (tile >> 1) & 1, abort_flag, status, kWhereFwdYFull);
      if (mine && tile >= kYS)
        mine = mbar_wait<true>(smem_u32(&yempty[ys]), ((tile / kYS) - 1) & 1, abort_flag, status, kWhereFwdYEmpty);
      if (!mine) *rabort = 1;
      const uint8_t* stage = sStage + st * p.stage_bytes;
      const uint32_t qs = smem_u32(stage + p.q_off);
      const int nsteps = min(kS, T - tile * kS);
      if (mine) {
        tc_fence_after_sync();
        const uint32_t tt = th + static_cast<uint32_t>(hb * kS * kHCols);
        uint32_t hr[4];
        tmem_ld_32x32b<4>(tt, hr);
        float yprev[4] = {0.f, 0.f, 0.f, 0.f};  // the previous step's share (stored one step late)
        uint32_t qlo = ld_shared_b32(qs + 4 * qd), qhi = ld_shared_b32(qs + 4 * qd + 16);
#pragma unroll 2
        for (int s = 0; s < nsteps; ++s) {
          const int sn = s + 1 < nsteps ? s + 1 : s;
          // q of the CTA's rows 2qd.. and 2qd+8.. of the next step, as bf16 pairs.
          const uint32_t nqlo = ld_shared_b32(qs + 2 * (sn * kRows + 2 * qd));
          const uint32_t nqhi = ld_shared_b32(qs + 2 * (sn * kRows + 2 * qd + 8));
          tmem_ld_wait();
          tmem_ld_fence_regs(hr);
          const uint32_t hc[4] = {hr[0], hr[1], hr[2], hr[3]};  // H_t, fp16 pairs
          tmem_ld_32x32b<4>(tt + kHCols * sn, hr);
          // y in fp16 operands: H_t (|H| <= 1) to fp16 as in the state
          // transform; q as staged in fp16 by the producer.
          const uint32_t qa[4] = {qlo, qlo, qhi, qhi};
          float yd[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma_f16_16816_zc(yd[nt], qa, movmatrix_trans(hc[2 * nt]), movmatrix_trans(hc[2 * nt + 1]));
          if (g == 0 && s > 0) {  // row 0 of the row-replicated result: columns 8nt + 2qd (+1)
            float* dst = sY + (ys * kS + s - 1) * kV + jcol0;
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
          float* dst = sY + (ys * kS + nsteps - 1) * kV + jcol0;
          *reinterpret_cast<float2*>(dst) = make_float2(yprev[0], yprev[1]);
          *reinterpret_cast<float2*>(dst + 8) = make_float2(yprev[2], yprev[3]);
        }
        // The tile's H has been read (the last, repeated load included).
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&hempty[2 * w + hb]));
      }
      named_bar_sync(2, CT);  // every readout warp's shares of the tile are written
      if (*rabort) break;
      if (threadIdx.x == 32 * kReadoutWarp0) {
        mbar_arrive(smem_u32(&yfull[ys]));
        mbar_arrive(smem_u32(&empty[st]));  // compute and readout warps are past the stage
      }
    }
    if (*rabort) *abort_flag = 1;
  } else if (warp == kProducerWarp) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const GateSrc gs{p.a.f, p.a.gate_a, p.a.gate_alpha, p.a.gate_beta, true};
    int issued = 0;
    bool ok = true;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int st = tile % kNS;
      if (tile >= kNS &&
          !mbar_wait(smem_u32(&empty[st]), ((tile / kNS) - 1) & 1, abort_flag, status, kWhereFwdEmpty)) {
        ok = false;
        break;
      }
      if (tile == p.stall_tile) {  // failure-detection test: this stage never fills
        issued = tile + 1;
        continue;
      }
      const int t0 = tile * kS;
      uint8_t* stage = sStage + st * p.stage_bytes;
      float fv = 0.f;
      if (t0 + lane < T) fv = gate_value(gs, (static_cast<int64_t>(b) * T + t0 + lane) * N + n, n);
      reinterpret_cast<float*>(stage + p.f_off)[lane] = fv;
      if constexpr (kY) {
        // q of step t0 + lane (the CTA's 16 rows), re-encoded as fp16 for
        // the readout's MMA once here instead of at every readout step; a
        // magnitude the fp16 operand cannot hold is reported.
        uint4 qv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
        if (t0 + lane < T) {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const uint16_t*>(p.a.q) +
              ((static_cast<int64_t>(b) * T + t0 + lane) * qk_heads(p.a.qkN, N) + qk_head(p.a.qkN, n)) * p.a.K +
              cta_rank * kRows);
          qv[0] = src[0];
          qv[1] = src[1];
        }
        uint32_t mag = 0u;
        uint32_t* qw = reinterpret_cast<uint32_t*>(qv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mag = __vmaxu2(mag, qw[i] & 0x7FFF7FFFu);
          qw[i] = bf16x2_to_f16x2(qw[i]);
        }
        if ((mag & 0xFFFFu) >= 0x4780u || (mag >> 16) >= 0x4780u)  // |q| >= 65536 (or not finite)
          report_device_error(status, kStatusCheck, kWhereQRange);
        uint4* dst = reinterpret_cast<uint4*>(stage + p.q_off + lane * kRows * 2);
        dst[0] = qv[0];
        dst[1] = qv[1];
      }
      __syncwarp();
      const uint32_t fb = smem_u32(&full[st]);
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, p.tx_bytes);
        tma_load_4d(smem_u32(stage + p.k_off), &tm_k, fb, cta_rank * kRows, qk_head(p.a.qkN, n), t0, b);
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
  } else if (warp == kReducerWarp && do_y) {
    // ---------------- readout reducer (sum over the chain's row blocks) ----------------
    const uint16_t* vg = static_cast<const uint16_t*>(p.a.v);
    const uint16_t* wr = static_cast<const uint16_t*>(p.a.w_r) + static_cast<int64_t>(n) * kV;
    const float wr0 = bf16_bits_to_f32(wr[2 * lane]), wr1 = bf16_bits_to_f32(wr[2 * lane + 1]);
    int done = 0;
    for (int tile = 0; tile < ntiles; ++tile) {
      const int ys = tile % kYS;
      const uint32_t par = (tile / kYS) & 1;
      const int t0 = tile * kS;
      const int nsteps = min(kS, T - t0);
      // v_t of this CTA's steps of the tile (s = cta_rank + i R), loaded
      // before the waits so that their latency overlaps them.
      uint32_t vr[kS];
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int s = cta_rank + i * R;
        vr[i] = s < nsteps ? *reinterpret_cast<const uint32_t*>(
                                 vg + ((static_cast<int64_t>(b) * T + t0 + s) * N + n) * kV + 2 * lane)
                           : 0u;
      }
      if (!mbar_wait(smem_u32(&yfull[ys]), par, abort_flag, status, kWhereFwdYFull)) break;
      fence_acq_rel_cluster();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&ypeer[ys]), lane));
      if (!mbar_wait<true>(smem_u32(&ypeer[ys]), par, abort_flag, status, kWhereFwdYPeer)) break;
      const uint32_t ybase = smem_u32(sY + ys * kS * kV);
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int s = cta_rank + i * R;
        if (s < nsteps) {
          const int64_t row = (static_cast<int64_t>(b) * T + t0 + s) * N + n;
          float a0 = 0.f, a1 = 0.f;
          for (int pr = 0; pr < R; ++pr) {  // fixed order over the chain's row blocks
            const uint32_t ra = mapa_shared(ybase, pr) + static_cast<uint32_t>((s * kV + 2 * lane) * 4);
            a0 += ld_shared_cluster_f32(ra);
            a1 += ld_shared_cluster_f32(ra + 4);
          }
          *reinterpret_cast<float2*>(p.a.y + row * kV + 2 * lane) =
              make_float2(fmaf(wr0, bf16lo(vr[i]), a0), fmaf(wr1, bf16hi(vr[i]), a1));
        }
      }
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&yempty[ys]), lane));
      done = tile + 1;
    }
    for (int tile = std::max(0, done - kYS); tile < done; ++tile) {
      if (!mbar_wait<true>(smem_u32(&yempty[tile % kYS]), (tile / kYS) & 1, abort_flag, status, kWhereFwdExit))
        break;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (do_y && warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int NT, bool kY, bool kCk, bool kZ>
cudaError_t launch_nt(const FwdArgs& a, cudaStream_t stream) {
  MmaFwdParams p{};
  p.a = a;
  p.R = a.K / kRows;
  p.ntiles = (a.T + kS - 1) / kS;
  // Test hook for failure detection (single-CTA chains only, so no cluster
  // peer is left waiting): the stall-tile option n >= 0 makes tile n never
  // arrive; the consumers' bounded waits expire and the status block reports it.
  p.stall_tile = p.R == 1 ? option_test_stall_tile() : -1;
  p.abuf_off = 0;
  p.stage_off = 4096;
  p.q_off = 0;
  p.k_off = align_up(kS * kRows * 2, 128);
  p.v_off = p.k_off + align_up(kS * kRows * 2, 128);
  p.f_off = p.v_off + align_up(kS * kV * 2, 128);
  p.stage_bytes = align_up(p.f_off + kS * 4, 128);
  p.y_off = p.stage_off + kNS * p.stage_bytes;
  p.bar_off = p.y_off + kYS * kS * kV * 4;
  p.misc_off = p.bar_off + (2 * kNS + 3 * kYS + 16) * 8;
  uint32_t smem = align_up(p.misc_off + 16, 128) + 1024;  // + the 1 KB alignment slack
  smem = std::max<uint32_t>(smem, 120 * 1024);  // one CTA per SM
  p.tx_bytes = kS * kRows * 2 + kS * kV * 2;  // k and v by TMA (q is staged by the producer's lanes)

  CUtensorMap mk, mv;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int qN = qk_heads(a.qkN, a.N);
  if (!make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, qN, a.K, kRows, kS) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, kS))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(mma_forward_kernel<NT, kY, kCk, kZ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.N * p.R));
  cfg.blockDim = dim3(kThreadsFor<NT>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.R);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mma_forward_kernel<NT, kY, kCk, kZ>, p, mk, mv);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// The warp-MMA family: V = 64 here, V = 16 in the register-resident kernel.
bool mma_forward_supported(int K, int V) {
  return (V == kV && K % kRows == 0 && K >= kRows && K <= 128) || mv_forward_supported(K, V);
}

cudaError_t launch_mma_forward(const FwdArgs& a, cudaStream_t stream) {
  if (a.V != kV) return launch_mv_forward(a, stream);
  const bool y = a.y != nullptr, ck = a.ckpt != nullptr;
  if (a.zstash != nullptr) {  // the training forward: readout, checkpoints and the stash
    if (y) return ck ? launch_nt<2, true, true, true>(a, stream) : launch_nt<2, true, false, true>(a, stream);
    return ck ? launch_nt<2, false, true, true>(a, stream) : launch_nt<2, false, false, true>(a, stream);
  }
  if (y) return ck ? launch_nt<2, true, true, false>(a, stream) : launch_nt<2, true, false, false>(a, stream);
  return ck ? launch_nt<2, false, true, false>(a, stream) : launch_nt<2, false, false, false>(a, stream);
}

}  // namespace m2rnn

