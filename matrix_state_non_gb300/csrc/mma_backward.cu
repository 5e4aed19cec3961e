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
// block, the blocks of a chain in one cluster (only dv_t and df_t sum over
// rows; dW is summed later over row blocks and batch in a fixed order).
// The time axis runs over chunks of C <= 32 steps, last chunk first.  For
// each chunk the forward is rerun from its checkpoint (section 2.6 of the
// notes describes the paper's rerun-and-cache backward; here only one or two
// chunks are cached), each thread caching its own Z_t and H_{t-1} values
// (fp32) in its own lane of tensor memory, so the cache never touches DRAM;
// then the chunk is walked backwards.  The two jobs run on separate warps:
// four recompute warps and four reverse warps, each owning 16 value columns,
// paired on the SM's four schedulers so that one's latency hides the other's.
// With C <= 16 two caches fit in the 512 TMEM columns and the recompute of
// chunk c-1 overlaps the reverse walk of chunk c; with 16 < C <= 32 the two
// alternate.  Per reverse step the serial chain is R -> D -> bf16(D) tile ->
// one named barrier -> 8 warp MMAs seeded with f R -> C_{t-1}.  Off the
// chain: dW += H_{t-1}^T D as 8 more warp MMAs per warp into register
// accumulators (H_{t-1}^T fragments by movmatrix, D fragments by
// ldmatrix.trans), and the row/column reductions for dq, dk, dv, df, also as
// warp MMAs against replicated vectors (no shuffle chains), written as
// per-step partials that a reducer warp sums (over warps, and over the
// cluster's CTAs for dv, df) and stores.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "mma_common.cuh"

namespace m2rnn {
namespace {

constexpr int kV = 64;
constexpr int kRows = 16;
constexpr int kPS = 32;      // reverse steps per partial tile
constexpr int kPStages = 2;
// Three warpgroups: 4 reverse warps, 4 recompute warps (one also loads), and
// the reducer warp with three idle ones.  The registers are rebalanced after
// launch: the reverse warps carry the most live state.
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;   // 65536 / 384, rounded down to the allocation unit of 8
constexpr int kReverseRegs = 240, kRecomputeRegs = kLaunchRegs, kReducerRegs = 96;
static_assert(kReverseRegs + kRecomputeRegs + kReducerRegs <= 3 * kLaunchRegs,
              "warpgroup register budgets exceed the launch's");
constexpr int kMaxChunk = 32;   // one chunk cache fills the 512 TMEM columns at 32 steps
constexpr int kTwoBufChunk = 16;  // up to 16 steps two caches fit: the recompute runs a chunk ahead
constexpr int kCBufs = 3;       // chunk input buffers: reverse, recompute, loading
constexpr int kSlotFloats = 4 * 16 + 4 * 16 + kV + 4 * 16;  // dq, dk row partials, dv, df row partials

struct MmaBwdParams {
  BwdArgs a;
  int R;
  int nchunks;
  int nptiles;
  int nbuf;  // TMEM cache buffers: 2 if ckpt_every <= kTwoBufChunk, else 1
  uint32_t htile_off, dtile_off, cbuf_off, cbuf_bytes, cq_off, ck_off, cv_off, cdy_off, cf_off;
  uint32_t hend_off, part_off, bar_off, misc_off;
  uint32_t tx_bytes;
};

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

  float* sPart = reinterpret_cast<float*>(smem + p.part_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* cfull = bars;
  uint64_t* tready = cfull + kCBufs;
  uint64_t* tfree = tready + 2;
  uint64_t* pfull = tfree + 2;
  uint64_t* ppeer = pfull + kPStages;
  uint64_t* pempty = ppeer + kPStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off);
  volatile int* vabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  volatile int* rabort = reinterpret_cast<volatile int*>(smem + p.misc_off + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off + 12);
  float* hend = reinterpret_cast<float*>(smem + p.hend_off);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCBufs; ++i) mbar_init(smem_u32(&cfull[i]), 32);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tready[i]), 4);
      mbar_init(smem_u32(&tfree[i]), 4);
    }
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(smem_u32(&pfull[i]), 1);
      mbar_init(smem_u32(&ppeer[i]), R);
      mbar_init(smem_u32(&pempty[i]), R);
    }
    *abort_flag = 0;
    *vabort = 0;
    *rabort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {  // the whole tensor memory: the per-thread chunk caches
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 8) {
    // Warps 0-3 walk the chunks backwards, warps 4-7 recompute them; warp w
    // and warp w + 4 share TMEM lanes 32(w % 4).. and the same fragment
    // positions, so thread i of the reverse warp reads exactly what thread i
    // of the recompute warp cached.
    const int w = warp & 3;
    const int g = lane >> 2, qd = lane & 3;
    const int ctid = threadIdx.x & 127;
    const int jcol0 = 16 * w + 2 * qd;           // this thread's columns: jcol0 + 8nt + {0,1}
    const int64_t row_g = static_cast<int64_t>(cta_rank) * kRows + g;
    const uint16_t* Wg = static_cast<const uint16_t*>(A.W) + static_cast<int64_t>(n) * kV * kV;
    // Cache buffer tb of this thread: TMEM lane 32w + lane, slot s = columns
    // 256 tb + 16 s .. + 15 holding {Z_s (8 values), H_{s-1} (8 values)}.
    const uint32_t tcache = tmem_base + (static_cast<uint32_t>(32 * w) << 16);
    const uint32_t htile0 = smem_u32(smem + p.htile_off);
    const uint32_t dtile0 = smem_u32(smem + p.dtile_off);

    if (warp >= 4) {
      // ======================= recompute warps (Eq. 10-11) =======================
      // Warp 4 also loads the chunk inputs, one chunk ahead of its own use:
      // q, k, v, dy by TMA, f gathered by the lanes (its global-load latency
      // hidden behind the chunk's recompute) and published at the chunk's end.
      const bool loader = (warp == 4);
      const uint16_t* fg = static_cast<const uint16_t*>(A.f);
      auto issue_chunk = [&](int li) -> float {
        const int t0 = (p.nchunks - 1 - li) * CL;
        uint8_t* buf = smem + p.cbuf_off + (li % kCBufs) * p.cbuf_bytes;
        const uint32_t fb = smem_u32(&cfull[li % kCBufs]);
        if (lane == 0) {
          mbar_expect_tx(fb, p.tx_bytes);
          tma_load_4d(smem_u32(buf + p.cq_off), &tm_q, fb, cta_rank * kRows, n, t0, b);
          tma_load_4d(smem_u32(buf + p.ck_off), &tm_k, fb, cta_rank * kRows, n, t0, b);
          tma_load_4d(smem_u32(buf + p.cv_off), &tm_v, fb, 0, n, t0, b);
          tma_load_4d(smem_u32(buf + p.cdy_off), &tm_dy, fb, 0, n, t0, b);
        }
        const int t = t0 + lane;
        return (lane < CL && t < T) ? bf16_bits_to_f32(fg[(static_cast<int64_t>(b) * T + t) * N + n]) : 0.f;
      };
      auto publish_chunk = [&](int li, float fv) {
        float* cfw = reinterpret_cast<float*>(smem + p.cbuf_off + (li % kCBufs) * p.cbuf_bytes + p.cf_off);
        if (lane < CL) cfw[lane] = fv;
        mbar_arrive(smem_u32(&cfull[li % kCBufs]));  // all 32 lanes: the phase's arrival count
      };
      if (loader) {
        if (lane == 0) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
          tma_prefetch_desc(&tm_v);
          tma_prefetch_desc(&tm_dy);
        }
        publish_chunk(0, issue_chunk(0));
      }
      // Forward transform fragments: B[k][col] = W[k][16w + col].
      uint32_t bw[2][4][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = 16 * w + 8 * nt + g;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const int k0 = 16 * kt + 2 * qd;
          bw[nt][kt][0] = static_cast<uint32_t>(Wg[k0 * kV + col]) |
                          (static_cast<uint32_t>(Wg[(k0 + 1) * kV + col]) << 16);
          bw[nt][kt][1] = static_cast<uint32_t>(Wg[(k0 + 8) * kV + col]) |
                          (static_cast<uint32_t>(Wg[(k0 + 9) * kV + col]) << 16);
        }
      }
      bool ok = true;
      int issued = 1;  // chunks whose loads have been issued
      for (int ci = 0; ci < p.nchunks; ++ci) {
        const int c = p.nchunks - 1 - ci;
        const int L = min(CL, T - c * CL);
        const int cb = ci % kCBufs, tb = ci % p.nbuf;
        bool mine = mbar_wait_timed(smem_u32(&cfull[cb]), (ci / kCBufs) & 1, status, kWhereBwdFull);
        // The cache buffer is free once the reverse warps have finished chunk
        // ci - nbuf; then the input buffer of chunk ci + 1 (last used by chunk
        // ci - 2) is free as well.
        if (mine && ci >= p.nbuf)
          mine = mbar_wait_timed(smem_u32(&tfree[tb]), ((ci / p.nbuf) - 1) & 1, status, kWhereBwdTFree);
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
        const float* cf = reinterpret_cast<const float*>(cbuf + p.cf_off);
        const uint32_t tbuf = tcache + 256 * tb;
        float h[2][4];
        if (c == 0) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) h[nt][0] = h[nt][1] = h[nt][2] = h[nt][3] = 0.f;
        } else {
          const float* src =
              A.ckpt + ((static_cast<int64_t>(chain) * A.n_ckpt + (c - 1)) * A.K + row_g) * kV + jcol0;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const float2 x0 = *reinterpret_cast<const float2*>(src + 8 * nt);
            const float2 x1 = *reinterpret_cast<const float2*>(src + 8 * kV + 8 * nt);
            h[nt][0] = x0.x; h[nt][1] = x0.y; h[nt][2] = x1.x; h[nt][3] = x1.y;
          }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int col = jcol0 + 8 * nt;
          st_shared_b32(htile0 + tile_off(g, col), pack2_bf16(h[nt][0], h[nt][1]));
          st_shared_b32(htile0 + tile_off(g + 8, col), pack2_bf16(h[nt][2], h[nt][3]));
        }
        named_bar_sync(2, 128);
        for (int s = 0; s < L; ++s) {
          const float k0 = bf16_bits_to_f32(ck[s * kRows + g]);
          const float k1 = bf16_bits_to_f32(ck[s * kRows + g + 8]);
          const float omf = 1.f - cf[s];
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(cv + s * kV + jcol0 + 8 * nt);
            const float v0 = bf16lo(vv), v1 = bf16hi(vv);
            acc[nt][0] = k0 * v0;
            acc[nt][1] = k0 * v1;
            acc[nt][2] = k1 * v0;
            acc[nt][3] = k1 * v1;
          }
          const uint32_t atile = htile0 + (s & 1) * 2048;
          uint32_t af[4][4];
#pragma unroll
          for (int kt = 0; kt < 4; ++kt) ldmatrix_x4(af[kt], ldsm_addr_a(atile, kt, lane));
#pragma unroll
          for (int kt = 0; kt < 4; ++kt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(acc[nt], af[kt], bw[nt][kt][0], bw[nt][kt][1]);
          const uint32_t otile = htile0 + ((s + 1) & 1) * 2048;
          uint32_t cache[16];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float z = tanh_fast(acc[nt][e]);
              cache[4 * nt + e] = __float_as_uint(z);
              cache[8 + 4 * nt + e] = __float_as_uint(h[nt][e]);  // H_{s-1}
              h[nt][e] = fmaf(omf, z - h[nt][e], h[nt][e]);
            }
            const int col = jcol0 + 8 * nt;
            st_shared_b32(otile + tile_off(g, col), pack2_bf16(h[nt][0], h[nt][1]));
            st_shared_b32(otile + tile_off(g + 8, col), pack2_bf16(h[nt][2], h[nt][3]));
          }
          tmem_st_32x32b_x16(tbuf + 16 * s, cache);
          named_bar_sync(2, 128);
        }
        tmem_st_wait();
        if (more) publish_chunk(ci + 1, fnext);
        // The chunk's final state, the reverse walk's first H_t.
        float4* he = reinterpret_cast<float4*>(hend + (tb * 128 + ctid) * 8);
        he[0] = make_float4(h[0][0], h[0][1], h[0][2], h[0][3]);
        he[1] = make_float4(h[1][0], h[1][1], h[1][2], h[1][3]);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tready[tb]));
        issued = ci + 2;
      }
      if (!ok) {
        *abort_flag = 1;
        // No TMA copy may still be writing when the CTA exits.
        if (loader)
          for (int li = max(0, issued - 2); li < min(issued, p.nchunks); ++li)
            mbar_wait_timed(smem_u32(&cfull[li % kCBufs]), (li / kCBufs) & 1, nullptr, kWhereBwdDrain);
      }
    } else {
      // ======================= reverse warps =======================
      warpgroup_reg_increase<kReverseRegs>();
      // Backward transform fragments: B[k = j][col = m] = W[16w + m][j] (D W^T).
      uint32_t bt[2][4][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int col = 16 * w + 8 * nt + g;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          const int k0 = 16 * kt + 2 * qd;
          bt[nt][kt][0] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + k0);
          bt[nt][kt][1] = *reinterpret_cast<const uint32_t*>(Wg + col * kV + k0 + 8);
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
      float dWacc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) dWacc[i][0] = dWacc[i][1] = dWacc[i][2] = dWacc[i][3] = 0.f;
      float dwr[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

      bool ok = true;
      int rs = 0;                  // reverse steps done so far (processing order)
      int pending_pfull = -1;      // partial tile whose last slot was written in the previous step
      for (int ci = 0; ci < p.nchunks && ok; ++ci) {
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
        const uint32_t tbuf = tcache + 256 * tb;
        // h = H_t for the chunk's last step; the next slot's TMEM load is
        // issued one step ahead and waited for at the top of the step.
        float h[2][4];
        {
          const float4* he = reinterpret_cast<const float4*>(hend + (tb * 128 + ctid) * 8);
          const float4 a0 = he[0], a1 = he[1];
          h[0][0] = a0.x; h[0][1] = a0.y; h[0][2] = a0.z; h[0][3] = a0.w;
          h[1][0] = a1.x; h[1][1] = a1.y; h[1][2] = a1.z; h[1][3] = a1.w;
        }
        uint32_t slot_regs[16];
        tmem_ld_32x32b<16>(tbuf + 16 * (L - 1), slot_regs);
        for (int s = L - 1; s >= 0; --s, ++rs) {
          const int ptile = rs / kPS, slot = rs % kPS, pst = ptile % kPStages;
          if (slot == 0) {
            // Partial tile ptile: wait until every CTA of the cluster has read
            // what this stage held two tiles ago.
            bool m2 = true;
            if (ptile >= kPStages)
              m2 = mbar_wait_timed<true>(smem_u32(&pempty[pst]), ((ptile / kPStages) - 1) & 1, status,
                                         kWhereBwdPeerEmpty);
            if (!m2) *vabort = 1;
            named_bar_sync(1, 128);
            if (*vabort) {
              ok = false;
              break;
            }
          }
          // Step inputs.
          const float q0 = bf16_bits_to_f32(cq[s * kRows + g]);
          const float q1 = bf16_bits_to_f32(cq[s * kRows + g + 8]);
          const float k0 = bf16_bits_to_f32(ck[s * kRows + g]);
          const float k1 = bf16_bits_to_f32(ck[s * kRows + g + 8]);
          const float ft = cf[s];
          const float omf = 1.f - ft;
          float u[2][2], vv[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const float2 uu = *reinterpret_cast<const float2*>(cdy + s * kV + jcol0 + 8 * nt);
            u[nt][0] = uu.x;
            u[nt][1] = uu.y;
            const uint32_t vb = *reinterpret_cast<const uint32_t*>(cv + s * kV + jcol0 + 8 * nt);
            vv[nt][0] = bf16lo(vb);
            vv[nt][1] = bf16hi(vb);
          }
          tmem_ld_wait();
          tmem_ld_fence_regs(slot_regs);
          float Z[2][4], Hp[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              Z[nt][e] = __uint_as_float(slot_regs[4 * nt + e]);
              Hp[nt][e] = __uint_as_float(slot_regs[8 + 4 * nt + e]);
            }
          if (s > 0) tmem_ld_32x32b<16>(tbuf + 16 * (s - 1), slot_regs);
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
          const uint32_t dt = dtile0 + (rs & 1) * 2048;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int col = jcol0 + 8 * nt;
            st_shared_b32(dt + tile_off(g, col), pack2_bf16(Dv[nt][0], Dv[nt][1]));
            st_shared_b32(dt + tile_off(g + 8, col), pack2_bf16(Dv[nt][2], Dv[nt][3]));
          }
          named_bar_sync(1, 128);
          if (pending_pfull >= 0 && threadIdx.x == 0) mbar_arrive(smem_u32(&pfull[pending_pfull % kPStages]));
          pending_pfull = -1;
          // Serial chain: C_{t-1} = f R + D W^T on the warp MMAs.
          float acc[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = ft * Rv[nt][e];
          uint32_t af[4][4];
#pragma unroll
          for (int kt = 0; kt < 4; ++kt) ldmatrix_x4(af[kt], ldsm_addr_a(dt, kt, lane));
#pragma unroll
          for (int kt = 0; kt < 4; ++kt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(acc[nt], af[kt], bt[nt][kt][0], bt[nt][kt][1]);
          // Off the chain: dW[16w.., :] += H_{t-1}^T D.
          {
            uint32_t ha[4];
            ha[0] = movmatrix_trans(pack2_bf16(Hp[0][0], Hp[0][1]));
            ha[1] = movmatrix_trans(pack2_bf16(Hp[1][0], Hp[1][1]));
            ha[2] = movmatrix_trans(pack2_bf16(Hp[0][2], Hp[0][3]));
            ha[3] = movmatrix_trans(pack2_bf16(Hp[1][2], Hp[1][3]));
#pragma unroll
            for (int nt2 = 0; nt2 < 4; ++nt2) {
              uint32_t bd[4];
              ldmatrix_x4_trans(bd, ldsm_addr_b_trans(dt, nt2, lane));
              mma_bf16_16816(dWacc[2 * nt2], ha, bd[0], bd[1]);
              mma_bf16_16816(dWacc[2 * nt2 + 1], ha, bd[2], bd[3]);
            }
          }
          // Off the chain: per-step partial reductions.
          float* part = sPart + (pst * kPS + slot) * kSlotFloats;
          {
            // Reductions on the tensor core (m16n8k16, fp32 accumulate), fp32
            // operands split into bf16 high + low parts (products of the parts
            // lose nothing that matters at fp32 accuracy):
            //   row sums     dq = H_t u, dk = D v, df rows = (R * (H_{t-1} - Z)) 1
            //                (A straight from the accumulator-layout registers,
            //                 B = the vector replicated over the 8 columns)
            //   column sums  dv = k^T D (A = k replicated over the rows,
            //                 B = D transposed with movmatrix)
            auto hl = [](float x0, float x1, uint32_t& hi, uint32_t& lo) {
              hi = pack2_bf16(x0, x1);
              lo = pack2_bf16(x0 - bf16lo(hi), x1 - bf16hi(hi));
            };
            uint32_t Ah[4], Al[4], Dh[4], Dl[4], Eh[4], El[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              float E[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) E[e] = Rv[nt][e] * (Hp[nt][e] - Z[nt][e]);
              hl(h[nt][0], h[nt][1], Ah[2 * nt], Al[2 * nt]);
              hl(h[nt][2], h[nt][3], Ah[2 * nt + 1], Al[2 * nt + 1]);
              hl(Dv[nt][0], Dv[nt][1], Dh[2 * nt], Dl[2 * nt]);
              hl(Dv[nt][2], Dv[nt][3], Dh[2 * nt + 1], Dl[2 * nt + 1]);
              hl(E[0], E[1], Eh[2 * nt], El[2 * nt]);
              hl(E[2], E[3], Eh[2 * nt + 1], El[2 * nt + 1]);
            }
            uint32_t uh0, ul0, uh1, ul1;
            hl(u[0][0], u[0][1], uh0, ul0);
            hl(u[1][0], u[1][1], uh1, ul1);
            const uint32_t vb0 = pack2_bf16(vv[0][0], vv[0][1]), vb1 = pack2_bf16(vv[1][0], vv[1][1]);  // exact
            const uint32_t one2 = 0x3F803F80u;  // bf16 pair (1, 1)
            float rq[4] = {0.f, 0.f, 0.f, 0.f}, rk[4] = {0.f, 0.f, 0.f, 0.f}, rf[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16_16816(rq, Ah, uh0, uh1);
            mma_bf16_16816(rq, Al, uh0, uh1);
            mma_bf16_16816(rq, Ah, ul0, ul1);
            mma_bf16_16816(rk, Dh, vb0, vb1);
            mma_bf16_16816(rk, Dl, vb0, vb1);
            mma_bf16_16816(rf, Eh, one2, one2);
            mma_bf16_16816(rf, El, one2, one2);
            uint32_t ka[4];
            ka[0] = ka[1] = *reinterpret_cast<const uint32_t*>(ck + s * kRows + 2 * qd);
            ka[2] = ka[3] = *reinterpret_cast<const uint32_t*>(ck + s * kRows + 2 * qd + 8);
            float rv[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              rv[nt][0] = rv[nt][1] = rv[nt][2] = rv[nt][3] = 0.f;
              mma_bf16_16816(rv[nt], ka, movmatrix_trans(Dh[2 * nt]), movmatrix_trans(Dh[2 * nt + 1]));
              mma_bf16_16816(rv[nt], ka, movmatrix_trans(Dl[2 * nt]), movmatrix_trans(Dl[2 * nt + 1]));
            }
            if (qd == 0) {  // column 0 of the row sums: rows g and g+8
              part[w * 16 + g] = rq[0];
              part[w * 16 + g + 8] = rq[2];
              part[64 + w * 16 + g] = rk[0];
              part[64 + w * 16 + g + 8] = rk[2];
              part[192 + w * 16 + g] = rf[0];
              part[192 + w * 16 + g + 8] = rf[2];
            }
            if (g == 0) {  // row 0 of the column sums
              *reinterpret_cast<float2*>(part + 128 + jcol0) = make_float2(rv[0][0], rv[0][1]);
              *reinterpret_cast<float2*>(part + 128 + jcol0 + 8) = make_float2(rv[1][0], rv[1][1]);
            }
            if (cta_rank == 0 && g == 0) {
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                dwr[nt][0] = fmaf(u[nt][0], vv[nt][0], dwr[nt][0]);
                dwr[nt][1] = fmaf(u[nt][1], vv[nt][1], dwr[nt][1]);
              }
            }
          }
          if (slot == kPS - 1 || rs == T - 1) pending_pfull = ptile;
          // C_{t-1}; H_{t-1} becomes the next step's H_t.
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              Cg[nt][e] = acc[nt][e];
              h[nt][e] = Hp[nt][e];
            }
        }
        if (!ok) break;
        // Every slot of this cache buffer has been read (the last load was
        // waited for at s = 0): the recompute may refill it.
        tc_fence_before_sync();
        __syncwarp();
        // This also frees the chunk's input buffer (the reverse warps read it last).
        if (lane == 0) mbar_arrive(smem_u32(&tfree[tb]));
      }
      if (ok) {
        named_bar_sync(1, 128);
        if (pending_pfull >= 0 && threadIdx.x == 0) mbar_arrive(smem_u32(&pfull[pending_pfull % kPStages]));
        // dW partial of this row block: rows m = 16w + g (+8), columns 8nt + 2qd (+1).
        float* dwp = A.dW_part + static_cast<int64_t>(blockIdx.x) * kV * kV;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int col = 8 * nt + 2 * qd;
          *reinterpret_cast<float2*>(dwp + (16 * w + g) * kV + col) = make_float2(dWacc[nt][0], dWacc[nt][1]);
          *reinterpret_cast<float2*>(dwp + (16 * w + g + 8) * kV + col) = make_float2(dWacc[nt][2], dWacc[nt][3]);
        }
        if (cta_rank == 0 && g == 0) {
          float* dst = A.dwr_part + static_cast<int64_t>(chain) * kV + jcol0;
          *reinterpret_cast<float2*>(dst) = make_float2(dwr[0][0], dwr[0][1]);
          *reinterpret_cast<float2*>(dst + 8) = make_float2(dwr[1][0], dwr[1][1]);
        }
      } else {
        *abort_flag = 1;
      }
    }
  } else {
    // The whole third warpgroup gives registers back at one instruction;
    // warps 9-11 then idle until the end.
    warpgroup_reg_decrease<kReducerRegs>();
  }
  if (warp == 8) {
    // ======================= reducer: partial tiles -> dq, dk, dv, df =======================
    const uint16_t* wr = static_cast<const uint16_t*>(A.w_r) + static_cast<int64_t>(n) * kV;
    const float wr0 = bf16_bits_to_f32(wr[2 * lane]), wr1 = bf16_bits_to_f32(wr[2 * lane + 1]);
    int done = 0;
    for (int ptile = 0; ptile < p.nptiles; ++ptile) {
      const int pst = ptile % kPStages;
      const uint32_t par = (ptile / kPStages) & 1;
      if (!mbar_wait(smem_u32(&pfull[pst]), par, abort_flag, status, kWhereBwdRec)) break;
      fence_acq_rel_cluster();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&ppeer[pst]), lane));
      if (!mbar_wait<true>(smem_u32(&ppeer[pst]), par, abort_flag, status, kWhereBwdPeer)) break;
      const int rs0 = ptile * kPS;
      const int nslots = min(kPS, T - rs0);
      const float* base = sPart + pst * kPS * kSlotFloats;
      // dq, dk: this CTA's 16 rows, summed over the four compute warps.
      for (int slot = 0; slot < nslots; ++slot) {
        const int t = T - 1 - (rs0 + slot);
        const int64_t rowt = (static_cast<int64_t>(b) * T + t) * N + n;
        const float* part = base + slot * kSlotFloats;
        const int i = lane & 15;
        const int off = (lane < 16) ? 0 : 64;
        const float sum = ((part[off + i] + part[off + 16 + i]) + part[off + 32 + i]) + part[off + 48 + i];
        float* dst = (lane < 16) ? A.dq : A.dk;
        dst[rowt * A.K + cta_rank * kRows + i] = sum;
      }
      // dv, df: summed over the cluster's row blocks, in fixed order.
      const uint32_t sbase = smem_u32(base);
      for (int slot = cta_rank; slot < nslots; slot += R) {
        const int t = T - 1 - (rs0 + slot);
        const int64_t rowt = (static_cast<int64_t>(b) * T + t) * N + n;
        float a0 = 0.f, a1 = 0.f, fsum = 0.f;
        for (int pr = 0; pr < R; ++pr) {  // fixed order over the chain's row blocks
          const uint32_t pb = mapa_shared(sbase, pr) + static_cast<uint32_t>(slot * kSlotFloats * 4);
          a0 += ld_shared_cluster_f32(pb + (128 + 2 * lane) * 4);
          a1 += ld_shared_cluster_f32(pb + (128 + 2 * lane + 1) * 4);
          fsum += ld_shared_cluster_f32(pb + (192 + 2 * lane) * 4) +
                  ld_shared_cluster_f32(pb + (192 + 2 * lane + 1) * 4);
        }
        const float2 uu = *reinterpret_cast<const float2*>(A.dy + rowt * kV + 2 * lane);
        *reinterpret_cast<float2*>(A.dv + rowt * kV + 2 * lane) = make_float2(fmaf(wr0, uu.x, a0), fmaf(wr1, uu.y, a1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) fsum += __shfl_xor_sync(0xffffffffu, fsum, o);  // fixed tree
        if (lane == 0) A.df[rowt] = fsum;
      }
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane < R) mbar_arrive_cluster(mapa_shared(smem_u32(&pempty[pst]), lane));
      done = ptile + 1;
    }
    for (int ptile = std::max(0, done - kPStages); ptile < done; ++ptile) {
      if (!mbar_wait<true>(smem_u32(&pempty[ptile % kPStages]), (ptile / kPStages) & 1, abort_flag, status,
                           kWhereBwdExit))
        break;
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

bool mma_backward_supported(int K, int V) { return V == kV && K % kRows == 0 && K >= kRows && K <= 128; }

size_t mma_backward_scratch_bytes(int, int, int, int, int) { return 0; }  // the cache is in TMEM

int mma_backward_max_chunk() { return kMaxChunk; }

cudaError_t launch_mma_backward(const BwdArgs& a, cudaStream_t stream) {
  if (a.ckpt_every > kMaxChunk) return cudaErrorInvalidValue;
  MmaBwdParams p{};
  p.a = a;
  p.R = a.K / kRows;
  const int C = a.ckpt_every;
  p.nchunks = (a.T + C - 1) / C;
  p.nptiles = (a.T + kPS - 1) / kPS;
  p.htile_off = 0;
  p.dtile_off = 4096;
  p.cbuf_off = 8192;
  p.cq_off = 0;
  p.ck_off = align_up(C * kRows * 2, 128);
  p.cv_off = p.ck_off + align_up(C * kRows * 2, 128);
  p.cdy_off = p.cv_off + align_up(C * kV * 2, 128);
  p.cf_off = p.cdy_off + align_up(C * kV * 4, 128);
  p.cbuf_bytes = align_up(p.cf_off + C * 4, 128);
  p.nbuf = (C <= kTwoBufChunk) ? 2 : 1;
  p.hend_off = p.cbuf_off + kCBufs * p.cbuf_bytes;
  p.part_off = p.hend_off + 2 * 128 * 8 * 4;
  p.bar_off = p.part_off + kPStages * kPS * kSlotFloats * 4;
  p.misc_off = p.bar_off + (kCBufs + 4 + 3 * kPStages) * 8;
  uint32_t smem = align_up(p.misc_off + 16, 128) + 1024;
  smem = std::max<uint32_t>(smem, 120 * 1024);
  p.tx_bytes = 2 * C * kRows * 2 + C * kV * 2 + C * kV * 4;

  CUtensorMap mq, mk, mv, mdy;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_tensor_map_btnx(&mq, a.q, bf, 2, a.B, a.T, a.N, a.K, kRows, C) ||
      !make_tensor_map_btnx(&mk, a.k, bf, 2, a.B, a.T, a.N, a.K, kRows, C) ||
      !make_tensor_map_btnx(&mv, a.v, bf, 2, a.B, a.T, a.N, kV, kV, C) ||
      !make_tensor_map_btnx(&mdy, a.dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.N, kV, kV, C))
    return cudaErrorInvalidValue;
  // The warpgroups' register budgets must fit in what the launch holds, or
  // the reverse warps' increase would wait forever: check the built kernel.
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, mma_backward_kernel);
  if (e != cudaSuccess) return e;
  if (kReverseRegs + kRecomputeRegs + kReducerRegs > 3 * fa.numRegs || fa.numRegs > kLaunchRegs)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(mma_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.B * a.N * p.R));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.R);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mma_backward_kernel, p, mq, mk, mv, mdy);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace m2rnn
