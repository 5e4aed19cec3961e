/*
 * m2rnn.h -- C ABI of the GB300 M2RNN scan library (libm2rnn.so).
 *
 * The operation is the matrix-state non-linear recurrence of "M2RNN:
 * Non-Linear RNNs with Matrix-Valued States for Scalable Language Modeling"
 * (reading notes, section 2.1, the paper's Eq. 10-12), per batch element b
 * and head n, from H_0 = 0:
 *
 *     Z_t = tanh(H_{t-1} W + k_t v_t^T)          H, Z: K x V;  W: V x V
 *     H_t = f_t H_{t-1} + (1 - f_t) Z_t          f_t: scalar in [0, 1]
 *     y_t = H_t^T q_t + w_r (*) v_t              q_t, k_t: K;  v_t, w_r, y_t: V
 *
 * and its backward-through-time (notes section 2.7, the chain-rule
 * correction of the paper's Algorithm 2; see m2rnn_backward).
 *
 * Conventions shared by every entry point
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, dense and
 *    row-major in the layout given, 16-byte aligned.  The library allocates
 *    no memory; all scratch comes from the caller's workspace.
 *  - Layouts: q, k [B,T,N,K]; v [B,T,N,V]; f [B,T,N]; W [N,V,V] with
 *    W[n][m][j] the coefficient from state column m to column j (so
 *    (H W)_{ij} = sum_m H_{im} W_{mj}); w_r [N,V]; y, dy [B,T,N,V];
 *    H_T, dH_T [B,N,K,V]; checkpoints [B,N,n_ckpt,K,V] (see below).
 *  - q, k, v, f, W and w_r all have the element type `dtype`.  Every output,
 *    the upstream gradients and the state are float32.
 *  - Calls are asynchronous and ordered on `cuda_stream` (a cudaStream_t;
 *    NULL = legacy default stream).  The return value reports argument
 *    errors, unsupported shapes and launch/CUDA errors.  Errors that only the
 *    device can see (a bounded wait that gave up, a failed bounds check) are
 *    recorded in the workspace status block and reported by
 *    m2rnn_sync_status.
 *  - Supported shapes: B, T, N >= 1; K, V in [1, 128].  bf16 inputs with
 *    K a multiple of 16 (and at most 128) run on tensor-core kernels: V = 64
 *    with the forward on warp MMAs (tcgen05 on request) and the backward on
 *    warp MMAs (ckpt_every <= 20, its dW and its dk, dv on tensor cores),
 *    V = 16 on warp-MMA scans with the state in registers (the backward
 *    for ckpt_every <= 32, <= 16 with K > 64), V = 128: the forward (K in {32, 64, 128}) on tcgen05, the
 *    backward with K = 128 and ckpt_every <= 16 on tcgen05 (every product:
 *    the state-gradient chain, dW, dk, dv, dq), with other K or longer
 *    chunks on warp MMAs with its dW on tcgen05.  Every other supported
 *    shape runs on the fp32 CUDA-core kernels.  Nothing runs on the host
 *    CPU.
 *  - The tensor-core kernels take W re-encoded as fp16, and the warp-MMA
 *    forwards with readout warps (V = 64; V = 16 with K <= 64) read out y
 *    with q as an fp16 operand: with bf16 inputs, an entry with
 *    |W| >= 65520, or (those forwards, y requested) |q| >= 65536, is
 *    reported by m2rnn_sync_status as M2RNN_ERR_DEVICE with location 301
 *    (W) or 302 (q); the call's results are then not valid.
 */
#ifndef M2RNN_H_
#define M2RNN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  M2RNN_OK = 0,
  M2RNN_ERR_INVALID_ARG = -1, /* NULL/misaligned pointer, bad size or flag  */
  M2RNN_ERR_UNSUPPORTED = -2, /* shape/dtype outside the supported set      */
  M2RNN_ERR_WORKSPACE = -3,   /* workspace NULL or smaller than required    */
  M2RNN_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed          */
  M2RNN_ERR_TIMEOUT = -5,     /* device: a bounded wait gave up             */
  M2RNN_ERR_DEVICE = -6       /* device: an internal check failed           */
} m2rnn_status;

typedef enum { M2RNN_F32 = 0, M2RNN_BF16 = 1 } m2rnn_dtype;

/* Library version, as MAJOR*10000 + MINOR*100 + PATCH. */
int m2rnn_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* m2rnn_status_string(int status);

/* Number of stored checkpoints for T steps taken every `ckpt_every` steps:
 * (T - 1) / ckpt_every.  Checkpoint c (0-based) holds the fp32 state
 * H_{(c+1) * ckpt_every}, i.e. the state at the start of chunk c+1; chunk 0
 * starts from H_0 = 0, which is never stored.  Returns -1 on bad arguments. */
int64_t m2rnn_checkpoint_count(int64_t T, int ckpt_every);

/* Bytes of device workspace m2rnn_forward needs (at least the 256-byte
 * status block).  0 on bad arguments. */
size_t m2rnn_forward_workspace_size(int64_t B, int64_t T, int64_t N, int64_t K,
                                    int64_t V, m2rnn_dtype dtype);

/* Bytes of device workspace m2rnn_backward needs.  `have_ckpt` != 0 means the
 * caller will pass the forward's checkpoints; otherwise the workspace also
 * holds the checkpoints the backward recomputes.  0 on bad arguments. */
size_t m2rnn_backward_workspace_size(int64_t B, int64_t T, int64_t N, int64_t K,
                                     int64_t V, m2rnn_dtype dtype, int ckpt_every,
                                     int have_ckpt);

/*
 * Forward scan (Eq. 10-12 from H_0 = 0).
 *   in : q, k, v, f, W, w_r      (dtype, layouts above)
 *   out: y   [B,T,N,V] fp32      (required)
 *        H_T [B,N,K,V] fp32      (may be NULL)
 *        ckpt [B,N,n_ckpt,K,V] fp32, n_ckpt = m2rnn_checkpoint_count(T,
 *             ckpt_every)        (may be NULL; ckpt_every is ignored then)
 *   workspace: >= m2rnn_forward_workspace_size(...) bytes of device memory,
 *        16-byte aligned; its status block is cleared by this call.
 * Outputs are overwritten.  Inputs are not modified.  Concurrent calls that
 * share a workspace race on its status block.
 */
int m2rnn_forward(const void* q, const void* k, const void* v, const void* f,
                  const void* W, const void* w_r, float* y, float* H_T,
                  float* ckpt, int ckpt_every, int64_t B, int64_t T, int64_t N,
                  int64_t K, int64_t V, m2rnn_dtype dtype, void* workspace,
                  size_t workspace_bytes, void* cuda_stream);

/*
 * Backward through time: gradients of L = sum(dy * y) + <dH_T, H_T> with
 * respect to every input (notes section 2.7, with the value-residual terms
 * restored):  u_t = dy_t,  C_T = dH_T,
 *     R_t = C_t + q_t u_t^T
 *     D_t = ((1 - f_t) R_t) (*) (1 - Z_t (*) Z_t)
 *     C_{t-1} = f_t R_t + D_t W^T
 *     dq_t = H_t u_t        dk_t = D_t v_t        dv_t = D_t^T k_t + w_r (*) u_t
 *     df_t = <R_t, H_{t-1} - Z_t>_F
 *     dW[n] = sum_{b,t} H_{t-1}^T D_t      dw_r[n] = sum_{b,t} u_t (*) v_t
 *   in : q, k, v, f, W, w_r (dtype); dy [B,T,N,V] fp32 (required);
 *        dH_T [B,N,K,V] fp32 (may be NULL = zero);
 *        ckpt: the forward's checkpoints for the same ckpt_every (may be NULL:
 *        they are recomputed into the workspace).
 *   out: dq, dk [B,T,N,K]; dv [B,T,N,V]; df [B,T,N]; dW [N,V,V]; dw_r [N,V];
 *        all fp32, all required, overwritten (not accumulated).
 *   ckpt_every: chunk length of the recompute, 1 <= ckpt_every <= 4096.
 *   workspace: >= m2rnn_backward_workspace_size(...) bytes.
 * dW and dw_r are reduced over b in a fixed order: results are bitwise
 * reproducible run to run.
 */
int m2rnn_backward(const void* q, const void* k, const void* v, const void* f,
                   const void* W, const void* w_r, const float* dy,
                   const float* dH_T, const float* ckpt, int ckpt_every,
                   float* dq, float* dk, float* dv, float* df, float* dW,
                   float* dw_r, int64_t B, int64_t T, int64_t N, int64_t K,
                   int64_t V, m2rnn_dtype dtype, void* workspace,
                   size_t workspace_bytes, void* cuda_stream);

/*
 * Forward scan from a given initial state, optionally with one q/k shared by
 * every head: as m2rnn_forward, with
 *   H_0 [B,N,K,V] fp32 (may be NULL = zero): the state before step 1;
 *   qk_heads: N (q, k are [B,T,N,K], one per head) or 1 (q, k are
 *        [B,T,1,K], shared by all N value heads: the multi-value heads of
 *        the reading notes, section 2.4; each head keeps its own v, f, W,
 *        w_r and state).  Anything else is M2RNN_ERR_INVALID_ARG.
 * With H_T set to the final state of one call, the next call over the
 * following steps continues the same sequence (the fixed-size recurrent
 * state of the reading notes, section 2.6): a sequence can run in pieces.
 * H_0 may equal H_T (each state element is read before it is overwritten).
 *   z_stash (may be NULL): m2rnn_z_stash_size bytes that receive Z_t of
 *        every step (fp16, an internal layout) for m2rnn_backward_state;
 *        only for the shapes where that size is non-zero (else
 *        M2RNN_ERR_UNSUPPORTED).  The backward then skips the rerun of the
 *        recurrence's transform and tanh: it advances the state from each
 *        checkpoint by the gate blend alone.  Pass `ckpt` too.
 */
int m2rnn_forward_state(const void* q, const void* k, const void* v,
                        const void* f, const void* W, const void* w_r,
                        const float* H_0, float* y, float* H_T, float* ckpt,
                        int ckpt_every, void* z_stash, int64_t B, int64_t T,
                        int64_t N,
                        int64_t qk_heads, int64_t K, int64_t V,
                        m2rnn_dtype dtype, void* workspace,
                        size_t workspace_bytes, void* cuda_stream);

/* Bytes of the Z stash of m2rnn_forward_state / m2rnn_backward_state
 * (B T N K V fp16 values), or 0 where the stash is not supported (it is for
 * bf16 inputs with V = 64 or V = 16 and K a multiple of 16, <= 128). */
size_t m2rnn_z_stash_size(int64_t B, int64_t T, int64_t N, int64_t K,
                          int64_t V, m2rnn_dtype dtype);

/* Bytes of device workspace m2rnn_backward_state needs (a shared q/k,
 * qk_heads = 1 with N > 1, adds room for the per-head dq, dk). */
size_t m2rnn_backward_state_workspace_size(int64_t B, int64_t T, int64_t N,
                                           int64_t qk_heads, int64_t K,
                                           int64_t V, m2rnn_dtype dtype,
                                           int ckpt_every, int have_ckpt);

/*
 * Backward through time from a given initial state: as m2rnn_backward, with
 *   H_0  [B,N,K,V] fp32 (may be NULL = zero): the forward's initial state;
 *   dH_0 [B,N,K,V] fp32 (may be NULL): receives dL/dH_0, the state gradient
 *        carried one step past t = 1 (C_0 in the recursion above);
 *   state_grad_clip: c > 0 clamps every newly formed state gradient C_{t-1}
 *        elementwise to [-c, c] (per-step clipping of the recurrent state
 *        gradient in BPTT, notes section 2.3; the result is then no longer
 *        the exact gradient); 0 = off; negative or NaN is
 *        M2RNN_ERR_INVALID_ARG;
 *   qk_heads: as for m2rnn_forward_state.  With a shared q/k (1), dq and dk
 *        are [B,T,1,K]: the per-head gradients summed over the heads in a
 *        fixed order (notes section 2.7).
 * When a sequence runs in pieces, dH_0 of a later piece is the dH_T of the
 * piece before it.  `ckpt`, if given, must come from m2rnn_forward_state
 * with the same H_0.  z_stash (may be NULL): the stash that same forward
 * call wrote, with its `ckpt` (required when T > ckpt_every), ckpt_every
 * <= 20 (V = 64) or within the V = 16 backward's chunk limit (32, or 16 for
 * K > 64); Z_t then comes from the stash in fp16 instead of a rerun.
 * workspace: m2rnn_backward_state_workspace_size bytes.
 */
int m2rnn_backward_state(const void* q, const void* k, const void* v,
                         const void* f, const void* W, const void* w_r,
                         const float* H_0, const float* dy, const float* dH_T,
                         const float* ckpt, int ckpt_every,
                         const void* z_stash, float* dq,
                         float* dk, float* dv, float* df, float* dW,
                         float* dw_r, float* dH_0, float state_grad_clip,
                         int64_t B, int64_t T, int64_t N, int64_t qk_heads,
                         int64_t K, int64_t V, m2rnn_dtype dtype,
                         void* workspace, size_t workspace_bytes,
                         void* cuda_stream);

/*
 * Forward scan with the forget gate computed inside the scan kernels from its
 * pre-activation (reading notes, section 2.2; the paper's Eq. 13 and 17):
 *     f_t = (1 + exp(a_t + beta))^(-alpha) = exp(-alpha softplus(a_t + beta))
 * per head, in fp32.  As m2rnn_forward_state with f replaced by
 *   a     [B,T,N] in `dtype`: the gate pre-activation;
 *   alpha [N] fp32 (alpha >= 0 keeps f in (0, 1]), beta [N] fp32.
 * `ckpt` from this call serves m2rnn_backward_gated with the same a, alpha,
 * beta.  Workspace: m2rnn_forward_workspace_size bytes.
 */
int m2rnn_forward_gated(const void* q, const void* k, const void* v,
                        const void* a, const float* alpha, const float* beta,
                        const void* W, const void* w_r, const float* H_0,
                        float* y, float* H_T, float* ckpt, int ckpt_every,
                        void* z_stash, int64_t B, int64_t T, int64_t N,
                        int64_t qk_heads,
                        int64_t K, int64_t V, m2rnn_dtype dtype,
                        void* workspace, size_t workspace_bytes,
                        void* cuda_stream);

/*
 * Backward of m2rnn_forward_gated: as m2rnn_backward_state, with the gate
 * gradient taken through to its parameters.  With x = a + beta and
 * s = softplus(x):
 *   da     [B,T,N] fp32 = df f (-alpha) sigmoid(x);
 *   dalpha [N] fp32     = sum over b, t of df f (-s);
 *   dbeta  [N] fp32     = sum over b, t of da;
 * sums in a fixed order.  Workspace: m2rnn_backward_state_workspace_size
 * bytes.
 */
int m2rnn_backward_gated(const void* q, const void* k, const void* v,
                         const void* a, const float* alpha, const float* beta,
                         const void* W, const void* w_r, const float* H_0,
                         const float* dy, const float* dH_T, const float* ckpt,
                         int ckpt_every, const void* z_stash, float* dq,
                         float* dk, float* dv, float* da, float* dalpha, float* dbeta, float* dW,
                         float* dw_r, float* dH_0, float state_grad_clip,
                         int64_t B, int64_t T, int64_t N, int64_t qk_heads,
                         int64_t K, int64_t V, m2rnn_dtype dtype,
                         void* workspace, size_t workspace_bytes,
                         void* cuda_stream);

/*
 * Output path of the block (reading notes, section 2.3, step 4): the readout
 * y is multiplied by the output gate g first, then RMS-normalised over the
 * full width of a token, all heads together (d = N V; the statistic spans
 * every head, notes Appendix C), with a per-channel weight w:
 *     x = y (*) g,   s = (sum_j x_j^2 / d + eps)^(-1/2),   out = w (*) x s.
 *   y   [B,T,N,V] fp32 (the scan's output);  g [B,T,N,V] in `dtype`;
 *   w   [N,V] fp32;  eps >= 0 (the notes omit it; it sits inside the root);
 *   out [B,T,N,V] fp32;  rstd [B,T] fp32 (may be NULL): receives s.
 * N V <= 16384.  No workspace; the status block is not used.
 */
int m2rnn_output_norm(const float* y, const void* g, const float* w, float eps,
                      float* out, float* rstd, int64_t B, int64_t T,
                      int64_t N, int64_t V, m2rnn_dtype dtype,
                      void* cuda_stream);

/* Bytes of device workspace m2rnn_output_norm_backward needs (per-block
 * partial sums of dw), 0 for an unsupported shape. */
size_t m2rnn_output_norm_backward_workspace_size(int64_t B, int64_t T,
                                                 int64_t N, int64_t V);

/*
 * Backward of m2rnn_output_norm (notes Appendix C, with the epsilon kept):
 * with p = w (*) dout and r = sum_j p_j x_j per token,
 *     dx = s p - r s^3 x / d,   dy = dx (*) g,   dg = dx (*) y,
 *     dw = sum over b, t of dout (*) x s   (fixed order).
 * dout, dy, dg [B,T,N,V] fp32; dw [N,V] fp32; other arguments as for
 * m2rnn_output_norm.  dy feeds m2rnn_backward_state / _gated as its dy.
 */
int m2rnn_output_norm_backward(const float* y, const void* g, const float* w,
                               const float* dout, float eps, float* dy,
                               float* dg, float* dw, int64_t B, int64_t T,
                               int64_t N, int64_t V, m2rnn_dtype dtype,
                               void* workspace, size_t workspace_bytes,
                               void* cuda_stream);

/*
 * One decoding step for a batch of states (serving: one new token per
 * (b, head)): H [B,N,K,V] fp32 is updated in place to H_t from H_{t-1}, and
 * y [B,N,V] fp32 receives y_t.  q, k [B,qk_heads,K]; v [B,N,V]; f [B,N];
 * W, w_r as above; qk_heads as for m2rnn_forward_state.  bf16 with V = 64
 * and K a multiple of 16 (<= 128) runs a dedicated kernel, other shapes the
 * scan kernels with T = 1; the workspace is
 * m2rnn_forward_workspace_size(B, 1, N, K, V, dtype) bytes.
 */
int m2rnn_decode_step(float* H, const void* q, const void* k, const void* v,
                      const void* f, const void* W, const void* w_r, float* y,
                      int64_t B, int64_t N, int64_t qk_heads, int64_t K,
                      int64_t V, m2rnn_dtype dtype, void* workspace,
                      size_t workspace_bytes, void* cuda_stream);

/*
 * Synchronises `cuda_stream`, then reads and clears the workspace status
 * block that the last call on this workspace wrote.  Returns M2RNN_OK,
 * M2RNN_ERR_TIMEOUT or M2RNN_ERR_DEVICE; `detail` (may be NULL) receives an
 * implementation-defined location code of the first device error.
 */
int m2rnn_sync_status(void* workspace, void* cuda_stream, uint32_t* detail);

/*
 * Backward scan for callers that cannot allocate device memory: the same
 * gradients as m2rnn_backward, with every scratch buffer taken from an array
 * of 32 MiB built into the library's device image instead of a caller
 * workspace.  (No counterpart in the paper: this is a deployment variant.)
 *
 * Who needs it: code that must not or cannot call cudaMalloc -- e.g. a
 * plug-in inside a framework that owns all device memory, or a path where an
 * allocation would synchronise the device or fail.  Such a caller passes only
 * inputs and outputs.
 *
 * Limits: bf16 inputs, V = 64, K a multiple of 16 (<= 128), 1 <= ckpt_every
 * <= 20, and `ckpt` (the forward's checkpoints for this ckpt_every) is
 * required whenever T > ckpt_every.  A problem whose scratch would exceed the
 * built-in 32 MiB returns M2RNN_ERR_WORKSPACE; other shapes return
 * M2RNN_ERR_UNSUPPORTED.  Nothing is allocated, on the host or the device.
 *
 * The first call on a device looks the array's device address up (with that
 * device current); make that first call before any stream capture on the
 * device.  Every GPU that loads the library holds the array until exit.  All
 * calls share the array and it keeps the last call's contents (this call
 * clears what must start at zero): calls that overlap on the GPU race and
 * corrupt each other's results.
 *
 * sync != 0: synchronise `cuda_stream` and return the device-side status
 * (M2RNN_ERR_TIMEOUT / M2RNN_ERR_DEVICE) of this call; sync == 0: return
 * after queuing the work, and read the device-side status later with
 * m2rnn_backward_noalloc_status -- before the next call on the device, which
 * clears it.  The array's address is looked up again if the device's
 * context has been replaced since (e.g. after cudaDeviceReset).
 */
int m2rnn_backward_noalloc(const void* q, const void* k, const void* v,
                           const void* f, const void* W, const void* w_r,
                           const float* dy, const float* dH_T,
                           const float* ckpt, int ckpt_every, float* dq,
                           float* dk, float* dv, float* df, float* dW,
                           float* dw_r, int64_t B, int64_t T, int64_t N,
                           int64_t K, int64_t V, m2rnn_dtype dtype, int sync,
                           void* cuda_stream);

/*
 * Device-side status of the last m2rnn_backward_noalloc call on the current
 * device (the status block inside the built-in array): synchronises
 * `cuda_stream` (the stream that call used), then reads and clears the block.
 * Returns M2RNN_OK, M2RNN_ERR_TIMEOUT (a bounded wait gave up) or
 * M2RNN_ERR_DEVICE (a failed device-side check); `detail` (may be NULL)
 * receives the location code of the first device error.  Allocates nothing.
 */
int m2rnn_backward_noalloc_status(void* cuda_stream, uint32_t* detail);

/* Which forward kernel family a call with these arguments would run:
 * 2 = warp-MMA tensor-core kernels, 1 = tcgen05 tensor-core kernels,
 * 0 = fp32 CUDA-core kernels, negative = the status the call would return. */
int m2rnn_path(int64_t K, int64_t V, m2rnn_dtype dtype);

/*
 * Process-wide switches for tests and measurements (normal use needs
 * neither).  No counterpart in the paper.
 *   M2RNN_OPT_KERNEL_FAMILY: the kernel family every later call uses, as
 *     coded by m2rnn_path: -1 automatic (the default), 0 fp32 CUDA cores,
 *     1 tcgen05, 2 warp MMA.  A family that cannot run a call's shape falls
 *     back to the automatic choice for that call.
 *   M2RNN_OPT_TEST_STALL_TILE: failure-detection test hook.  n >= 0 makes the
 *     warp-MMA forward's input producer withhold input tile n of chains that
 *     run on one CTA (K = 16), so that the consumers' bounded waits expire
 *     and the status block reports M2RNN_ERR_TIMEOUT; -1 (the default) is off.
 * Initial values come from the environment variables M2RNN_KERNEL (auto |
 * tcgen05 | mma | simt) and M2RNN_TEST_STALL_TILE, read once, at the first
 * call that needs them; later changes of the environment have no effect.
 * `previous` (may be NULL) receives the old value.  Returns M2RNN_OK, or
 * M2RNN_ERR_INVALID_ARG for an unknown option or an out-of-range value.
 * Changing a switch while another host thread is inside a call is a race.
 */
enum { M2RNN_OPT_KERNEL_FAMILY = 0, M2RNN_OPT_TEST_STALL_TILE = 1 };
int m2rnn_set_option(int option, int value, int* previous);

#ifdef __cplusplus
}
#endif

#endif /* M2RNN_H_ */
