/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule library (libgdn.so).
 *
 * The operator is the gated delta rule of "Gated Delta Networks: Improving
 * Mamba2 with Delta Rule", §3.1 eq. 10:
 *
 *     S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T,
 *     o_t = S_t q_t,          S_t in R^{dv x dk},
 *
 * evaluated in the chunkwise WY/UT form of the same page, §3.3 (with the
 * decay mask Gamma in the intra-chunk output term, as derived on
 * "【论文解读】Gated Delta Network", §二(一)2(3)-(4)), and as a single-token
 * decode step (decay first, then correct the decayed prediction:
 * "Gated DeltaNet：先忘一点，再按误差更新记忆", "为什么再加一个遗忘门？").
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing, keeps no global state, never synchronises
 *     the device (except gdn_check_device_error) and enqueues all work on
 *     `stream` (a cudaStream_t; NULL means the legacy default stream).
 *   - Layouts are row-major and contiguous:
 *         q, k        [B, T, H, dk]     token-major, dtype `dt`
 *         v, out      [B, T, H, dv]     dtype `dt`
 *         g, beta     [B, T, H]         fp32; g = log(alpha) (<= 0 for a decay)
 *         states      [N, H, dv, dk]    fp32 (row j of S holds dk entries)
 *         cu_seqlens  [N + 1]           int32, device
 *   - Alignment: q, k, v, out and states 16 bytes (gdn_chunk_fwd); state
 *     16 bytes and q, k, v, out their element size (decode); g, beta
 *     and cu_seqlens 4 bytes; the workspace 256 bytes.
 *   - q is multiplied by `scale` after the optional per-token-head L2
 *     normalisation of q and k (use_qk_l2norm != 0: x / sqrt(sum x^2 + 1e-6)).
 *   - Gate values are device data and are not validated; any finite values
 *     are accepted (beta outside (0,1) included).
 *   - Host-side validation is synchronous and returns a status before any
 *     work is enqueued; a launch failure returns GDN_ERR_CUDA.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,     /* NULL/misaligned pointer, bad size or shape   */
    GDN_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. head dims)  */
    GDN_ERR_WORKSPACE = 3,       /* workspace missing or smaller than required  */
    GDN_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed        */
    GDN_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up waiting (see check below)  */
    GDN_ERR_RANGE = 6            /* a value left the range of an fp16 operand   */
} gdn_status;

typedef enum {
    GDN_F32 = 0,
    GDN_BF16 = 1
} gdn_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *gdn_status_string(gdn_status s);

/*
 * Bytes of device workspace gdn_chunk_fwd needs for this problem size.
 * num_seqs is the number of packed sequences when cu_seqlens is used, else 0.
 * Returns 0 for an invalid or unsupported size.
 */
size_t gdn_chunk_fwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                    int32_t num_seqs, gdn_dtype dt);

/*
 * Number of kernels one gdn_chunk_fwd call of this problem size enqueues on
 * its stream (same arguments as gdn_chunk_fwd_workspace_size): 2 on the
 * tensor-core path (bf16, dk = 128, dv a multiple of 128), 3 on the CUDA-core
 * path, 1 when there are no tokens.  Returns 0 for an invalid or unsupported
 * size.  Host-only; touches no device.
 */
int32_t gdn_chunk_fwd_kernel_count(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                   int32_t num_seqs, gdn_dtype dt);

/*
 * Chunked forward pass (prefill / training forward) of the gated delta rule.
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.3: per chunk
 * of C = chunk_size tokens the UT transform
 *     U~ = [I + strictLower(diag(beta)(Gamma o K K^T))]^{-1} diag(beta) V
 * (and the matching W<-), then the inter-chunk recurrence
 *     S_[t+1] = gamma^C S_[t] + (U~ - W<- S_[t]^T)^T K->,
 *     O_[t]   = Q<- S_[t]^T + (Q K^T o Gamma)(U~ - W<- S_[t]^T).
 *
 *   q, k, v       inputs (layouts above), dtype dt.
 *   g, beta       fp32 per token-head.
 *   init_state    [N, H, dv, dk] fp32 initial state per sequence, or NULL for
 *                 zeros ("state carry": pass a previous call's final_state).
 *   cu_seqlens    NULL: N = B sequences of T tokens each.  Non-NULL: packed
 *                 variable-length input, B must be 1, N = num_seqs, sequence n
 *                 is tokens [cu[n], cu[n+1]) of the T axis; cu[0] = 0,
 *                 cu[N] = T, non-decreasing (device data, not validated by
 *                 the host).  The state resets at every boundary to
 *                 init_state[n] (or 0).  Chunks never cross a boundary.
 *   out           [B, T, H, dv] dtype dt, written for every token.
 *   final_state   [N, H, dv, dk] fp32, or NULL to skip; may alias init_state.
 *   B, T, H       batch, tokens per row, heads (T >= 0, B, H >= 1).
 *   dk, dv        head dims: dk in {64, 128, 256}; dv a multiple of 32 up to 256
 *                 (others return GDN_ERR_UNSUPPORTED).  bf16 with dk = 128 and dv
 *                 a multiple of 128 runs on the tensor cores, every other size on
 *                 the CUDA cores.
 *   dt            GDN_F32 or GDN_BF16 (q, k, v and out); arithmetic is fp32.
 *   scale         multiplier of q (commonly 1/sqrt(dk)).
 *   chunk_size    must be 64.
 *   workspace     device scratch of at least gdn_chunk_fwd_workspace_size()
 *                 bytes, 256-byte aligned; its first 256 bytes hold the
 *                 device error word read by gdn_check_device_error.
 * Precision: arithmetic and accumulation are fp32.  On the tensor-core path
 * (bf16, dk = 128, dv a multiple of 128) the MMA operands are rounded: the
 * state copy, W<- and the raw q, k, v are bf16, T diag(beta) is a bf16 hi + lo
 * pair, and the three operands of the intra-chunk product
 * (U~ - W<- S^T) [Q K^T o Gamma | K->] are fp16, whose 11 significand bits
 * keep that product accurate where its terms nearly cancel (nearly parallel
 * keys with beta close to 2).  fp16 holds magnitudes up to 65504: a call in
 * which U~ - W<- S^T, Q K^T o Gamma or K-> exceeds that records
 * GDN_ERR_RANGE in the device error word (read by gdn_check_device_error).
 * Values below about 6e-5 in magnitude are carried with reduced relative
 * precision (fp16 subnormals), which is negligible against entries of
 * ordinary size in the same product.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE,
 *         GDN_ERR_CUDA.  Nothing is enqueued when an error is returned
 *         before the first launch.
 */
gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *g, const float *beta,
                         const float *init_state,
                         const int32_t *cu_seqlens, int32_t num_seqs,
                         void *out, float *final_state,
                         int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                         gdn_dtype dt, float scale, int32_t use_qk_l2norm, int32_t chunk_size,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Backward pass of gdn_chunk_fwd: the gradients of a loss L with respect to q,
 * k, v, g, beta and the initial state, given dL/dout and dL/dfinal_state.
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.3: the chunkwise
 * form is differentiated chunk by chunk -- a reverse scan over the chunks
 * carries the state gradient dS = gamma^C dS' + dO^T Q<- - dV_new^T W<- with
 * dV_new = K-> dS'^T + (Q K^T o Gamma)^T dO, and each chunk's inputs get their
 * gradients through the UT transform in parallel.  The forward states are
 * recomputed from the inputs (nothing from the forward call is needed).
 *   q, k, v, g, beta, init_state, cu_seqlens, B, T, H, dk, dv, dt, scale,
 *   use_qk_l2norm, chunk_size   as in gdn_chunk_fwd.
 *   dout          [B, T, H, dv] dtype dt: dL/dout.
 *   dfinal_state  [N, H, dv, dk] fp32: dL/dfinal_state, or NULL for zeros.
 *   dq, dk, dv    outputs [B, T, H, dk|dk|dv] dtype dt.
 *   dg, dbeta     outputs [B, T, H] fp32.
 *   dinit_state   output [N, H, dv, dk] fp32, or NULL to skip.
 *   workspace     at least gdn_chunk_bwd_workspace_size() bytes, 256-byte aligned
 *                 (fp32 intermediates, about 0.66 MB per chunk and head at
 *                 dk = dv = 128).
 * dk in {64, 128, 256}, dv as gdn_chunk_fwd.  fp32 inputs and other head sizes run
 * fp32 kernels on the CUDA cores (products on the tensor cores as three tf32 passes,
 * fp32-accurate).  For bf16 inputs with dk = 128 and dv a multiple of 128 the
 * chunk-start states and V_new come from the tensor-core chunked forward (its
 * precision, see gdn_chunk_fwd); with dk = dv = 128 every step runs on the tcgen05
 * tensor cores, fp32 intermediates entering each product as a bf16 (high, low) pair
 * (high.high + high.low + low.high in an fp32 accumulator, which keeps about 16
 * significand bits) and the raw bf16 inputs as exact operands.  Five launches then:
 * prep, the chunk-local and saving-recurrence pair of the forward scan, the reverse
 * scan and the local step.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA.
 */
size_t gdn_chunk_bwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                    int32_t num_seqs, gdn_dtype dt);

gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *g, const float *beta,
                         const float *init_state,
                         const int32_t *cu_seqlens, int32_t num_seqs,
                         const void *dout, const float *dfinal_state,
                         void *dq, void *dk_, void *dv_, float *dg, float *dbeta, float *dinit_state,
                         int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                         gdn_dtype dt, float scale, int32_t use_qk_l2norm, int32_t chunk_size,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step per (sequence, head), state updated in place.
 * "Gated DeltaNet：先忘一点，再按误差更新记忆", "为什么再加一个遗忘门？" and
 * "Decode 递归":  Sbar = alpha S;  S <- Sbar + beta (v - Sbar k) k^T;
 * o = S q (with the updated S).
 *   state   [N, H, dv, dk] fp32, read once and written once.
 *   q, k    [N, H, dk] dtype dt;  v, out [N, H, dv] dtype dt.
 *   g, beta [N, H] fp32.
 *   dk in {64, 128, 256}, dv a multiple of 8.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA.
 */
gdn_status gdn_decode_step(float *state,
                           const void *q, const void *k, const void *v,
                           const float *g, const float *beta,
                           void *out,
                           int32_t N, int32_t H, int32_t dk, int32_t dv, gdn_dtype dt,
                           float scale, int32_t use_qk_l2norm, void *stream);

/*
 * T successive decode tokens per (sequence, head) in one call (speculative or
 * multi-token decode), state updated in place.  "Gated DeltaNet：先忘一点，再按
 * 误差更新记忆", "Decode 递归": the steps compose in order, so the result is
 * exactly that of T gdn_decode_step calls on tokens 0..T-1 (and of
 * gdn_chunk_fwd over the same T tokens with init_state = state).  The state
 * is read once and written once per call, whatever T is.
 *   state   [N, H, dv, dk] fp32.
 *   q, k    [N, T, H, dk] dtype dt (token-major within each sequence);
 *   v, out  [N, T, H, dv] dtype dt;  g, beta [N, T, H] fp32.
 *   T >= 0 (T = 0 or N = 0: nothing is enqueued); other rules as gdn_decode_step.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA.
 */
gdn_status gdn_decode_multi(float *state,
                            const void *q, const void *k, const void *v,
                            const float *g, const float *beta,
                            void *out,
                            int32_t N, int32_t T, int32_t H, int32_t dk, int32_t dv, gdn_dtype dt,
                            float scale, int32_t use_qk_l2norm, void *stream);

/*
 * Reads and clears the device error word at the start of `workspace`
 * (synchronises `stream`).  Returns GDN_OK, GDN_ERR_DEVICE_TIMEOUT when a
 * kernel gave up on a bounded wait, GDN_ERR_RANGE when a tensor-core operand
 * left the fp16 range (see gdn_chunk_fwd), or GDN_ERR_CUDA.
 */
gdn_status gdn_check_device_error(void *workspace, void *stream);

/*
 * Self-test of the failure path (no counterpart on the pages).  Enqueues on
 * `stream` one kernel that waits, with the same bounded wait the tensor-core
 * kernels use for every mbarrier phase, on a phase that nothing completes.
 * After limit_us microseconds (1 .. 1e6) the wait gives up and the kernel
 * records the timeout in the device error word at the start of `workspace`
 * (256-byte aligned, at least 256 bytes; the word is cleared first), then
 * exits: nothing faults, and a following gdn_check_device_error on the same
 * workspace returns GDN_ERR_DEVICE_TIMEOUT (and clears the word).  Returns
 * GDN_OK once enqueued, GDN_ERR_INVALID_ARG for a bad pointer or limit,
 * GDN_ERR_CUDA if the launch fails.
 */
gdn_status gdn_selftest_wait_timeout(void *workspace, uint32_t limit_us, void *stream);

/*
 * Block prologue: q, k, v, g, beta from their linear projections, in one pass.
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.4 "Token mixing
 * block" and Fig. 1: q, k, v = SiLU(short causal depthwise convolution of the
 * projection); alpha from its projection in Mamba2's parameterisation, beta
 * from its projection through a sigmoid:
 *     y_t    = silu(sum_{j<K} w[h][c][j] x_{t-K+1+j})   (tap K-1: current token)
 *     g_t    = log alpha_t = -exp(A_log[h]) softplus(a_t + dt_bias[h])
 *     beta_t = 1 / (1 + exp(-b_t))
 * The outputs are the q, k, v, g, beta of gdn_chunk_fwd / gdn_decode_multi
 * (whose use_qk_l2norm applies the L2 normalisation of q and k).
 *   xq, xk        [B, T, H, dk] dtype dt;  xv [B, T, H, dv] dtype dt.
 *   wq, wk        [H, dk, K] fp32;  wv [H, dv, K] fp32 (one filter per channel).
 *   a, b          [B, T, H] fp32;  A_log, dt_bias [H] fp32.
 *   conv_state_in [N, K-1, H, 2 dk + dv] dtype dt: the K-1 inputs before each
 *                 sequence (oldest first; channels ordered q, k, v), or NULL
 *                 for zeros.  conv_state_out, same layout, receives the K-1
 *                 most recent inputs of each sequence (NULL to skip); it must
 *                 not overlap conv_state_in.
 *   cu_seqlens    as gdn_chunk_fwd (NULL: N = B sequences of T tokens).
 *   q, k, v       outputs [B, T, H, dk|dk|dv] dtype dt;  g, beta [B, T, H] fp32.
 *   K in 1..4; dk, dv multiples of 8 up to 256; x*, q, k, v and the states
 *   16-byte aligned, the fp32 arrays 4-byte aligned.
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA.
 */
gdn_status gdn_prologue(const void *xq, const void *xk, const void *xv,
                        const float *wq, const float *wk, const float *wv,
                        const float *a, const float *b, const float *A_log, const float *dt_bias,
                        const void *conv_state_in, void *conv_state_out,
                        const int32_t *cu_seqlens, int32_t num_seqs,
                        void *q, void *k, void *v, float *g, float *beta,
                        int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, int32_t K,
                        gdn_dtype dt, void *stream);

/*
 * Block prologue and chunked forward in one call: the output and final state
 * of gdn_chunk_fwd on the q, k, v, g, beta that gdn_prologue would make from
 * these projections, without q, k, v, g or beta ever being written to memory.
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.4 "Token mixing
 * block" and Fig. 1 (short convolution + SiLU, gate activations) feeding §3.3
 * (the chunkwise form).  The short convolution and SiLU run on each chunk's
 * q and k tiles inside the chunk-local kernel and on its v tile inside the
 * recurrence; the gates are activated as they are read.  The result is bit
 * for bit that of gdn_prologue followed by gdn_chunk_fwd (same roundings).
 *   xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, conv_state_in,
 *   conv_state_out, K           as gdn_prologue (conv_state_out receives the
 *                               K-1 most recent projection inputs of each
 *                               sequence; NULL to skip).
 *   init_state, cu_seqlens, num_seqs, out, final_state, B, T, H, scale,
 *   use_qk_l2norm, chunk_size   as gdn_chunk_fwd.
 *   dt            GDN_BF16 only; dk = 128, dv a multiple of 128 (the tensor-core
 *                 path); other sizes return GDN_ERR_UNSUPPORTED.
 *   workspace     at least gdn_prologue_chunk_fwd_workspace_size() bytes,
 *                 256-byte aligned (as gdn_chunk_fwd's, plus the convolved q
 *                 of each chunk, 16 KB per chunk and head).
 * Errors: GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA.
 */
size_t gdn_prologue_chunk_fwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                             int32_t num_seqs, gdn_dtype dt);

gdn_status gdn_prologue_chunk_fwd(const void *xq, const void *xk, const void *xv,
                                  const float *wq, const float *wk, const float *wv,
                                  const float *a, const float *b, const float *A_log, const float *dt_bias,
                                  const void *conv_state_in, void *conv_state_out,
                                  const float *init_state, const int32_t *cu_seqlens, int32_t num_seqs,
                                  void *out, float *final_state,
                                  int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, int32_t K,
                                  gdn_dtype dt, float scale, int32_t use_qk_l2norm, int32_t chunk_size,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * gdn_chunk_fwd_noalloc -- gdn_chunk_fwd for callers that cannot allocate.
 * The pages have no counterpart of this call: it exists for callers that may
 * not call cudaMalloc or any allocating routine where they run the operator
 * (plugin hosts and serving runtimes that plan all device memory up front,
 * bindings without a device allocator) and so cannot pass a workspace.
 *
 * Same arguments, semantics and errors as gdn_chunk_fwd, minus the
 * workspace.  The scratch is a fixed GDN_NOALLOC_SCRATCH_BYTES array inside
 * the library's device image: every GPU that loads the library holds it
 * until the process exits, and this call allocates and frees nothing.
 *   - The call runs the CUDA-core kernels, whose scratch need is 256 B plus
 *     64 * (12 + 4 * (dk + dv)) B per chunk slot and head, with B * ceil(T/64)
 *     slots (floor(T/64) + N + 1 for packed input).  A problem needing more
 *     than GDN_NOALLOC_SCRATCH_BYTES is rejected with GDN_ERR_WORKSPACE
 *     before any work is enqueued (for example B=1, H=8, T=2048, dk=dv=128
 *     needs 16.2 MiB and fits; H=16 needs 32.4 MiB and does not).
 *   - Every call looks up the array's device address (cudaGetSymbolAddress,
 *     with the call's device current), so the address stays valid across a
 *     device reset.  While `stream` is being captured the lookup is skipped and
 *     the address found by the last uncaptured call on that device is used:
 *     make at least one call on each device (and one after any cudaDeviceReset)
 *     before capturing.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents (the call clears what must start at zero).  Calls that
 *     overlap on the GPU race on it: order them (one stream, or events).
 *   - The device error word lives in the array, so gdn_check_device_error
 *     does not apply to this call.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)

gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *g, const float *beta,
                                 const float *init_state,
                                 const int32_t *cu_seqlens, int32_t num_seqs,
                                 void *out, float *final_state,
                                 int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                 gdn_dtype dt, float scale, int32_t use_qk_l2norm, int32_t chunk_size,
                                 void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
