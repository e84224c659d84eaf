/*
 * moe.h - C ABI of libmoe, the B300 (sm_103a) Mixtral sparse mixture-of-experts
 * feed-forward layer.
 *
 * The layer (page "The Evolving Transformer - 05 Mixtral", section 05, the
 * formula y = sum_j w_j * E_{i_j}(x) and classes MoERouter / MoE):
 *   logits  l = x Wg^T                         (bias-free gate, d -> E)
 *   (i, w)  = top-k of l, softmax over those k  (= softmax over all E, top-k,
 *                                               renormalise over the k chosen)
 *   E_e(x)  = W2_e (silu(W1_e x) * (W3_e x))    (section 04, SwiGLU; W1 gate,
 *                                               W3 up, W2 down)
 *   out[t]  = sum_j w[t,j] E_{i[t,j]}(x[t])
 * Block form (section 06, Block; section 03, RMSNorm):
 *   out = x + MoE(RMSNorm(x)),  RMSNorm(x) = x (mean(x^2) + eps)^-1/2 gamma.
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller, unless a
 *    parameter says "host".  The library never frees or keeps them.
 *  - Row-major layouts; every operand is contiguous along its last index:
 *      x[T,d], Wg[E,d], W1[E,dff,d], W3[E,dff,d], W2[E,d,dff], out[T,d].
 *    Device pointers must be 16-byte aligned (256-byte for the tensor-core
 *    path's x_perm / h_perm / W1 / W3 / W2).
 *  - dtype is MOE_DTYPE_BF16 (bf16 storage, fp32 accumulate) or
 *    MOE_DTYPE_F32 (fp32 storage and arithmetic, no TF32).
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) of the device that owns the output pointer.  No entry point
 *    synchronises the host unless it says so.
 *  - Return value: MOE_OK (0) or a negative MOE_E* code.  Arguments are
 *    validated on the host before anything is enqueued; a failed check
 *    enqueues nothing.  Nothing aborts the process.
 *  - Device-side failures (an out-of-range expert index, a bounded wait that
 *    ran out) do not trap: the kernel records a MOE_E* code in a per-device
 *    status word and returns.  Read it with moe_get_device_status().
 *  - T = 0 is a valid no-op.
 *
 * Supported shapes: 1 <= k <= min(E, 8), 1 <= E <= 64, d % 8 == 0 (f32:
 * d % 4 == 0).  The bf16 expert path (tcgen05 tensor cores) also needs
 * d % 64 == 0 and dff % 64 == 0.  Anything else returns MOE_EUNSUPPORTED.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* The same type as cudaStream_t; pass a cudaStream_t (or NULL) directly. */
typedef struct CUstream_st* moe_stream_t;

enum moe_status {
  MOE_OK = 0,
  MOE_EINVAL = -1,       /* null pointer, negative size, misaligned pointer   */
  MOE_EUNSUPPORTED = -2, /* valid arguments outside the supported shapes      */
  MOE_ECUDA = -3,        /* a CUDA runtime/driver call failed                 */
  MOE_ETIMEOUT = -4,     /* a device-side bounded wait ran out (device status)*/
  MOE_ENOMEM = -5,       /* workspace too small, or allocation failed         */
  MOE_EDEVICE = -6       /* device-side bounds check failed (device status)   */
};

enum moe_dtype { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };

/* Short text for a status code (static storage). */
const char* moe_status_string(int status);

/* ABI version (major * 100 + minor). */
int moe_version(void);

/*
 * Steps a1 + a2 - router (section 05, MoERouter): fp32 gate logits
 * l[t,e] = sum_c x[t,c] Wg[e,c], then the k largest logits in descending
 * order (equal logits: lower expert index first), then their softmax.
 *   x[T,d], Wg[E,d]          in: dtype
 *   topk_idx[T,k] int32      out: chosen experts, slot 0 = largest logit
 *   topk_w[T,k]   fp32       out: gate weights, sum to 1 per token
 *   logits_opt[T,E] fp32     out, optional (NULL to skip)
 */
int moe_router_topk(const void* x, const void* Wg, int T, int d, int E, int k,
                    int32_t* topk_idx, float* topk_w, float* logits_opt,
                    int dtype, moe_stream_t stream);

/*
 * Step a0 - RMSNorm (section 03): xn = x (mean(x^2) + eps)^-1/2 gamma,
 * computed in fp32 and rounded once to dtype.  x[T,d], gamma[d], xn[T,d].
 */
int moe_rmsnorm(const void* x, const void* gamma, float eps, void* xn,
                int T, int d, int dtype, moe_stream_t stream);

/*
 * Step a3 - dispatch (section 05, class MoE groups tokens per expert; the
 * page notes production stacks batch tokens per expert).  With Tk = T*k and
 * the flat pair index f = t*k + j:
 *   counts[E]      out: n_e = #{f : topk_idx[f] == e}
 *   offsets[E+1]   out: exclusive prefix sum of counts, offsets[E] = Tk
 *   slot_pos[Tk]   out: row of pair f in expert-contiguous order; stable:
 *                  within an expert, rows follow ascending f
 *   row_src[Tk]    out: row_src[slot_pos[f]] = f / k (source token)
 *   x_perm[Tk,d]   out: x_perm[p] = x[row_src[p]]
 * An index outside [0,E) is skipped and sets MOE_EDEVICE in the device
 * status; the outputs are then incomplete.
 */
int moe_permute(const void* x, const int32_t* topk_idx, int T, int d, int E, int k,
                int32_t* counts, int32_t* offsets, int32_t* row_src, int32_t* slot_pos,
                void* x_perm, int dtype, moe_stream_t stream);

/*
 * The row copy of step a3 on its own, for moving routed rows between
 * orders (the expert-parallel layer regroups the rows it received per
 * expert with it): dst[i] = src[row_idx[i]] for i < n_rows, rows of
 * row_bytes bytes (a multiple of 16; src and dst 16-byte aligned),
 * row_idx[n_rows] int32 (device).  An index outside [0, src_rows) is skipped
 * (its row of dst is left as it was) and sets MOE_EDEVICE in the device
 * status.
 */
int moe_gather_rows(const void* src, int src_rows, const int32_t* row_idx, int n_rows, void* dst,
                    size_t row_bytes, moe_stream_t stream);

/*
 * Step a4 - grouped gate/up GEMM with the SwiGLU fused into its epilogue
 * (section 04): for expert e and every row p in [offsets[e], offsets[e+1]),
 *   h_perm[p, f] = silu(sum_c x_perm[p,c] W1[e,f,c]) * sum_c x_perm[p,c] W3[e,f,c]
 * x_perm[Tk,d] in, h_perm[Tk,dff] out, offsets[E+1] in (device).
 * bf16: fp32 accumulation in tensor memory, h rounded once to bf16.
 */
int moe_expert_gate_up(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3,
                       void* h_perm, int Tk, int d, int dff, int E, int dtype, moe_stream_t stream);

/*
 * Step a5 - grouped down-projection GEMM (section 04):
 *   y_perm[p, c] = sum_f h_perm[p,f] W2[e,c,f]   for p in expert e's rows.
 * h_perm[Tk,dff] in, y_perm[Tk,d] out (dtype).
 */
int moe_expert_down(const void* h_perm, const int32_t* offsets, const void* W2,
                    void* y_perm, int Tk, int d, int dff, int E, int dtype, moe_stream_t stream);

/*
 * Steps a4 + a5 in one call (section 04: each expert's whole SwiGLU):
 *   y_perm[p] = W2_e (silu(W1_e x_perm[p]) * (W3_e x_perm[p]))  for p in expert e's rows.
 * x_perm[Tk,d] in, y_perm[Tk,d] out (dtype), offsets[E+1] in (device).  The
 * hidden activations h[Tk,dff] live in scratch taken from cudaMallocAsync
 * on `stream` (the device's stream-ordered pool) and released on the same
 * stream; MOE_ENOMEM if that allocation fails.
 */
int moe_expert_ffn(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3,
                   const void* W2, void* y_perm, int Tk, int d, int dff, int E, int dtype,
                   moe_stream_t stream);

/*
 * As moe_expert_ffn on caller scratch: h_perm[Tk,dff] (dtype, 16-byte
 * aligned) receives the hidden activations silu(W1_e x) * (W3_e x).
 */
int moe_expert_ffn_ws(const void* x_perm, const int32_t* offsets, const void* W1, const void* W3,
                      const void* W2, void* h_perm, void* y_perm, int Tk, int d, int dff, int E,
                      int dtype, moe_stream_t stream);

/*
 * Step a6 - combine fused with the un-permute (section 05, class MoE adds the
 * chosen experts' outputs with their weights; section 06 adds the residual):
 *   out[t,c] = sum_j topk_w[t,j] y_perm[slot_pos[t*k+j], c]  (+ residual[t,c])
 * summed in fp32, rounded once to dtype.  residual_opt may be NULL.
 */
int moe_combine(const void* y_perm, const int32_t* slot_pos, const float* topk_w,
                const void* residual_opt, void* out, int T, int d, int k, int dtype,
                moe_stream_t stream);

/*
 * Bytes of scratch moe_forward_ws, moe_block_forward_ws and moe_forward_ex
 * (bf16 or fp32 experts) need for T tokens; 0 for invalid sizes.
 */
size_t moe_workspace_bytes(int T, int d, int dff, int E, int k, int dtype);

/*
 * Byte offsets of the layer's intermediates inside that scratch (host
 * call, no device work): offs[0..9] = topk_idx [T,k] int32, topk_w [T,k]
 * fp32, counts [E] int32, offsets [E+1] int32, row_src [T*k] int32,
 * slot_pos [T*k] int32, x_perm [T*k,d], h_perm [T*k,dff], y_perm [T*k,d],
 * xn [T,d] (block form); offs[10] = total bytes.  After a forward call these
 * hold that call's values (the backward reads them as `saved`).
 */
int moe_forward_workspace_offsets(int T, int d, int dff, int E, int k, int dtype, size_t* offs);

/*
 * The whole layer, a1..a6, on caller-provided scratch `workspace` of at least
 * moe_workspace_bytes() bytes (256-byte aligned).  dtype selects the
 * bf16 tensor-core path or the fp32 path.
 */
int moe_forward_ws(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                   void* out, int T, int d, int dff, int E, int k, int dtype,
                   void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * The whole layer in bf16, one call.  Scratch comes from cudaMallocAsync on
 * `stream` (the device's stream-ordered pool) and is released on the same
 * stream.
 */
int moe_forward(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                void* out, int T, int d, int dff, int E, int k, moe_stream_t stream);

/* As moe_forward, fp32 storage and arithmetic (CUDA-core path). */
int moe_forward_f32(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                    void* out, int T, int d, int dff, int E, int k, moe_stream_t stream);

/*
 * Block form, a0..a6 (section 06, Block, MoE half): out = x + MoE(RMSNorm(x)).
 * gamma[d]; the normalised activation is rounded once to dtype before the
 * router and the experts.  _ws takes caller scratch as moe_forward_ws.
 */
int moe_block_forward_ws(const void* x, const void* gamma, float eps, const void* Wg,
                         const void* W1, const void* W3, const void* W2, void* out,
                         int T, int d, int dff, int E, int k, int dtype,
                         void* workspace, size_t workspace_bytes, moe_stream_t stream);
int moe_block_forward(const void* x, const void* gamma, float eps, const void* Wg,
                      const void* W1, const void* W3, const void* W2, void* out,
                      int T, int d, int dff, int E, int k, moe_stream_t stream);

/*
 * The layer with every option, on caller scratch, recording caller-created
 * CUDA events at its step boundaries (for timing the steps of one call):
 *  - gamma_opt != NULL selects the block form (as moe_block_forward_ws);
 *  - W1q != NULL selects int8 expert weights (W1q..W2s as moe_forward_w8_ws;
 *    W1, W3, W2 are then ignored; bf16 only);
 *  - events (NULL, or 5 cudaEvent_t; NULL entries skipped) are recorded on
 *    `stream` before the router, after dispatch, after the gate/up GEMM,
 *    after the down GEMM and after the combine.
 * workspace as moe_forward_ws (moe_workspace_bytes()).  Same results as the
 * corresponding entry point.
 */
int moe_forward_ex(const void* x, const void* gamma_opt, float eps, const void* Wg, const void* W1,
                   const void* W3, const void* W2, const int8_t* W1q, const float* W1s, const int8_t* W3q,
                   const float* W3s, const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff,
                   int E, int k, int dtype, void* workspace, size_t workspace_bytes, void* const* events,
                   moe_stream_t stream);

/*
 * End-to-end call with HOST activations: copies x_host[T,d] (pinned host
 * memory for best speed) to the device, runs moe_forward_ws, and copies the
 * result back to out_host[T,d].  Weights stay resident on the device.
 * `workspace` must hold moe_workspace_bytes() + 2*T*d*elem bytes.
 * Synchronises `stream` before returning, so out_host is ready on return.
 */
size_t moe_forward_host_workspace_bytes(int T, int d, int dff, int E, int k, int dtype);
int moe_forward_host(const void* x_host, const void* Wg, const void* W1, const void* W3,
                     const void* W2, void* out_host, int T, int d, int dff, int E, int k,
                     int dtype, void* workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * ---- int8 weight-only expert weights ------------------------------------
 * KerasFormers Mixtral docs, "Lower memory": the weights alone may be
 * quantised to int8 while activations stay bf16.  The docs do not give the
 * scheme; this library uses symmetric per-output-channel codes: each row of
 * an nn.Linear weight W[rows, cols] (W1/W3: rows = E*dff, cols = d; W2:
 * rows = E*d, cols = dff) gets one fp32 scale s = max|row| / 127 and codes
 * q = round-half-even(w / s) clamped to [-127, 127] (both divisions IEEE
 * fp32, so the codes are reproducible bit for bit); a zero row has s = 0 and
 * q = 0.  The layer then uses s[row] * q[row, col] in place of W.  The expert
 * weights take half the bytes of bf16 (plus 4 bytes per row), which is what
 * bounds the layer at small batches.  The router's Wg stays bf16.
 */

/*
 * Quantise a bf16 matrix W[rows, cols] (device) to q[rows, cols] int8 and
 * scale[rows] fp32 (device, caller-owned).  cols % 8 == 0; W and q 16-byte
 * aligned.  Inputs are expected finite.
 */
int moe_quantize_int8(const void* W, int rows, int cols, int8_t* q, float* scale, moe_stream_t stream);

/*
 * Step a4 with int8 weights: as moe_expert_gate_up (bf16 x_perm and h_perm),
 * with W1q/W3q [E,dff,d] int8 and W1s/W3s [E*dff] fp32 row scales:
 *   h_perm[p,f] = silu(W1s[e,f] * sum_c x_perm[p,c] W1q[e,f,c])
 *                 * (W3s[e,f] * sum_c x_perm[p,c] W3q[e,f,c])
 * fp32 accumulation, h rounded once to bf16.  All pointers 16-byte aligned.
 */
int moe_expert_gate_up_w8(const void* x_perm, const int32_t* offsets, const int8_t* W1q, const float* W1s,
                          const int8_t* W3q, const float* W3s, void* h_perm, int Tk, int d, int dff, int E,
                          moe_stream_t stream);

/*
 * Step a5 with int8 weights: y_perm[p,c] = W2s[e,c] * sum_f h_perm[p,f] W2q[e,c,f],
 * W2q [E,d,dff] int8, W2s [E*d] fp32; bf16 h_perm / y_perm.
 */
int moe_expert_down_w8(const void* h_perm, const int32_t* offsets, const int8_t* W2q, const float* W2s,
                       void* y_perm, int Tk, int d, int dff, int E, moe_stream_t stream);

/*
 * The whole bf16 layer with int8 expert weights (a1..a6).  x[T,d], Wg[E,d],
 * out[T,d] bf16; the six weight arguments as above.  _ws takes caller scratch
 * (256-byte aligned) of at least moe_workspace_bytes(T, d, dff, E, k,
 * MOE_DTYPE_BF16) bytes; the other takes it from cudaMallocAsync on `stream`.
 *
 * The codes are widened to bf16 on the SM (exactly: every code is a bf16
 * value) straight into the tensor cores' operand memory, and the per-row
 * scales are applied to the fp32 accumulators; no bf16 copy of the weights
 * is made, so moe_forward_w8_workspace_bytes() equals moe_workspace_bytes()
 * of the bf16 layer.
 */
size_t moe_forward_w8_workspace_bytes(int T, int d, int dff, int E, int k);
int moe_forward_w8_ws(const void* x, const void* Wg, const int8_t* W1q, const float* W1s, const int8_t* W3q,
                      const float* W3s, const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff,
                      int E, int k, void* workspace, size_t workspace_bytes, moe_stream_t stream);
int moe_forward_w8(const void* x, const void* Wg, const int8_t* W1q, const float* W1s, const int8_t* W3q,
                   const float* W3s, const int8_t* W2q, const float* W2s, void* out, int T, int d, int dff, int E,
                   int k, moe_stream_t stream);

/*
 * ---- backward (training) ------------------------------------------------
 * Mixtral 8x7B model reference page, Training: the experts and the router are
 * trained together.  For L = sum(out * dout), out = the bf16 layer, these
 * calls compute dL/dx, dL/dWg, dL/dW1, dL/dW3, dL/dW2.  The top-k choice is
 * piecewise constant, so the router receives its gradient through the softmax
 * over the k chosen logits only:
 *   dy_j = w_j dout,  dw_j = <dout, y_j>,  dl_j = w_j (dw_j - sum_i w_i dw_i)
 *   dh = dy W2_e,  da = dh * b * silu'(a),  db = dh * silu(a)  (a = x W1_e^T, b = x W3_e^T)
 *   dx = sum_j (da W1_e + db W3_e) + sum_j dl_j Wg[i_j]
 *   dW2_e = sum dy^T h,  dW1_e = sum da^T x,  dW3_e = sum db^T x,  dWg[i_j] += dl_j x
 * Inputs: dout[T,d] bf16 and the forward's inputs.  `saved` is the scratch
 * that moe_forward_ws(x, Wg, W1, W3, W2, out, ..., MOE_DTYPE_BF16, saved,
 * saved_bytes, ...) or moe_forward_train_ws filled for the same inputs,
 * unmodified since (it holds the routing, the permutation, x_perm, h and
 * y_perm).  `keep` is NULL, or the buffer that moe_forward_train_ws filled
 * in that same call: then da = dh p and db = dh q come from the kept p and q
 * instead of a and b recomputed (one GEMM of 4*T*k*d*dff flop less).
 * Outputs (overwritten):
 * dx[T,d] bf16; dWg[E,d], dW1[E,dff,d], dW3[E,dff,d], dW2[E,d,dff] fp32 (an
 * expert no token chose gets zeros).  dh is formed in fp32 from the exact
 * dout rows and the fp32 gate weight; the intermediates da, db, the permuted
 * dx and (for dW2 only) dy are bf16; every GEMM accumulates in fp32 on the
 * tensor cores.  Recomputed, a and b are fp32; kept, p and q are formed in
 * fp32 from the forward's fp32 a and b and rounded once to bf16, which
 * perturbs da and db by one bf16 rounding relative to themselves (keeping a
 * itself in bf16 would not: silu'(a) crosses zero near a = -1.28).
 * Shapes as the bf16 forward.  The block form is not differentiated here.
 */
/*
 * The training forward: moe_forward_ws in bf16 (same `out`, same scratch
 * contents) that also keeps, for moe_backward_ws, the local derivatives of
 * the SwiGLU h = silu(a) b at the gate/up GEMM's a = x W1_e^T, b = x W3_e^T:
 * p = b silu'(a) and q = silu(a), formed in fp32 and rounded to bf16, in
 * keep[2][T*k][dff] (device, caller-owned, 16-byte aligned; plane 0 = p,
 * plane 1 = q, rows in the permuted order of the scratch's x_perm):
 * 4*T*k*dff bytes.  Errors as moe_forward_ws; keep == NULL is MOE_EINVAL.
 */
int moe_forward_train_ws(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                         void* out, void* keep, int T, int d, int dff, int E, int k, void* workspace,
                         size_t workspace_bytes, moe_stream_t stream);
size_t moe_backward_workspace_bytes(int T, int d, int dff, int E, int k);
int moe_backward_ws(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3,
                    const void* W2, const void* saved, size_t saved_bytes, const void* keep, void* dx,
                    float* dWg, float* dW1, float* dW3, float* dW2, int T, int d, int dff, int E, int k,
                    void* workspace, size_t workspace_bytes, moe_stream_t stream);
/* As moe_backward_ws, scratch from cudaMallocAsync on `stream`. */
int moe_backward(const void* dout, const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                 const void* saved, size_t saved_bytes, const void* keep, void* dx, float* dWg, float* dW1,
                 float* dW3, float* dW2, int T, int d, int dff, int E, int k, moe_stream_t stream);

/*
 * Scratch size built into moe_forward_noalloc (16 MiB per GPU).
 */
#define MOE_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * The whole bf16 layer, as moe_forward, for callers that must not allocate
 * device memory while they run: for example an application whose memory
 * manager owns the device budget and forbids allocation after start-up, or a
 * latency-critical loop where an allocation could synchronise the device.
 * The pages have no counterpart; this is a deployment variant of moe_forward.
 *  - Scratch is a 16 MiB (MOE_NOALLOC_SCRATCH_BYTES) array inside the
 *    library's device image: every GPU that loads the library holds it until
 *    the process exits.  Nothing is allocated per call (no cudaMalloc,
 *    cudaMallocAsync or cudaFree).
 *  - A layer that needs more scratch than that, i.e.
 *    moe_workspace_bytes(T, d, dff, E, k, MOE_DTYPE_BF16) >
 *    MOE_NOALLOC_SCRATCH_BYTES (at d=4096, d_ff=14336, k=2: T > 170), is
 *    rejected with MOE_ENOMEM before anything is enqueued.
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *  - All calls share the one array, and it keeps the last call's contents.
 *    Nothing in it needs to start at zero, but calls that overlap on the GPU
 *    (other streams, other host threads) race on it: serialise them.
 */
int moe_forward_noalloc(const void* x, const void* Wg, const void* W1, const void* W3, const void* W2,
                        void* out, int T, int d, int dff, int E, int k, moe_stream_t stream);

/*
 * Device status word of the device that owns `stream`: synchronises the
 * stream, writes the first MOE_E* code a kernel recorded since the last reset
 * (MOE_OK if none) to *status, and clears it when reset != 0.
 */
int moe_get_device_status(moe_stream_t stream, int* status, int reset);

/*
 * Limit, in nanoseconds, for every device-side spin wait launched after this
 * call (default 2e9).  A wait that runs out records MOE_ETIMEOUT and the
 * kernel returns early.  ns <= 0 restores the default.  Host-side setting,
 * process-wide.
 */
int moe_set_wait_limit_ns(long long ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
