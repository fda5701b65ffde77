/*
 * pb.h — C ABI of the GB300 (sm_103a) forward pass of the parallel transformer block
 *
 *     y = x + MLP(LN(x)) + Attention(LN(x))
 *
 * (MegaScale reading notes, section 1.1 "Parallel Transformer Block", eq. (4)), where
 *   LN         = LayerNorm with gamma/beta, computed ONCE and shared by both branches;
 *   MLP(z)     = GeLU(z W1) W2               (Megatron-LM notes, section 2.1, Y = GeLU(XA)B);
 *   Attention  = multi-head attention on the [q | k | v] = z Wqkv projection (Megatron-LM
 *                notes, section 2.2), each query attending to the most recent `window`
 *                tokens of its own sequence, itself included (MegaScale reading notes,
 *                section 1.1 "Sliding Window Attention", eqs. (5)-(6)), followed by Wo.
 *
 * The library fuses the two branches: one GEMM against [Wqkv | W1] (GeLU in its
 * epilogue), one sliding-window flash attention kernel, and one GEMM of
 * [attn | GeLU(h)] against [Wo ; W2] with the residual added in its epilogue.
 *
 * Conventions for every entry point:
 *  - Tensors are bf16 (IEEE bfloat16 bit patterns), row-major, on the CURRENT CUDA
 *    device unless stated. Weights use the pages' Y = X W convention: [in, out].
 *  - Token rows are ordered (batch, position): x and y are [batch*seq, hidden].
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All work is
 *    enqueued asynchronously on it; no call synchronises the host, except
 *    pb_get_status, which reads a word the kernels write.
 *  - The library allocates NO device memory. The caller owns every buffer: inputs,
 *    outputs, the per-handle weight workspace and the per-call scratch.
 *  - Every function returns pb_status; no C++ exception crosses the ABI. Argument
 *    errors are detected before anything is enqueued. pb_last_error_message() returns
 *    a thread-local description of the last failure on the calling thread.
 *  - Device-side failures (a bounded wait inside a kernel that ran out) do not fault the
 *    GPU: the kernel records PB_ERR_DEVICE_TIMEOUT in the handle's status word and
 *    returns; pb_get_status reports it.
 */
#ifndef PB_H_
#define PB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pb_status {
  PB_OK = 0,
  PB_ERR_INVALID_ARG = 1,     /* NULL/misaligned pointer, bad size, partial aliasing   */
  PB_ERR_UNSUPPORTED = 2,     /* shape outside the supported set (see pb_dims)         */
  PB_ERR_WORKSPACE = 3,       /* workspace or scratch smaller than required            */
  PB_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (message has why)   */
  PB_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait expired; results are invalid  */
  PB_ERR_BAD_HANDLE = 6,      /* NULL, destroyed or foreign handle, or wrong device    */
  PB_ERR_RANGE = 7            /* PB_OPERANDS_FP16 only: a weight or an activation that */
                              /* feeds a GEMM exceeded the fp16 range (|v| > 65504)    */
} pb_status;

/*
 * Shape of one block. Supported (else PB_ERR_UNSUPPORTED):
 *   batch, seq >= 1; window >= 1 (window >= seq is full causal attention);
 *   head_dim in {64, 128}; hidden = heads * head_dim; hidden % 64 == 0; ffn % 64 == 0;
 *   batch * seq < 2^31; ln_eps > 0.
 */
typedef struct pb_dims {
  int32_t batch;
  int32_t seq;
  int32_t hidden;    /* H */
  int32_t heads;     /* nh */
  int32_t head_dim;  /* dh, H = nh * dh */
  int32_t ffn;       /* F, width of the MLP (4H on the pages) */
  int32_t window;    /* w: key k is visible to query i iff 0 <= i - k < w */
  float ln_eps;      /* LayerNorm epsilon, inside the square root */
  int32_t variant;   /* PB_BLOCK_LN_GELU (eq. (4) as written) or PB_BLOCK_RMS_SWIGLU */
} pb_dims;

/* Block variants. PB_BLOCK_RMS_SWIGLU replaces the LayerNorm by RMSNorm
 * (x / sqrt(mean x^2 + eps) * gamma; ln_beta unused) and the GeLU MLP by SwiGLU,
 * silu(z W_gate) * (z W_up) then W2: the fused "RMSNorm" and "SiLU + elementwise
 * multiply" kernels of the MegaScale reading notes, section 1.3 (named there without a
 * definition; the standard forms are used). */
typedef enum pb_block_variant { PB_BLOCK_LN_GELU = 0, PB_BLOCK_RMS_SWIGLU = 1 } pb_block_variant;

/*
 * Parameters of one block (device pointers, bf16). They are read only by pb_create,
 * which packs them into the workspace; they may be freed once the stream has passed
 * pb_create's work.
 *   ln_gamma, ln_beta : [H]     (ln_beta unused, may be NULL, for PB_BLOCK_RMS_SWIGLU)
 *   wqkv              : [H, 3H]; columns [Q | K | V], head j of each owns columns
 *                       [j*dh, (j+1)*dh) of its H-wide block
 *   w1                : [H, F]    (first MLP linear, "A" of Y = GeLU(XA)B); for
 *                       PB_BLOCK_RMS_SWIGLU [H, 2F] = [W_gate | W_up], and b1 is [2F]
 *   wo                : [H, H]    (attention output projection)
 *   w2                : [F, H]    (second MLP linear, "B")
 *   b_qkv [3H], b1 [F], b_o [H], b2 [H] : optional biases, NULL = none.
 */
typedef struct pb_weights {
  const void* ln_gamma;
  const void* ln_beta;
  const void* wqkv;
  const void* w1;
  const void* wo;
  const void* w2;
  const void* b_qkv;
  const void* b1;
  const void* b_o;
  const void* b2;
} pb_weights;

/* Byte offsets of the intermediates inside the scratch buffer of a forward call, valid
 * after the stream passes it (for inspection and tests):
 *   xn   [T, H]          LN(x)                      (bf16, fp16 with PB_OPERANDS_FP16)
 *   qk   [T, 2H]         [q | k], head-major columns (bf16)
 *   vt   [batch, heads, dh, seq_pad] v transposed per head, seq_pad = seq rounded up to 8
 *   act  [T, H + F]      [attention output (before Wo) | GeLU(h)]  (bf16 / fp16)
 *   q8, qscale           the FP8 operands of PB_OPERANDS_FP8 (see the fields)
 *   io, io2 [T, H]       bf16 staging of the host-buffer entry points
 *   res0, res1 [T, H]    fp32 residual stream between the layers of a stack
 *   sk                   stream-K partial tiles (fp32) and flags of the two GEMMs
 * T = batch * seq, F' = F (GeLU) or 2F (SwiGLU).
 * A training scratch (pb_forward_train / pb_backward, train_total bytes) has the same
 * regions up to `total`, then:
 *   hpre   [T, F']       h before the activation (bf16; SwiGLU: W1cat's interleaved order)
 *   lse    [batch * heads, seq64]  fp32 log2-sum-exp of each attention row's scores x
 *                        log2(e) / sqrt(dh); seq64 = seq rounded up to 64
 *   d_attn [T, H]        dL/d(attention output) (bf16)
 *   delta  [batch * heads, seq64]  fp32 dO . O per row
 *   dq_acc [T, H]        fp32 dq accumulator
 *   dz     [T, 3H + F']  [dq | dk | dv | dh], dL/d[q | k | v | h] (bf16, W1cat order)
 *   dxn    [T, H]        fp32 dL/dLN(x)
 *   stats  [T]           fp32 (mean, rstd) per row
 *   partials             fp32 partial column sums of the parameter gradients */
typedef struct pb_scratch_layout {
  size_t xn;
  size_t qk;
  size_t vt;
  size_t act;
  size_t io;
  size_t io2;
  size_t res0;
  size_t res1;
  size_t sk;  /* stream-K partial tiles and flags of the GEMMs */
  size_t q8;      /* PB_OPERANDS_FP8: [T, H + F] E4M3 codes of act (xn holds LN(x)'s codes) */
  size_t qscale;  /* PB_OPERANDS_FP8: [2T] fp32 row scales of LN(x), then of act */
  size_t seq_pad;
  size_t total;
  size_t hpre;
  size_t lse;
  size_t d_attn;
  size_t delta;
  size_t dq_acc;
  size_t dz;
  size_t dxn;
  size_t stats;
  size_t partials;
  size_t train_total;
} pb_scratch_layout;

/* Precision of the two GEMMs' operands. The pages' mixed-precision recipe computes in
 * bf16 with fp32 accumulation (Megatron-LM notes, section 5.4-5.5; performance notes,
 * "BF16 / FP16 / FP8"), which is the default. PB_OPERANDS_FP16 stores LN(x), the packed
 * weights, the attention output and GeLU(h) as fp16 instead: the same 16 bits and the
 * same tensor-core rate, 3 more mantissa bits, and a range limit of 65504 that the
 * kernels check (PB_ERR_RANGE). Attention (q, k, v, P) stays bf16 in both modes.
 * PB_OPERANDS_FP8 runs both GEMMs on FP8 E4M3 operands (the performance notes' FP8
 * recipe: E4M3 for the forward pass, only the GEMMs in FP8, LayerNorm, softmax and the
 * residual in bf16 / fp32) with current scaling per row: each row of LN(x) and of
 * [attention output | GeLU(h)], and each output channel of the packed weights, is scaled
 * by 448 / its largest magnitude; the GEMM epilogue multiplies the fp32 sum back by both
 * scales. Needs H and H + F to be multiples of 128; pb_forward_serial does not support it.
 * Not the reference precision: its results differ from the bf16 path by the E4M3 rounding
 * (3 mantissa bits). */
typedef enum pb_operand_precision {
  PB_OPERANDS_BF16 = 0,
  PB_OPERANDS_FP16 = 1,
  PB_OPERANDS_FP8 = 2
} pb_operand_precision;

typedef struct pb_options {
  int32_t operand_precision; /* pb_operand_precision */
  uint64_t wait_limit_ns;    /* limit of every bounded wait in the kernels; 0 = 2e9 */
} pb_options;

typedef struct pb_handle pb_handle;

/* Guard gaps (a debugging aid for out-of-bounds writes; the pages have no counterpart).
 * pb_set_guard_bytes(g) makes every workspace and scratch layout computed afterwards leave
 * g unused bytes after each of its regions (before the next region's 1024-byte alignment):
 * pb_weight_workspace_bytes, pb_create, pb_scratch_bytes, pb_train_scratch_bytes,
 * pb_get_scratch_layout and every call that takes a scratch buffer. No kernel reads or
 * writes those bytes, so a caller that fills the buffers with a known pattern can check
 * after its calls that nothing ran past the end of a region. g <= 1 MiB (else
 * PB_ERR_INVALID_ARG); default 0. It is process-wide: set it before sizing the buffers and
 * creating the handles that use them, and keep it until they are released (a handle keeps
 * the workspace layout of its pb_create; a scratch sized under another setting is too small
 * or laid out differently, and too small is reported as PB_ERR_WORKSPACE). */
pb_status pb_set_guard_bytes(size_t bytes);
pb_status pb_get_guard_bytes(size_t* bytes);

/* Bytes of the per-handle weight workspace (packed [Wqkv | W1] and [Wo ; W2] in the
 * K-major layout the tensor cores read, biases, LN parameters and the status word). */
pb_status pb_weight_workspace_bytes(const pb_dims* dims, size_t* bytes);

/* Bytes of the scratch one forward call needs (shared by all layers of a stack), and
 * its layout. */
pb_status pb_scratch_bytes(const pb_dims* dims, size_t* bytes);
pb_status pb_get_scratch_layout(const pb_dims* dims, pb_scratch_layout* layout);

/* Creates a handle for one block on the current device. `workspace` (device, 256-byte
 * aligned, >= pb_weight_workspace_bytes) is owned by the caller and must outlive the
 * handle. Enqueues the weight packing on `stream`. */
pb_status pb_create(const pb_dims* dims, const pb_weights* weights, void* workspace,
                    size_t workspace_bytes, void* stream, pb_handle** out);

/* pb_create with options (NULL = defaults: bf16 operands, 2 s wait limit). */
pb_status pb_create_ex(const pb_dims* dims, const pb_weights* weights, const pb_options* options,
                       void* workspace, size_t workspace_bytes, void* stream, pb_handle** out);

/* One block: y = x + MLP(LN(x)) + Attention(LN(x)). x, y: [batch*seq, hidden] bf16,
 * 16-byte aligned; y may equal x (in place), partial overlap is PB_ERR_INVALID_ARG.
 * `scratch` (device, 256-byte aligned, >= pb_scratch_bytes) must not be used by another
 * call that may run concurrently. */
pb_status pb_forward(pb_handle* h, const void* x, void* y, void* scratch, size_t scratch_bytes,
                     void* stream);

/* ------------------------------------------------------------------------------------
 * Training: the block's backward pass (the pages' subject is training: MFU counts the
 * forward's 2 and the backward's 4 FLOPs per weight and token, performance notes "MFU").
 * pb_forward_train is pb_forward that also keeps, in a training scratch, what the
 * backward reads: h before its activation and each attention row's log-sum-exp. The
 * attention probabilities are not kept; pb_backward recomputes them (the selective
 * recomputation of the MegaScale reading notes, section 1.3). Supported: bf16 operands
 * (PB_OPERANDS_BF16), head_dim 64 or 128; other operand precisions give
 * PB_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------------------- */

/* Bytes of the training scratch of pb_forward_train / pb_backward (train_total). */
pb_status pb_train_scratch_bytes(const pb_dims* dims, size_t* bytes);

/* pb_forward, keeping hpre and lse in `scratch` (>= pb_train_scratch_bytes) for a
 * following pb_backward on the same handle, x and scratch. */
pb_status pb_forward_train(pb_handle* h, const void* x, void* y, void* scratch,
                           size_t scratch_bytes, void* stream);

/* Gradients of the block, all device pointers: dx bf16 [T, H] (dL/dx, the residual path
 * included); every parameter gradient fp32 in the layout of its pb_weights entry
 * (dwqkv [H, 3H], dw1 [H, F'] = [gate | up] for SwiGLU, dwo [H, H], dw2 [F, H], biases
 * [3H], [F'], [H], [H], dgamma and dbeta [H]). NULL skips a bias gradient or dbeta. */
typedef struct pb_grads {
  void* dx;
  float* dgamma;
  float* dbeta;
  float* dwqkv;
  float* dw1;
  float* dwo;
  float* dw2;
  float* db_qkv;
  float* db1;
  float* db_o;
  float* db2;
} pb_grads;

/* The backward pass for upstream gradient dy (bf16 [T, H]) after pb_forward_train(h, x,
 * ...) with the same scratch: d_attn and dh from one GEMM against W2cat, the attention
 * backward (P recomputed from q, k and lse), dLN(x) from one GEMM against W1cat, the
 * normalisation backward plus dy (dx), and the weight gradients as two GEMMs over the
 * tokens ([dWo ; dW2] = act^T dy, [dWqkv | dW1] = LN(x)^T dz). accumulate != 0 adds the
 * fp32 parameter gradients to what the buffers hold (dx is always overwritten). */
pb_status pb_backward(pb_handle* h, const void* x, const void* dy, const pb_grads* grads,
                      int32_t accumulate, void* scratch, size_t scratch_bytes, void* stream);

/* The serial (standard) transformer block of eq. (3) (MegaScale reading notes, section 1.1,
 * "Parallel Transformer Block") on the handle's weights, for comparison with pb_forward:
 *   h = x + Attn(LN(x)),   y = h + MLP(LN'(h)),   MLP(z) = GeLU(z W1 + b1) W2 + b2,
 * with Attn(.) W_o + b_o as in pb_forward. The printed eq. (3) omits the attention term from
 * the outer sum; the derivation beside it (the parallel block replaces LN(x + h2) by LN(x))
 * requires it, so it is included. LN' has parameters ln2_gamma / ln2_beta (device bf16
 * [H], 16-byte aligned), or the handle's LayerNorm when both are NULL (eq. (3) writes the
 * same LN twice). x, y, scratch as in pb_forward (x == y allowed); h is kept in fp32 in
 * scratch res0. Seven kernel launches instead of four: the MLP waits for the attention
 * output. */
pb_status pb_forward_serial(pb_handle* h, const void* x, void* y, const void* ln2_gamma,
                            const void* ln2_beta, void* scratch, size_t scratch_bytes,
                            void* stream);

/* A stack of residual blocks (MegaScale reading notes, section 1.1: L layers give a
 * receptive field of L*w), x_{l+1} = block_l(x_l). All handles must have the same
 * dims. Between layers the residual stream stays in fp32 (scratch res0/res1; the pages
 * keep residual accumulation in BF16/FP32, performance notes, "BF16 / FP16 / FP8"): only
 * x and the final y are bf16. */
pb_status pb_forward_stack(pb_handle* const* layers, int32_t n_layers, const void* x, void* y,
                           void* scratch, size_t scratch_bytes, void* stream);

/* As pb_forward_stack, with y in fp32 (float [batch*seq, hidden], 16-byte aligned, not
 * overlapping x): the residual stream the stack carries between its layers, returned
 * without the final rounding to bf16 (the same stream as pb_forward_stack's y before that
 * rounding). For callers that keep the residual stream in fp32 across stacks. */
pb_status pb_forward_stack_f32(pb_handle* const* layers, int32_t n_layers, const void* x,
                               float* y, void* scratch, size_t scratch_bytes, void* stream);

/* As pb_forward_stack, with x and y in HOST memory (pinned memory gives asynchronous
 * copies): copies x to the device, runs the stack, copies y back, all on `stream`.
 * The caller synchronises the stream before reading y. */
pb_status pb_forward_stack_host(pb_handle* const* layers, int32_t n_layers, const void* x_host,
                                void* y_host, void* scratch, size_t scratch_bytes, void* stream);

/* A sequence of n_steps independent passes of the stack over host inputs, the loop of a
 * resident model serving a stream of batches: step s copies x_host[s] in, runs the stack,
 * copies y_host[s] out. Two device staging buffers (scratch io and io2) alternate and the
 * copies run on a copy stream the library creates in layers[0] on first use (released by
 * pb_destroy), so the input of step s + 1 and the output of step s - 1 move while step s
 * computes on `stream`. When `stream` reaches the point after this call, every y_host[s]
 * is written. x_host, y_host: arrays of n_steps host pointers (pinned memory for
 * asynchronous copies); a y_host[s] may equal an x_host[t] only if t <= s. The handles
 * must not be used by another host thread meanwhile. */
pb_status pb_forward_stack_host_steps(pb_handle* const* layers, int32_t n_layers,
                                      int32_t n_steps, const void* const* x_host,
                                      void* const* y_host, void* scratch, size_t scratch_bytes,
                                      void* stream);

/* Reads the handle's device status word (blocks until the word can be read on the
 * handle's device) and returns PB_OK or the first device-side error recorded since
 * the last pb_clear_status. */
pb_status pb_get_status(pb_handle* h);
pb_status pb_clear_status(pb_handle* h, void* stream);

/* Sets the limit, in nanoseconds, of every bounded wait inside this handle's kernels
 * (default 2e9). A wait that reaches it records PB_ERR_DEVICE_TIMEOUT and the kernel
 * returns. */
pb_status pb_set_wait_limit_ns(pb_handle* h, uint64_t limit_ns);

/* Per-kernel timing of this handle's forward calls. pb_trace_enable(h, n) makes the
 * next n forward calls record CUDA events (host-side event objects, no device memory)
 * around each of the block's four kernels on the call's stream; n = 0 turns tracing off.
 * pb_trace_read waits for the recorded events and returns in ms[4] the summed
 * milliseconds of [LayerNorm, first GEMM, attention, second GEMM] over the traced calls,
 * and their number in *calls. */
pb_status pb_trace_enable(pb_handle* h, int32_t n_calls);
pb_status pb_trace_read(pb_handle* h, float* ms, int32_t* calls);

/* Destroys the handle (host memory only; the caller frees the workspace). */
pb_status pb_destroy(pb_handle* h);

const char* pb_status_string(pb_status s);
const char* pb_last_error_message(void);

/* ------------------------------------------------------------------------------------
 * Single steps of the block, exported for testing and reuse. Same conventions.
 * ---------------------------------------------------------------------------------- */

/* Per-row current scaling of a bf16 [rows, cols] matrix to FP8 E4M3, the quantizer of
 * PB_OPERANDS_FP8 (performance notes, "BF16 / FP16 / FP8"), in fixed fp32 steps:
 * amax = max |x[r,:]|, inv = 448 / amax (0 if amax = 0), scales[r] = amax / 448,
 * codes[r,c] = E4M3(x[r,c] * inv) rounded to nearest even and saturated at +-448.
 * x: device bf16 [rows, cols], codes: device [rows, cols] bytes, scales: device fp32
 * [rows]; cols % 8 == 0, pointers 16-byte aligned. */
pb_status pb_quantize_rows_e4m3(int64_t rows, int32_t cols, const void* x, void* codes,
                                void* scales, void* stream);

/* LayerNorm (the LN of eq. (4)): out[r,:] = (x[r,:] - mean) / sqrt(var + eps) * gamma
 * + beta, biased variance, fp32 statistics. x, out: [rows, H] bf16; gamma, beta: [H]
 * bf16. H % 8 == 0, H <= 16384. beta == NULL gives RMSNorm instead (the fused kernel of
 * section 1.3): out[r,:] = x[r,:] / sqrt(mean x^2 + eps) * gamma. */
pb_status pb_layernorm(int64_t rows, int32_t H, const void* x, const void* gamma,
                       const void* beta, float eps, void* out, void* stream);

/* C[M, N] = A[M, K] * B[N, K]^T on the tensor cores (bf16 inputs, fp32 accumulation,
 * bf16 output rounded to nearest even): the contraction of every linear layer of the
 * block with the weight stored K-major. A, B, C 16-byte aligned; K % 64 == 0,
 * N % 32 == 0. `scratch` (device, 256-byte aligned, >= pb_gemm_scratch_bytes, or NULL)
 * lets the last waves of tiles be split along K across the SMs (stream-K); with NULL every
 * tile is computed whole. Calls that share a scratch buffer must not overlap on the GPU.
 * `status` (device int, may be NULL) receives PB_ERR_DEVICE_TIMEOUT if a bounded wait
 * runs out. */
pb_status pb_gemm_scratch_bytes(size_t* bytes);
pb_status pb_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, const void* B, void* C,
                       void* scratch, size_t scratch_bytes, int* status, void* stream);

/* pb_gemm_bf16 with either operand stored MN-major, the layouts of the backward pass's
 * GEMMs (activations stored token-major are MN-major when the contraction runs over
 * tokens): a_mn = 0: A is [M, K] (K contiguous), a_mn = 1: A is [K, M] (M contiguous);
 * b_mn = 0: B is [N, K], b_mn = 1: B is [K, N]. C[m, n] = sum_k A(m, k) B(n, k), bf16.
 * N % 32 == 0; a K-major operand needs K % 8 == 0, an MN-major one M (or N) % 8 == 0;
 * a ragged last block of K is zero filled. Otherwise as pb_gemm_bf16. */
pb_status pb_gemm_bf16_layout(int32_t M, int32_t N, int32_t K, const void* A, int32_t a_mn,
                              const void* B, int32_t b_mn, void* C, void* scratch,
                              size_t scratch_bytes, int* status, void* stream);

/* pb_gemm_bf16 for callers that cannot allocate device memory: plugins inside an engine or
 * framework whose device memory all belongs to the host program's allocator (they are
 * handed inputs and outputs, nothing more), and latency-bound paths where a cudaMalloc
 * could synchronise the device or block. The pages have no counterpart; it is a
 * convenience of this library. It computes the same product with the same stream-K
 * schedule as pb_gemm_bf16 with scratch, so its output is bit-identical to that call's,
 * with the scratch in a fixed array of the library's own device memory (25,171,968 bytes
 * per GPU, held until the process exits) instead of a caller buffer. It allocates nothing
 * and calls no allocating routine. Limits: GPUs with at most 192 SMs (96 CTA pairs);
 * otherwise PB_ERR_UNSUPPORTED, before anything is enqueued. The first call on each device
 * looks up the array's address (cudaGetSymbolAddress) in the device's primary context,
 * which must stay alive for the rest of the process; make that first call before any
 * stream capture. All calls share the one array, which keeps the last call's contents
 * (each call leaves its flags cleared): calls that can overlap on the GPU (other streams,
 * other host threads) race on it and must be serialised by the caller. */
pb_status pb_gemm_bf16_static(int32_t M, int32_t N, int32_t K, const void* A, const void* B,
                              void* C, int* status, void* stream);

/* Sliding-window causal attention alone (section 1.1, eqs. (5)-(6)) from the scratch
 * layout's qk and vt buffers into columns [0, H) of `act` ([T, act_ld] bf16). */
pb_status pb_swa_attention(const pb_dims* dims, const void* qk, const void* vt, void* act,
                           int64_t act_ld, int* status, void* stream);

/* Failure-detection self-test: one thread waits, with the kernels' bounded-wait
 * routine, on an mbarrier that nothing arrives at. After `limit_ns` it records
 * PB_ERR_DEVICE_TIMEOUT in *status (a device int) and the kernel returns; no copy, MMA
 * or tensor memory is involved, so the context stays usable. */
pb_status pb_wait_probe(uint64_t limit_ns, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PB_H_ */
