/*
 * gpt2.h -- C ABI of the B300 GPT-2 training-step library (libgpt2_b300.so).
 *
 * One training iteration of GPT-2 on one GPU, as the pages state the problem
 * (nanoGPT guide, Part IV "The full life of one training iteration", Stages
 * 4-5): token + learned position embedding, pre-norm blocks of causal
 * multi-head self-attention and a tanh-GELU MLP, final LayerNorm, a
 * weight-tied LM head over a padded vocabulary, next-token cross-entropy,
 * backward, global grad-norm clip and AdamW.
 *
 * Conventions shared by every call
 *   - Return value: 0 on success, or a negative GPT2_E* code. The message of
 *     the last failure of a model is returned by gpt2_last_error().
 *   - Device work is enqueued on the model's stream (gpt2_set_stream) and is
 *     asynchronous unless a call says it synchronises. Errors raised on the
 *     device (bad token ids, an expired bounded wait) are recorded in a device
 *     status word and reported by the next call that synchronises.
 *   - The library owns every parameter, gradient, optimizer-state and
 *     activation buffer (device memory it allocates in gpt2_create, or for
 *     the decoding step on its first call, and frees in gpt2_destroy). The
 *     caller owns the token/target buffers and the
 *     stream; they must stay valid until the stream has passed the call.
 *   - Tokens are int32 (ids < 2^16 on the pages; nanoGPT guide Deep dive 3).
 *   - Not thread-safe: one host thread per model at a time.
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* error codes */
#define GPT2_OK                0
#define GPT2_EINVAL           -1   /* bad argument or configuration            */
#define GPT2_ENOMEM           -2   /* device or host allocation failed         */
#define GPT2_ECUDA            -3   /* a CUDA runtime/driver call failed        */
#define GPT2_ESTATE           -4   /* call out of order (e.g. backward first)  */
#define GPT2_ERANGE           -5   /* token or target id outside its range     */
#define GPT2_ETIMEOUT         -6   /* a bounded device-side wait expired       */
#define GPT2_ENONFINITE       -7   /* non-finite grad norm: update skipped     */

/* precision modes */
#define GPT2_FP32              0   /* every op in fp32, no tensor cores          */
#define GPT2_BF16              1   /* bf16 operands on tcgen05 tensor cores,
                                      fp32 accumulation, fp32 master state    */

/* buffer selectors for gpt2_copy_tensor / gpt2_set_tensor */
#define GPT2_PARAM             0
#define GPT2_GRAD              1
#define GPT2_ADAM_M            2
#define GPT2_ADAM_V            3

/*
 * Model configuration (nanoGPT guide Deep dive 1 GPTConfig; "Let's reproduce
 * GPT-2", 00:28:08 and 02:06:54).
 *   n_layer, n_head, d_model: L, H, C; head size hs = C / H.
 *   vocab_size: real vocabulary V (65 or 50257).
 *   padded_vocab: Vp >= V, a multiple of 64; 0 means V rounded up to a
 *     multiple of 128 (50304 for GPT-2). Columns V..Vp-1 of the logits are
 *     masked out of the softmax; rows V..Vp-1 of wte stay parameters.
 *   block_size: rows of the position table wpe (maximum T).
 *   batch_size, seq_len: B and T of every forward call, fixed at create.
 *   grad_accum_steps: micro-steps per optimizer step; each micro-step's loss
 *     gradient is divided by it (sotaaz Section 3). 0 means 1.
 *   precision: GPT2_FP32 or GPT2_BF16.
 */
typedef struct {
    int n_layer;
    int n_head;
    int d_model;
    int vocab_size;
    int padded_vocab;
    int block_size;
    int batch_size;
    int seq_len;
    int grad_accum_steps;
    int precision;
} gpt2_config;

typedef struct gpt2_model gpt2_model;   /* opaque; owns all device memory */

/*
 * gpt2_create -- allocate a model on the current CUDA device and initialise
 * its parameters ("Let's reproduce GPT-2" 01:13:47; nanoGPT guide Deep dive 1):
 * wte, wpe and every Linear weight ~ N(0, 0.02^2); attn_proj.W and
 * mlp_proj.W ~ N(0, (0.02/sqrt(2 n_layer))^2); biases 0; LayerNorm gain 1,
 * shift 0. The normals come from a counter-based generator (SplitMix64 +
 * Box-Muller): tensor k (canonical order), element i uses state
 * seed ^ (k*2^40 + i). Grads, Adam moments and the step counter start at 0.
 *   cfg: read only, copied. out: receives the new model (NULL on failure).
 * Errors: EINVAL (NULL, sizes <= 0, d_model % n_head != 0, seq_len >
 * block_size, padded_vocab < vocab_size, a shape the chosen precision does
 * not support), ENOMEM, ECUDA. Synchronises. On failure everything already
 * allocated is freed. Testing hook: with GPT2_FAIL_ALLOC_AT=n in the
 * environment, the n-th device allocation (from 0) fails with ENOMEM before
 * any cudaMalloc (allocation 0 precedes every CUDA call of gpt2_create).
 */
int gpt2_create(const gpt2_config* cfg, uint64_t seed, gpt2_model** out);

/* Free every device buffer of the model. NULL is a no-op. Synchronises. */
void gpt2_destroy(gpt2_model* model);

/* Enqueue all later work on cuda_stream (a cudaStream_t; NULL = legacy
 * default stream). The caller keeps ownership of the stream. Inside
 * gpt2_backward the weight-gradient work (dW GEMMs, bias gradients) runs on a
 * second stream that the library owns; it is forked from and joined back to
 * this stream by events before gpt2_backward returns, so the caller sees one
 * ordered stream (and a stream capture records both branches). gpt2_step's
 * AdamW also runs there, group by group in the order the next gpt2_forward
 * reads the parameters (which waits for each group just before using it), and
 * gpt2_zero_grad queues behind it; every other call that touches model state
 * (gpt2_sync, tensor copies, profiling, gpt2_set_stream) first makes this
 * stream wait for it. gpt2_get_loss does not (the loss comes from the forward). */
int gpt2_set_stream(gpt2_model* model, void* cuda_stream);

/*
 * gpt2_forward -- GPT.forward(idx, targets) (nanoGPT guide Part IV Stage 4):
 * logits = ln_f(blocks(wte[idx] + wpe[0:T])) wte^T and, with targets, the
 * mean next-token cross-entropy over targets != -1 (ignore_index = -1).
 *   d_tokens:  device int32 [B*T], row-major (b, t); ids in [0, V).
 *   d_targets: device int32 [B*T] in [0, V) or -1, or NULL for logits only
 *              (a later gpt2_backward then fails with ESTATE).
 *   h_loss:    host float* receiving the mean loss (synchronises), or NULL
 *              (no synchronisation; read it later with gpt2_get_loss).
 * With targets, the logits buffer is overwritten in place by d loss/d logits
 * for the following backward (fused softmax-cross-entropy).
 * Errors: EINVAL (NULL tokens); ERANGE reported when synchronising if an id
 * was out of range (the kernels clamp it and keep going).
 */
int gpt2_forward(gpt2_model* model, const int32_t* d_tokens, const int32_t* d_targets,
                 float* h_loss);

/*
 * gpt2_forward_last -- the forward of generation ("Let's reproduce GPT-2",
 * 00:37:02 the sampling loop; nanoGPT guide Deep dive 1, the LM head applied
 * to the last position only at inference): the blocks run on the [B, T]
 * context as in gpt2_forward, then the tied head on position t-1 of each
 * sequence only. Positions t..T-1 may hold anything (causal attention keeps
 * them out of position t-1).
 *   d_tokens: device int32 [B*T] (the model's B and T); t in [1, T].
 *   d_logits: device fp32 [B, V] row-major, caller-owned; receives the logits
 *             of position t-1 of every sequence (real vocabulary only).
 * No loss, no backward afterwards (ESTATE). Does not synchronise.
 * Errors: EINVAL (NULL pointers, t outside [1, T]); ERANGE as gpt2_forward.
 */
int gpt2_forward_last(gpt2_model* model, const int32_t* d_tokens, int t, float* d_logits);

/*
 * gpt2_decode_step -- one generation step with the key/value cache. The
 * pages' sampling loop ("Let's reproduce GPT-2", 00:37:02; nanoGPT guide,
 * sample.py) runs the whole context through the model for every new token;
 * with absolute position embeddings the keys and values of the earlier
 * positions do not change, so this step computes position t-1 alone and
 * reads the others' keys and values from the cache that gpt2_forward_last and
 * earlier steps left in the model. The logits equal gpt2_forward_last's on
 * the context extended by the new tokens, up to rounding.
 *   d_tokens: device int32 [B], the token at position t-1 of every sequence.
 *   t:        in [1, T]; positions 0..t-2 must be cached: the last call on
 *             this model was gpt2_forward_last with a t' >= t-1 or
 *             gpt2_decode_step with t' >= t-1, and no training forward,
 *             optimizer step, gpt2_set_tensor or gpt2_load came after it.
 *   d_logits: device fp32 [B, V] row-major, caller-owned; receives the logits
 *             of position t-1 of every sequence (real vocabulary only).
 * Once a context holds T tokens, the pages' crop shifts every position, so
 * the next token needs gpt2_forward_last on the cropped context. The first
 * call allocates the step's row buffers (B rows of 30 C bytes in bf16, 52 C
 * in fp32) and the decoding attention's span partials (B H ceil(T/64)
 * (hs + 2) floats); no backward afterwards (ESTATE). Does not synchronise.
 * Errors: EINVAL (NULL pointers, t outside [1, T], a head size above 128);
 * ESTATE (positions 0..t-2 not cached); ENOMEM; ERANGE as gpt2_forward.
 */
int gpt2_decode_step(gpt2_model* model, const int32_t* d_tokens, int t, float* d_logits);

/*
 * gpt2_backward -- gradient of (loss / grad_accum_steps) added (+=) into the
 * gradient buffers (nanoGPT guide Part IV Stage 4 "backward() accumulates
 * gradients"). Needs a preceding gpt2_forward with targets (else ESTATE).
 */
int gpt2_backward(gpt2_model* model);

/*
 * gpt2_step -- clip then AdamW (nanoGPT guide Part IV Stage 5; sotaaz Section 3):
 *   norm = ||all gradients||_2 (wte once); every gradient is scaled by
 *   min(1, clip / (norm + 1e-6)); then with t = t + 1, for each parameter:
 *   p *= 1 - lr*weight_decay (2-D parameters only: wte, wpe, Linear weights),
 *   m = beta1 m + (1-beta1) g, v = beta2 v + (1-beta2) g^2,
 *   p -= lr * (m / (1-beta1^t)) / (sqrt(v / (1-beta2^t)) + eps).
 * If norm is not finite the update is skipped on the device (t unchanged).
 *   h_grad_norm: host float* receiving the pre-clip norm (synchronises; the
 *   call then returns ENONFINITE for a skipped update), or NULL.
 * The gradient buffers are left unscaled (the clip coefficient is applied
 * inside the update); call gpt2_zero_grad before the next micro-step.
 */
int gpt2_step(gpt2_model* model, float lr, float beta1, float beta2, float eps,
              float weight_decay, float clip, float* h_grad_norm);

/* optimizer.zero_grad() (nanoGPT guide Part IV Stage 5): gradients = 0. */
int gpt2_zero_grad(gpt2_model* model);

/* Warmup + cosine learning rate (nanoGPT guide Stage 1 and Lab 4; "Let's
 * reproduce GPT-2" 02:21:06): it < warmup: lr_max*(it+1)/warmup; it > horizon:
 * lr_min; otherwise lr_min + 0.5*(1+cos(pi*(it-warmup)/(horizon-warmup)))*
 * (lr_max-lr_min). Host-only arithmetic; no GPU needed. */
double gpt2_lr_schedule(int64_t it, int64_t warmup, int64_t horizon, double lr_max,
                        double lr_min);

/* ---------------------------------------------------------------- inspection */

/* Synchronise the stream and report any recorded device error. */
int gpt2_sync(gpt2_model* model);

/* Make the model's stream wait for everything the library queued on its
 * second stream (a pending AdamW update and zero_grad), without synchronising
 * the host: work the caller enqueues on the stream afterwards (an event, a
 * copy of the parameters) sees the finished update. */
int gpt2_join(gpt2_model* model);

/* Mean loss of the last forward with targets (synchronises). */
int gpt2_get_loss(gpt2_model* model, float* h_loss);

/* Enqueue a copy of the last forward's mean loss into h_loss (4 bytes of host
 * memory, page-locked for the copy to be asynchronous) on the model's stream,
 * without synchronising: the value is there once the stream has reached this
 * point (e.g. after gpt2_sync). A training loop reads the loss of every step
 * this way without stalling the device. Device-side conditions are reported by
 * the next synchronising call. Errors: EINVAL (NULL pointers). */
int gpt2_get_loss_async(gpt2_model* model, float* h_loss);

/* Testing hook for failure detection (no counterpart on the pages). Every
 * pipeline wait inside the library's single-CTA tensor-core kernels gives up
 * after `cycles` SM cycles (0 restores the default, about two seconds), after
 * which the kernel records ERR_TIMEOUT, drains its copies, frees its tensor
 * memory and returns; the next synchronising call reports GPT2_ETIMEOUT and
 * the model stays usable. CTA-pair GEMMs keep the default limit. A limit of a
 * few hundred cycles makes waits expire on purpose. Synchronises. */
int gpt2_set_wait_limit(gpt2_model* model, unsigned int cycles);

/* Number of parameter tensors (canonical order: wte, wpe, per layer ln1.g,
 * ln1.b, attn.W, attn.b, attn_proj.W, attn_proj.b, ln2.g, ln2.b, fc.W, fc.b,
 * mlp_proj.W, mlp_proj.b, then lnf.g, lnf.b). */
int gpt2_num_tensors(const gpt2_model* model);

/* Name (static string owned by the model), rank, shape and decay flag of
 * tensor i. Any out pointer may be NULL. */
int gpt2_tensor_info(const gpt2_model* model, int i, const char** name, int* ndim,
                     int64_t shape[2], int* decays);

/* Copy tensor i of buffer `which` (GPT2_PARAM/GRAD/ADAM_M/ADAM_V) to host fp32
 * h_dst (prod(shape) floats). Synchronises. */
int gpt2_copy_tensor(gpt2_model* model, int i, int which, float* h_dst);

/* Overwrite tensor i of buffer `which` from host fp32 h_src; the bf16 copy the
 * tensor cores read is refreshed too. Synchronises. */
int gpt2_set_tensor(gpt2_model* model, int i, int which, const float* h_src);

/* Copy rows [row0, row0+nrows) of the logits buffer, real columns 0..V-1, as
 * fp32 into h_dst [nrows*V]. After a forward without targets these are the
 * logits; after one with targets they are d loss/d logits. Synchronises. */
int gpt2_copy_logits(gpt2_model* model, int64_t row0, int64_t nrows, float* h_dst);

/* Copy the per-row losses of the last forward with targets (fp32 [nrows];
 * 0 for ignored rows). Synchronises. */
int gpt2_copy_row_losses(gpt2_model* model, int64_t row0, int64_t nrows, float* h_dst);

/* Checkpoint of the training state: the pages' ckpt.pt holds the model, the
 * optimizer state and the iteration (nanoGPT guide, "train.py": saving and
 * --init_from=resume). gpt2_save writes the configuration, the AdamW step
 * counter and the fp32 parameter, first-moment and second-moment arenas to the
 * file `path` (created or truncated). gpt2_load reads such a file into a model
 * created with the same configuration (EINVAL otherwise, and for a file that is
 * not a checkpoint of this library): it replaces parameters, moments and the
 * step counter, rebuilds the bf16 weight copy from the fp32 parameters, and
 * leaves the gradients as they are. Training resumed from a checkpoint is
 * bit-identical to training that never stopped. Both synchronise; EINVAL also
 * for I/O failures (the message names the file). The header and configuration
 * are checked before anything is overwritten; a file truncated inside the
 * arrays leaves the model's parameters and moments partly replaced (load a
 * good checkpoint, or recreate the model). Format: 16-byte magic
 * "GPT2B300CKPT\0v1\0", the ten int32 fields of gpt2_config, int64 arena
 * length n, int32 step counter, then three arrays of n little-endian fp32. */
int gpt2_save(gpt2_model* model, const char* path);
int gpt2_load(gpt2_model* model, const char* path);

/* Parameter count; the tied matrix counted once (nanoGPT guide Deep dive 1).
 * include_wpe: count the position table; padded: count wte as Vp rows. */
int64_t gpt2_num_params(const gpt2_model* model, int include_wpe, int padded);

/* Host-side init of tensor k of a model with configuration cfg, exactly as
 * gpt2_create computes it (fp32 values into h_dst). Needs no GPU. */
int gpt2_host_init_tensor(const gpt2_config* cfg, uint64_t seed, int k, float* h_dst);

/* Message of the last failure of this model (or of the last failed
 * gpt2_create when model is NULL). Never NULL. */
const char* gpt2_last_error(const gpt2_model* model);

/*
 * Per-site profiling. Every launch site of forward/backward/step/zero_grad
 * (one Linear's GEMM, a LayerNorm, the cross-entropy, AdamW, ...) counts its
 * calls, its kernel launches and its algorithmic work: FLOPs of the method
 * (2*M*N*K for a GEMM; the causal attention products) and the HBM bytes its
 * operands and results must move at least once. With profiling on, CUDA events
 * are also recorded on the model's stream around each site and their elapsed
 * times summed (adds one event pair per site; for measurement, not the timed
 * training loop). While event timing is on, the backward's weight-gradient
 * work stays on the model's stream so that every site is timed alone.
 *   gpt2_profile(model, on): fold pending timings, clear every entry, set
 *     event timing on/off. Counting is always on.
 *   gpt2_profile_count: synchronise, fold pending timings, return the number
 *     of sites seen since the last gpt2_profile call.
 *   gpt2_profile_entry: totals of site i; `name` is a static string. Any out
 *     pointer may be NULL.
 */
int gpt2_profile(gpt2_model* model, int on);
int gpt2_profile_count(gpt2_model* model);
int gpt2_profile_entry(gpt2_model* model, int i, const char** name, int64_t* calls,
                       int64_t* kernels, double* ms, double* flops, double* bytes);

/* Library version string. */
const char* gpt2_version(void);

/* ------------------------------------------------------- op-level entry points
 * The individual kernels of the path, for testing and measurement. All
 * pointers are device pointers; work goes on `stream` (cudaStream_t).
 * Return EINVAL for shapes a kernel does not support, ECUDA on launch failure.
 */

/* D[m,n] = sum_k A(m,k) B(n,k) on tcgen05 tensor cores; A, B bf16, fp32
 * accumulate, D written as bf16 (out_bf16 != NULL) or fp32 (out_f32 != NULL,
 * accumulate != 0 adds into it). A(m,k) is at A[m*lda + k] if a_kmajor else
 * A[k*lda + m]; B(n,k) likewise with ldb, b_kmajor. bias (fp32 [N]) optional.
 * lda, ldb, ldd multiples of 8; pointers 16-byte aligned. */
int gpt2_op_gemm_bf16(int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                      const void* B, int64_t ldb, int b_kmajor, const float* bias,
                      void* out_bf16, float* out_f32, int64_t ldd, int accumulate,
                      void* stream);

/* The two GELU epilogues of the MLP's GEMMs (nanoGPT guide Deep dive 1, the
 * MLP block c_fc -> GELU(tanh) -> c_proj; "Let's reproduce GPT-2" on the tanh
 * approximation), same operand conventions as gpt2_op_gemm_bf16, all outputs
 * bf16 [M, N] with row stride ldd:
 *   backward == 0: pre = A B^T + bias (bias fp32 [N] or NULL);
 *                  out = gelu'(pre), out2_or_aux = gelu(pre)
 *                  (the forward of c_fc, saving the derivative for the backward)
 *   backward != 0: out = (A B^T) * aux with aux = out2_or_aux (bf16 [M, N], the
 *                  saved gelu'(pre)); bias must be NULL
 *                  (the input gradient of c_proj carried through the GELU)
 * tanh is the hardware approximation (absolute error about 2^-11).
 * EINVAL for NULL pointers, a bias with backward != 0, or shapes/alignments
 * gpt2_op_gemm_bf16 rejects. */
int gpt2_op_gemm_bf16_gelu(int M, int N, int K, const void* A, int64_t lda, int a_kmajor,
                           const void* B, int64_t ldb, int b_kmajor, const float* bias,
                           int backward, void* out, void* out2_or_aux, int64_t ldd,
                           void* stream);

/* Synchronise `stream` and report device-side conditions raised by the
 * op-level calls (including gpt2_op_attention_bwd_noalloc) on the current
 * device since the previous gpt2_op_sync: GPT2_ETIMEOUT if a bounded wait
 * inside a kernel expired (the kernel then skipped its remaining work, so its
 * outputs are incomplete). Clears the recorded conditions. Allocates nothing. */
int gpt2_op_sync(void* stream);

/* Testing hook (no counterpart on the pages): the bounded-wait limit, in SM
 * cycles, of the op-level calls' single-CTA kernels on the current device
 * (0 = the default, about two seconds); see gpt2_set_wait_limit. Creates the
 * status word of the allocating op-level calls if it does not exist yet. */
int gpt2_op_set_wait_limit(unsigned int cycles);

/* One sampling step of generation ("Let's reproduce GPT-2", 00:37:02; nanoGPT
 * guide, sample.py), per row r < rows of logits (device fp32, row stride ld
 * >= V, V columns):
 *   x = logits / temperature; with 0 < top_k < V only the entries >= the k-th
 *   largest x are kept (ties with it too, as the pages' topk mask keeps them);
 *   p = softmax over the kept entries; the token is the smallest j whose
 *   cumulative p exceeds u[r] (device fp32, u in [0, 1), caller-drawn).
 * temperature <= 0 takes the argmax (lowest index on ties) instead.
 *   out: device int32 [rows] receives the tokens.
 *   ctx: optional device int32 [rows, T] context holding t tokens per row
 *        (1 <= t <= T <= 1024): the token is written at position t, or, when
 *        t == T, the row shifts left by one and the token goes to T-1 (the
 *        pages' crop of the context to the block size). NULL: no append.
 * Deterministic (fixed-order reductions). Errors: EINVAL for bad sizes. */
int gpt2_op_sample(const float* logits, int rows, int V, int64_t ld, float temperature, int top_k,
                   const float* u, int32_t* out, int32_t* ctx, int T, int t, void* stream);

/* Causal attention forward on a fused qkv buffer [B*T, 3C] (bf16 when
 * precision == GPT2_BF16, else fp32): out [B*T, C], lse fp32 [B, H, T]
 * (natural log of each softmax row's normaliser, scores scaled by 1/sqrt(hs)). */
int gpt2_op_attention_fwd(int precision, int B, int T, int H, int hs, const void* qkv,
                          void* out, float* lse, void* stream);

/* Causal attention backward: given dout [B*T, C], qkv, out and lse from the
 * forward, writes dqkv [B*T, 3C]. scratch: fp32 [B*H*T] for rowsum(dout*out). */
int gpt2_op_attention_bwd(int precision, int B, int T, int H, int hs, const void* qkv,
                          const void* out, const float* lse, const void* dout, void* dqkv,
                          float* scratch, void* stream);

/* Allocation-free variant of gpt2_op_attention_bwd (this entry point has no
 * counterpart on the pages: it exists for callers that may not allocate device
 * memory themselves, e.g. a plugin whose host application owns every device
 * allocation, or code bound by a no-cudaMalloc-after-start-up policy).
 * Arguments, layouts and results are those of gpt2_op_attention_bwd without
 * `scratch`: the fp32 rowsum(dout*out) scratch instead lives in a fixed array
 * of 2^20 floats (4 MiB) compiled into the library, which every device that
 * loads the library holds until the process exits. The caller still owns and
 * passes qkv, out, lse, dout and dqkv.
 *  - B*H*T must be <= 2^20 (1,048,576): larger sizes return GPT2_EINVAL with a
 *    message in gpt2_last_error(NULL), before any device work.
 *  - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it; make that
 *    first call outside any stream capture.
 *  - Every call on a device shares the one array, which keeps the previous
 *    call's contents (each call rewrites every row it reads, so no clearing is
 *    needed). Calls that may overlap on the GPU (different streams, no ordering
 *    between them) race on it: order them on one stream or with events.
 *  - A bounded-wait expiry inside its kernels is recorded in a status word
 *    that is also compiled into the library, and reported by gpt2_op_sync.
 * Return codes as gpt2_op_attention_bwd. */
int gpt2_op_attention_bwd_noalloc(int precision, int B, int T, int H, int hs, const void* qkv,
                                  const void* out, const float* lse, const void* dout,
                                  void* dqkv, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_H */
