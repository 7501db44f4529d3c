// Shared definitions for the GPT-2 training-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <atomic>
#include <cstdlib>
#include <utility>

typedef __nv_bfloat16 bf16;

// Device status word bits (DevState::err).
#define ERR_TOKEN_RANGE   1u
#define ERR_TARGET_RANGE  2u
#define ERR_TIMEOUT       4u

// Scalars that live on the device so a whole step can run without host syncs.
struct DevState {
    double loss_sum;     // sum of per-row losses of the last forward
    float loss;          // loss_sum / n_valid
    int n_valid;         // targets != -1 in the last forward
    float inv_count;     // 1 / (n_valid * grad_accum_steps): d loss / d logits scale
    float grad_norm;     // pre-clip global norm of the last step
    float clip_coef;     // min(1, clip / (norm + 1e-6))
    int skip;            // 1 if the last step was skipped (non-finite norm)
    int step_t;          // AdamW step counter t
    float bc1, bc2;      // 1 - beta1^t, 1 - beta2^t for the current step
    unsigned int err;    // ERR_* bits, sticky until read by the host
    unsigned int timeout_site;
    unsigned int wait_limit;   // bounded-wait limit in SM cycles for single-CTA
                               // kernels; 0 means WAIT_LIMIT_CYCLES
};

// A GEMM operand: element (row r, reduction index k) of the logical [R, K]
// matrix sits at ptr[r*ld + k] when kmajor, else at ptr[k*ld + r].
struct GemmOperand {
    const void* ptr;
    int64_t ld;
    bool kmajor;
};

// GEMM epilogues. D[m,n] = acc[m,n] = sum_k A(m,k) B(n,k).
enum EpiKind : int {
    EPI_STORE_ACT = 0,   // out_act[m,n]  = acc + bias[n]
    EPI_GELU = 1,        // pre = acc + bias[n]; out_act[m,n] = gelu'(pre); out2_act[m,n] = gelu(pre)
    EPI_RESID = 2,       // out_f32[m,n]  = resid_f32[m,n] + acc + bias[n] (fp32 SIMT GEMM only)
    EPI_GELU_BWD = 3,    // out_act[m,n]  = acc * aux_act[m,n] (aux: the gelu'(pre) saved by EPI_GELU)
    EPI_ACCUM_F32 = 4,   // out_f32[m,n] += acc
    EPI_STORE_F32 = 5,   // out_f32[m,n]  = acc + bias[n]
};

struct GemmEpi {
    int kind;
    const float* bias;     // [N] or nullptr
    void* out;             // act or f32 per kind
    int64_t ldo;
    void* out2;            // EPI_GELU post-activation output (act)
    int64_t ldo2;
    const void* aux;       // EPI_RESID: f32 residual input; EPI_GELU_BWD: act gelu'(pre)
    int64_t ld_aux;
};

#define CUDA_OK(expr) do { cudaError_t e__ = (expr); if (e__ != cudaSuccess) return e__; } while (0)

// Programmatic dependent launch. Every kernel is launched with programmatic
// stream serialization (when enabled), so it may start while the kernel before
// it on the stream is finishing: it first runs its own set-up (barriers, TMEM,
// tensor-map prefetch), then pdl_wait() blocks until the previous kernel has
// completed and its writes are visible; nothing touches global memory before
// that. pdl_trigger() lets the next kernel be scheduled once every CTA of this
// one has issued it or exited: the short kernels issue it at their start (the
// next kernel's CTAs then fill the SMs their last wave frees), the persistent
// tensor-core kernels once a CTA has issued its last copies (so that waiting
// successors do not hold SMs while there is still work for them).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// PDL on unless GPT2_PDL=0 in the environment (read once per process).
inline bool pdl_on() {
    static const bool on = [] {
        const char* e = getenv("GPT2_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

// kern<<<grid, block, smem, s>>>(args...) with programmatic stream serialization.
template <typename... KArgs, typename... Args>
inline cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_on() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// tanh-form GELU (Hendrycks & Gimpel) and its derivative, fp32. The forward
// Linear that applies GELU saves gelu'(pre) (not pre): the backward then only
// multiplies by it.
__device__ __forceinline__ float gelu_f(float x) {
    const float a = 0.7978845608028654f, c = 0.044715f;
    float t = tanhf(a * (x + c * x * x * x));
    return 0.5f * x * (1.0f + t);
}
__device__ __forceinline__ float gelu_grad_f(float x) {
    const float a = 0.7978845608028654f, c = 0.044715f;
    float t = tanhf(a * (x + c * x * x * x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * a * (1.0f + 3.0f * c * x * x);
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Bounded device-side waits measure elapsed time on the SM's own cycle
// counter (monotonic for the warp that reads it) and give up after
// WAIT_LIMIT_CYCLES, about two seconds at B300 clocks; they then report
// ERR_TIMEOUT. The global nanosecond timer is not used: the CUDA driver may adjust
// it while a kernel runs, which would end a wait early.
__device__ __forceinline__ long long wait_clock() { return clock64(); }
#define WAIT_LIMIT_CYCLES 4000000000ll

// The limit a kernel's pipeline waits use: DevState::wait_limit when set
// (a test lowers it to make a wait run out), else WAIT_LIMIT_CYCLES. Kernels
// keep it in the shared-memory word right after their abort flag. Waits that
// drain in-flight copies after an abort always use WAIT_LIMIT_CYCLES, and so
// does every wait of a CTA pair: the peer's copies complete on the leader's
// barriers, so only a long wait covers them.
__device__ __forceinline__ unsigned int wait_limit_of(const DevState* st) {
    const unsigned int l = st ? st->wait_limit : 0u;
    return l ? l : (unsigned int)WAIT_LIMIT_CYCLES;
}

// ------------------------------------------------------------------ launchers
// All launchers return cudaSuccess or the launch error; `st` may be null.
namespace k {

cudaError_t validate_inputs(const int32_t* tok, const int32_t* tgt, int M, int V, DevState* st,
                            int accum, cudaStream_t s);
cudaError_t embed_fwd(const int32_t* tok, const float* wte, const float* wpe, float* x, int M,
                      int T, int C, int V, cudaStream_t s);
// Embedding backward, dwte[tok[m]] += dx[m] and dwpe[t] += sum_b dx[b*T+t],
// deterministic, in two parts: the sort of the token ids (depends on the
// tokens only) and the segmented sums of dx rows that use it.
size_t embed_bwd_workspace(int M, int C);
cudaError_t embed_bwd_sort(const int32_t* tok, int M, int V, void* workspace, cudaStream_t s);
cudaError_t embed_bwd_apply(const float* dx, float* dwte, float* dwpe, int M, int T, int C,
                            void* workspace, cudaStream_t s);

// Decoding with the key/value cache (one new position p per sequence):
// x[b] = wte[tok[b]] + wpe[p] for b < B (ids clamped and flagged), and the
// causal attention of the query row p of qkv [B, T, 3C] over the key/value
// rows 0..p, written to out [B, C] (hs <= 128), through a workspace of
// attention_decode_workspace_floats floats.
cudaError_t embed_rows(const int32_t* tok, const float* wte, const float* wpe, float* x, int B, int p, int C,
                       int V, DevState* st, cudaStream_t s);
size_t attention_decode_workspace_floats(int B, int T, int H, int hs);
template <typename Act>
cudaError_t attention_decode(const Act* qkv, Act* out, float* part, int B, int T, int H, int hs, int p,
                             cudaStream_t s);

// u = LN(x') with x' = x, or x' = x + y written to x_out when y != nullptr
// (the residual add of the preceding branch fused into the LayerNorm).
template <typename Act>
cudaError_t layernorm_fwd(const float* x, const Act* y, float* x_out, const float* g,
                          const float* b, Act* u, float* mu, float* rstd, int M, int C,
                          cudaStream_t s);
// dres (+)= LN backward of du; dres_act = Act copy of the new dres;
// dg, db += parameter gradients; dsum (optional) += column sums of the new
// dres (the bias gradient of the Linear whose output gradient it is). All
// two-stage, fixed order.
template <typename Act>
cudaError_t layernorm_bwd(const Act* du, const float* x, const float* g, const float* mu,
                          const float* rstd, float* dres, Act* dres_act, bool accumulate, float* dg,
                          float* db, float* dsum, int M, int C, float* partial, cudaStream_t s);
size_t layernorm_bwd_partial_floats(int M, int C);
// layernorm_bwd in its two parts: the row pass (dres, dres_act, and the
// per-block partials of dg, db and, with want_dsum, dsum into `partial`), and
// the fixed-order reduction of those partials (which may run on another stream
// once the row pass is done).
template <typename Act>
cudaError_t layernorm_bwd_rows(const Act* du, const float* x, const float* g, const float* mu,
                               const float* rstd, float* dres, Act* dres_act, bool accumulate,
                               bool want_dsum, int M, int C, float* partial, cudaStream_t s);
cudaError_t layernorm_bwd_params(const float* partial, int M, int C, float* dg, float* db, float* dsum,
                                 cudaStream_t s);

// db[n] += sum_m dy[m, n]; fixed-order two-stage reduction.
template <typename T>
cudaError_t colsum_add(const T* dy, int64_t ld, int M, int N, float* db, float* partial,
                       cudaStream_t s);
size_t colsum_partial_floats(int M, int N);
// db[n] += sum over g < groups of partial[g * N + n], in group order.
cudaError_t colsum_partials_add(const float* partial, int groups, int N, float* db, cudaStream_t s);

template <typename Act>
cudaError_t cross_entropy(Act* logits, const int32_t* tgt, float* row_loss, int M, int V, int Vp,
                          DevState* st, cudaStream_t s);
cudaError_t loss_reduce(const float* row_loss, int M, DevState* st, cudaStream_t s);

// One sampling step per row of logits (temperature, top-k keeping ties, softmax,
// inverse-CDF draw from u[row]); ctx (optional, int32 [rows, T], t valid
// tokens per row) receives the token at position t, or shifted in at T-1.
cudaError_t sample(const float* logits, int rows, int V, int64_t ld, float temperature, int top_k,
                   const float* u, int32_t* out, int32_t* ctx, int T, int t, cudaStream_t s);

cudaError_t grad_norm(const float* g, int64_t n, double* partial, int nparts, cudaStream_t s);
cudaError_t step_finalize(const double* partial, int nparts, float clip, float beta1, float beta2,
                          DevState* st, cudaStream_t s);
cudaError_t adamw(float* p, const float* g, float* m, float* v, bf16* p_bf16, int64_t n,
                  int64_t decay_end, int64_t bf16_end, float lr, float beta1, float beta2, float eps,
                  float wd, const DevState* st, cudaStream_t s);
cudaError_t f32_to_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t s);
cudaError_t splitk_reduce_add(const float* partial, int splits, int64_t n, float* out,
                              cudaStream_t s);

// attention on a fused qkv [B*T, 3C]
cudaError_t attention_fwd_f32(const float* qkv, float* out, float* lse, int B, int T, int H, int hs,
                              cudaStream_t s);
cudaError_t attention_bwd_f32(const float* qkv, const float* out, const float* lse,
                              const float* dout, float* dqkv, float* Dbuf, int B, int T, int H,
                              int hs, cudaStream_t s);
// tcgen05 flash attention (head size 64); bounded waits report into st
cudaError_t attention_fwd_bf16(const bf16* qkv, bf16* out, float* lse, int B, int T, int H, int hs,
                               DevState* st, cudaStream_t s);
// the tcgen05 backward; Dbuf [B,H,T] (scratch) receives rowsum(dout * out)
cudaError_t attention_bwd_bf16(const bf16* qkv, const bf16* out, const float* lse,
                               const bf16* dout, bf16* dqkv, float* Dbuf, int B, int T, int H,
                               int hs, DevState* st, cudaStream_t s);
cudaError_t attention_bwd_tc(const bf16* qkv, const bf16* out, const bf16* dout, const float* lse,
                             float* D, bf16* dqkv, int B, int T, int H, int hs, DevState* st,
                             cudaStream_t s);
bool attention_bf16_supported(int T, int hs);

// GEMMs
cudaError_t gemm_f32(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                     cudaStream_t s);
// tcgen05 GEMM; splits > 1 writes fp32 partials [splits][M][N] to epi.out
// (kind EPI_STORE_F32, no bias) for a later splitk_reduce_add.
cudaError_t gemm_bf16_tc(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                         int splits, DevState* st, cudaStream_t s);
bool gemm_bf16_tc_supported(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi);
// D = A B^T for at most 16 rows of A (bf16, both operands K-major), weight
// streaming without tensor cores; epilogues STORE_ACT, GELU, STORE_F32.
bool gemm_rows_supported(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi);
cudaError_t gemm_rows_bf16(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                           cudaStream_t s);

int num_sms();   // SM count of the current device
// Bit of the current device in a per-device set-up mask: kernel attributes
// (the dynamic shared-memory limit) and occupancy figures are per device, so
// host code that caches them keeps one flag per device (devices 0..63).
inline unsigned long long device_bit() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0) d = 0;
    return 1ull << (d & 63);
}

}  // namespace k
