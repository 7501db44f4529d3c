// Linear layers on a handful of rows (the B rows of one position per
// sequence: the LM head of generation's last position, and every Linear of a
// decoding step with the key/value cache). With M <= GR_MAX_M rows the
// product is bound by reading the weight matrix once, not by the tensor rate:
// a tensor-core tile of 128 rows would be almost all padding, and the
// persistent tcgen05 GEMM's set-up dominates such a launch. Here each CTA
// stages the M input rows in shared memory; each warp streams weight rows
// (16-byte loads, the 32 lanes covering 512 consecutive bytes) and keeps one
// fp32 partial sum per input row, reduced across the warp at the end.
//   out[m, n] = sum_k A[m, k] W[n, k] (+ bias[n]), epilogues as the GEMM's:
//   STORE_ACT (bf16), GELU (gelu'(pre) and gelu(pre), bf16), STORE_F32 (fp32).
#include "common.cuh"

namespace k {

namespace {

constexpr int GR_THREADS = 256;
constexpr int GR_WARPS = GR_THREADS / 32;
constexpr int GR_MAX_M = 16;
constexpr int GR_R = 4;                  // weight rows per warp at a time

__device__ __forceinline__ float gr_tanh(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// gelu(x) = 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), and its
// derivative 0.5 (1 + t) + 0.5 x (1 - t^2) du/dx, from one tanh.
__device__ __forceinline__ void gr_gelu(float x, float& g, float& dg) {
    const float k0 = 0.7978845608028654f, k1 = 0.7978845608028654f * 0.044715f;
    const float x2 = x * x;
    const float t = gr_tanh(x * fmaf(k1, x2, k0));
    const float hx = 0.5f * x;
    g = fmaf(hx, t, hx);
    dg = fmaf(hx * fmaf(-t, t, 1.0f), fmaf(3.0f * k1, x2, k0), fmaf(0.5f, t, 0.5f));
}

template <int KIND, int MR>
__global__ void __launch_bounds__(GR_THREADS)
gemm_rows_kernel(const bf16* __restrict__ A, int64_t lda, const bf16* __restrict__ W, int64_t ldw, int M,
                 int N, int K, const float* __restrict__ bias, void* __restrict__ out, int64_t ldo,
                 bf16* __restrict__ out2, int64_t ldo2) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t gr_sm[];
    bf16* sA = (bf16*)gr_sm;                      // [MR][K], rows past M zero
    const int K8 = K / 8;                         // 16-byte pieces per row
    for (int i = threadIdx.x; i < MR * K8; i += GR_THREADS) {
        const int m = i / K8, c = i % K8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) v = *(const uint4*)(A + (int64_t)m * lda + 8 * c);
        *(uint4*)(sA + (int64_t)m * K + 8 * c) = v;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // each warp takes GR_R consecutive weight rows at a time: their loads are
    // in flight together and every staged input piece serves all of them
    for (int n0 = (blockIdx.x * GR_WARPS + warp) * GR_R; n0 < N; n0 += gridDim.x * GR_WARPS * GR_R) {
        float acc[GR_R][MR];
#pragma unroll
        for (int r = 0; r < GR_R; r++)
#pragma unroll
            for (int m = 0; m < MR; m++) acc[r][m] = 0.f;
        for (int c = lane; c < K8; c += 32) {
            float wf[GR_R][8];
#pragma unroll
            for (int r = 0; r < GR_R; r++) {
                uint4 wv = make_uint4(0u, 0u, 0u, 0u);
                if (n0 + r < N) wv = __ldg((const uint4*)(W + (int64_t)(n0 + r) * ldw + 8 * c));
                const __nv_bfloat162* w2 = (const __nv_bfloat162*)&wv;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float2 f = __bfloat1622float2(w2[e]);
                    wf[r][2 * e] = f.x;
                    wf[r][2 * e + 1] = f.y;
                }
            }
#pragma unroll
            for (int m = 0; m < MR; m++) {
                const uint4 av = *(const uint4*)(sA + (int64_t)m * K + 8 * c);
                const __nv_bfloat162* a2 = (const __nv_bfloat162*)&av;
                float af[8];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float2 f = __bfloat1622float2(a2[e]);
                    af[2 * e] = f.x;
                    af[2 * e + 1] = f.y;
                }
#pragma unroll
                for (int r = 0; r < GR_R; r++)
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[r][m] = fmaf(af[e], wf[r][e], acc[r][m]);
            }
        }
        // Reduce the GR_R * MR sums across the warp by halving: at offset o a
        // lane keeps the upper half of its current values if bit o of its
        // lane id is set, else the lower half, and adds the partner's copy of
        // the half it keeps. After the five steps lane L holds the complete
        // sums of flat indices 2L and 2L+1 (flat index r * MR + m).
        static_assert(GR_R * MR == 64, "the halving reduction assumes 64 sums per lane");
        float* v = &acc[0][0];
#pragma unroll
        for (int step = 0; step < 5; step++) {
            const int o = 16 >> step, h = 32 >> step;
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < h; i++) {
                const float send = up ? v[i] : v[i + h];
                const float recv = __shfl_xor_sync(0xffffffffu, send, o);
                v[i] = (up ? v[i + h] : v[i]) + recv;
            }
        }
        const int r = (2 * lane) / MR, m0 = (2 * lane) % MR, n = n0 + r;
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int m = m0 + q;
            if (m < M && n < N) {
                float x = v[q];
                if (bias) x += bias[n];
                if (KIND == EPI_STORE_F32) {
                    ((float*)out)[(int64_t)m * ldo + n] = x;
                } else if (KIND == EPI_GELU) {
                    float g, dg;
                    gr_gelu(x, g, dg);
                    ((bf16*)out)[(int64_t)m * ldo + n] = __float2bfloat16_rn(dg);
                    out2[(int64_t)m * ldo2 + n] = __float2bfloat16_rn(g);
                } else {
                    ((bf16*)out)[(int64_t)m * ldo + n] = __float2bfloat16_rn(x);
                }
            }
        }
    }
}

template <int KIND>
cudaError_t launch_rows(int M, int N, int K, const bf16* A, int64_t lda, const bf16* W, int64_t ldw,
                        const GemmEpi& e, cudaStream_t s) {
    const size_t smem = (size_t)GR_MAX_M * K * sizeof(bf16);
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        CUDA_OK(cudaFuncSetAttribute(gemm_rows_kernel<KIND, GR_MAX_M>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        attr_done.fetch_or(dbit);
    }
    const int want = (N + GR_WARPS * GR_R - 1) / (GR_WARPS * GR_R);
    const int grid = want < 2 * num_sms() ? want : 2 * num_sms();
    (void)pdl_launch(gemm_rows_kernel<KIND, GR_MAX_M>, grid, GR_THREADS, smem, s, A, lda, W, ldw, M, N, K, e.bias,
                     e.out, e.ldo, (bf16*)e.out2, e.ldo2);
    return cudaGetLastError();
}

}  // namespace

// Used where it measured faster than the tensor-core GEMM on 16 rows
// (GPT-2 124M decoding): K <= 1024 and N <= 4096 (the q/k/v, attention output
// and fc projections); the 3072-deep MLP output projection and the
// 50,304-column LM head keep the persistent tcgen05 GEMM.
bool gemm_rows_supported(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& e) {
    if (M < 1 || M > GR_MAX_M || N < 1 || K < 8 || K % 8) return false;
    if (K > 1024 || N > 4096) return false;
    if (!A.kmajor || !B.kmajor || A.ld % 8 || B.ld % 8) return false;
    if (((uintptr_t)A.ptr & 15) || ((uintptr_t)B.ptr & 15)) return false;
    if ((size_t)GR_MAX_M * K * sizeof(bf16) > 200 * 1024) return false;
    return e.kind == EPI_STORE_ACT || e.kind == EPI_GELU || e.kind == EPI_STORE_F32;
}

cudaError_t gemm_rows_bf16(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& e, cudaStream_t s) {
    if (!gemm_rows_supported(M, N, K, A, B, e)) return cudaErrorInvalidValue;
    const bf16* a = (const bf16*)A.ptr;
    const bf16* w = (const bf16*)B.ptr;
    switch (e.kind) {
        case EPI_STORE_ACT: return launch_rows<EPI_STORE_ACT>(M, N, K, a, A.ld, w, B.ld, e, s);
        case EPI_GELU: return launch_rows<EPI_GELU>(M, N, K, a, A.ld, w, B.ld, e, s);
        default: return launch_rows<EPI_STORE_F32>(M, N, K, a, A.ld, w, B.ld, e, s);
    }
}

}  // namespace k
