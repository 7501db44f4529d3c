// fp32 SIMT GEMM for the fp32-math mode (no tensor cores): D = A B^T with the
// same operand conventions and epilogues as the tcgen05 path. 64x64 output
// tile per CTA, k-slab of 16 staged in shared memory, 4x4 outputs per thread.
#include "common.cuh"

namespace k {

static constexpr int SB = 64, SK = 16;

__device__ __forceinline__ float ld_op(const float* p, int64_t ld, bool kmajor, int r, int kk) {
    return kmajor ? p[(int64_t)r * ld + kk] : p[(int64_t)kk * ld + r];
}

__global__ void __launch_bounds__(256)
gemm_f32_kernel(int M, int N, int K, const float* __restrict__ A, int64_t lda, bool ak,
                const float* __restrict__ B, int64_t ldb, bool bk, GemmEpi epi) {
    pdl_wait();
    pdl_trigger();
    __shared__ float As[SK][SB + 4];
    __shared__ float Bs[SK][SB + 4];
    const int m0 = blockIdx.y * SB, n0 = blockIdx.x * SB;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SK) {
        for (int i = threadIdx.x; i < SB * SK; i += 256) {
            int r, kk;
            if (ak) { r = i / SK; kk = i % SK; } else { kk = i / SB; r = i % SB; }
            int gm = m0 + r, gk = k0 + kk;
            As[kk][r] = (gm < M && gk < K) ? ld_op(A, lda, ak, gm, gk) : 0.f;
            if (bk) { r = i / SK; kk = i % SK; } else { kk = i / SB; r = i % SB; }
            int gn = n0 + r;
            gk = k0 + kk;
            Bs[kk][r] = (gn < N && gk < K) ? ld_op(B, ldb, bk, gn, gk) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SK; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            float bias = epi.bias ? epi.bias[n] : 0.f;
            switch (epi.kind) {
                case EPI_STORE_ACT:
                case EPI_STORE_F32:
                    ((float*)epi.out)[(int64_t)m * epi.ldo + n] = v + bias;
                    break;
                case EPI_GELU: {
                    float pre = v + bias;
                    ((float*)epi.out)[(int64_t)m * epi.ldo + n] = gelu_grad_f(pre);
                    ((float*)epi.out2)[(int64_t)m * epi.ldo2 + n] = gelu_f(pre);
                    break;
                }
                case EPI_RESID:
                    ((float*)epi.out)[(int64_t)m * epi.ldo + n] =
                        ((const float*)epi.aux)[(int64_t)m * epi.ld_aux + n] + v + bias;
                    break;
                case EPI_GELU_BWD:
                    ((float*)epi.out)[(int64_t)m * epi.ldo + n] =
                        v * ((const float*)epi.aux)[(int64_t)m * epi.ld_aux + n];
                    break;
                case EPI_ACCUM_F32:
                    ((float*)epi.out)[(int64_t)m * epi.ldo + n] += v;
                    break;
            }
        }
    }
}

cudaError_t gemm_f32(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                     cudaStream_t s) {
    dim3 grid((N + SB - 1) / SB, (M + SB - 1) / SB);
    (void)pdl_launch(gemm_f32_kernel, grid, 256, 0, s, M, N, K, (const float*)A.ptr, A.ld, A.kmajor,
                                         (const float*)B.ptr, B.ld, B.kmajor, epi);
    return cudaGetLastError();
}

}  // namespace k
