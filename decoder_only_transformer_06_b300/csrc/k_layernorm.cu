// LayerNorm forward and backward (nn.LayerNorm semantics, eps = 1e-5, biased
// variance; "Build GPT from scratch" forty-line model, nanoGPT guide Deep
// dive 1). One warp per row; lane l owns columns l, l+32, ... so the loads of
// a warp are contiguous. fp32 math throughout; the normalised output is
// written in the activation type (bf16 operand of the next GEMM, or fp32).
#include "common.cuh"

namespace k {

static constexpr float LN_EPS = 1e-5f;
static constexpr int LN_WARPS = 8;

template <typename Act, int EPL>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_fwd_kernel(const float* __restrict__ x, const float* __restrict__ g,
              const float* __restrict__ b, Act* __restrict__ u, float* __restrict__ mu_out,
              float* __restrict__ rstd_out, int M, int C) {
    int row = blockIdx.x * LN_WARPS + threadIdx.x / 32;
    int lane = threadIdx.x % 32;
    if (row >= M) return;
    const float* xr = x + (int64_t)row * C;
    float v[EPL];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        v[j] = c < C ? xr[c] : 0.f;
        s += v[j];
    }
    float mean = warp_sum(s) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        float d = c < C ? v[j] - mean : 0.f;
        q += d * d;
    }
    float var = warp_sum(q) / (float)C;
    float rstd = 1.0f / sqrtf(var + LN_EPS);
    Act* ur = u + (int64_t)row * C;
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        if (c < C) ur[c] = from_f<Act>((v[j] - mean) * rstd * g[c] + b[c]);
    }
    if (lane == 0) {
        mu_out[row] = mean;
        rstd_out[row] = rstd;
    }
}

// Backward of y = xhat*g + b, xhat = (x - mu)*rstd:
//   dxhat = dy*g; dx = rstd*(dxhat - mean(dxhat) - xhat*mean(dxhat*xhat));
//   dg = sum_rows dy*xhat; db = sum_rows dy.
// Rows are dealt to warps in a fixed pattern; each CTA writes its dg/db
// partial, and ln_param_reduce adds the partials in CTA order.
template <typename Act, int EPL>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_bwd_kernel(const Act* __restrict__ du, const float* __restrict__ x,
              const float* __restrict__ g, const float* __restrict__ mu,
              const float* __restrict__ rstd_in, float* __restrict__ dres,
              Act* __restrict__ dres_act, int accumulate, float* __restrict__ partial, int M,
              int C) {
    extern __shared__ float sm[];   // [LN_WARPS][2][C]
    int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float pg[EPL], pb[EPL], gv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        pg[j] = 0.f;
        pb[j] = 0.f;
        gv[j] = c < C ? g[c] : 0.f;
    }
    int stride = gridDim.x * LN_WARPS;
    for (int row = blockIdx.x * LN_WARPS + warp; row < M; row += stride) {
        const Act* dur = du + (int64_t)row * C;
        const float* xr = x + (int64_t)row * C;
        float m = mu[row], rs = rstd_in[row];
        float dy[EPL], xh[EPL];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; j++) {
            int c = lane + 32 * j;
            if (c < C) {
                dy[j] = to_f(dur[c]);
                xh[j] = (xr[c] - m) * rs;
            } else {
                dy[j] = 0.f;
                xh[j] = 0.f;
            }
            float dxh = dy[j] * gv[j];
            s1 += dxh;
            s2 += dxh * xh[j];
            pg[j] += dy[j] * xh[j];
            pb[j] += dy[j];
        }
        s1 = warp_sum(s1) / (float)C;
        s2 = warp_sum(s2) / (float)C;
        float* dr = dres + (int64_t)row * C;
        Act* da = dres_act + (int64_t)row * C;
#pragma unroll
        for (int j = 0; j < EPL; j++) {
            int c = lane + 32 * j;
            if (c < C) {
                float dx = rs * (dy[j] * gv[j] - s1 - xh[j] * s2);
                float o = accumulate ? dr[c] + dx : dx;
                dr[c] = o;
                da[c] = from_f<Act>(o);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        if (c < C) {
            sm[(warp * 2 + 0) * C + c] = pg[j];
            sm[(warp * 2 + 1) * C + c] = pb[j];
        }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        float a = 0.f, bb = 0.f;
        for (int w = 0; w < LN_WARPS; w++) {
            a += sm[(w * 2 + 0) * C + c];
            bb += sm[(w * 2 + 1) * C + c];
        }
        partial[(int64_t)blockIdx.x * 2 * C + c] = a;
        partial[(int64_t)blockIdx.x * 2 * C + C + c] = bb;
    }
}

__global__ void ln_param_reduce(const float* __restrict__ partial, int nblocks, int C,
                                float* __restrict__ dg, float* __restrict__ db) {
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float a = 0.f, b = 0.f;
    for (int k = 0; k < nblocks; k++) {
        a += partial[(int64_t)k * 2 * C + c];
        b += partial[(int64_t)k * 2 * C + C + c];
    }
    dg[c] += a;
    db[c] += b;
}

static int ln_bwd_blocks(int M) {
    int want = (M + LN_WARPS - 1) / LN_WARPS;
    int cap = num_sms() * 4;
    return want < cap ? want : cap;
}

size_t layernorm_bwd_partial_floats(int M, int C) { return (size_t)ln_bwd_blocks(M) * 2 * C; }

#define LN_DISPATCH(EPLV, CALL)                       \
    if (epl <= EPLV) { CALL(EPLV); return cudaGetLastError(); }

template <typename Act>
cudaError_t layernorm_fwd(const float* x, const float* g, const float* b, Act* u, float* mu,
                          float* rstd, int M, int C, cudaStream_t s) {
    int epl = (C + 31) / 32;
    int blocks = (M + LN_WARPS - 1) / LN_WARPS;
#define LNF(E) ln_fwd_kernel<Act, E><<<blocks, LN_WARPS * 32, 0, s>>>(x, g, b, u, mu, rstd, M, C)
    LN_DISPATCH(2, LNF)
    LN_DISPATCH(4, LNF)
    LN_DISPATCH(8, LNF)
    LN_DISPATCH(12, LNF)
    LN_DISPATCH(16, LNF)
    LN_DISPATCH(24, LNF)
    LN_DISPATCH(32, LNF)
    LN_DISPATCH(48, LNF)
    LN_DISPATCH(64, LNF)
#undef LNF
    return cudaErrorInvalidValue;
}

template <typename Act>
cudaError_t layernorm_bwd(const Act* du, const float* x, const float* g, const float* mu,
                          const float* rstd, float* dres, Act* dres_act, bool accumulate, float* dg,
                          float* db, int M, int C, float* partial, cudaStream_t s) {
    int epl = (C + 31) / 32;
    int blocks = ln_bwd_blocks(M);
    size_t smem = (size_t)LN_WARPS * 2 * C * sizeof(float);
    cudaError_t e = cudaErrorInvalidValue;
#define LNB(E)                                                                                  \
    do {                                                                                        \
        cudaFuncSetAttribute(ln_bwd_kernel<Act, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             (int)smem);                                                        \
        ln_bwd_kernel<Act, E><<<blocks, LN_WARPS * 32, smem, s>>>(                              \
            du, x, g, mu, rstd, dres, dres_act, accumulate ? 1 : 0, partial, M, C);             \
        e = cudaGetLastError();                                                                 \
    } while (0)
    if (epl <= 2) LNB(2);
    else if (epl <= 4) LNB(4);
    else if (epl <= 8) LNB(8);
    else if (epl <= 12) LNB(12);
    else if (epl <= 16) LNB(16);
    else if (epl <= 24) LNB(24);
    else if (epl <= 32) LNB(32);
    else if (epl <= 48) LNB(48);
    else if (epl <= 64) LNB(64);
#undef LNB
    if (e != cudaSuccess) return e;
    ln_param_reduce<<<(C + 255) / 256, 256, 0, s>>>(partial, blocks, C, dg, db);
    return cudaGetLastError();
}

template cudaError_t layernorm_fwd<float>(const float*, const float*, const float*, float*, float*,
                                          float*, int, int, cudaStream_t);
template cudaError_t layernorm_fwd<bf16>(const float*, const float*, const float*, bf16*, float*,
                                         float*, int, int, cudaStream_t);
template cudaError_t layernorm_bwd<float>(const float*, const float*, const float*, const float*,
                                          const float*, float*, float*, bool, float*, float*, int,
                                          int, float*, cudaStream_t);
template cudaError_t layernorm_bwd<bf16>(const bf16*, const float*, const float*, const float*,
                                         const float*, float*, bf16*, bool, float*, float*, int,
                                         int, float*, cudaStream_t);

}  // namespace k
