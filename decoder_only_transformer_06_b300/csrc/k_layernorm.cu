// LayerNorm forward and backward (nn.LayerNorm semantics, eps = 1e-5, biased
// variance; "Build GPT from scratch" forty-line model, nanoGPT guide Deep
// dive 1). One warp per row; lane l owns columns l, l+32, ... so the loads of
// a warp are contiguous. fp32 math throughout; the normalised output is
// written in the activation type (bf16 operand of the next GEMM, or fp32).
#include "common.cuh"

namespace k {

static constexpr float LN_EPS = 1e-5f;
static constexpr int LN_WARPS = 8;

// With y != nullptr the row is first formed as x + y (the residual add of
// the preceding block branch, whose Linear output y is in the activation
// type) and written to x_out, the residual stream the backward reads.
template <typename Act, int EPL>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_fwd_kernel(const float* __restrict__ x, const Act* __restrict__ y, float* __restrict__ x_out,
              const float* __restrict__ g, const float* __restrict__ b, Act* __restrict__ u,
              float* __restrict__ mu_out, float* __restrict__ rstd_out, int M, int C) {
    pdl_wait();
    pdl_trigger();
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
        if (y && c < C) {
            v[j] += to_f(y[(int64_t)row * C + c]);
            x_out[(int64_t)row * C + c] = v[j];
        }
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
              Act* __restrict__ dres_act, int accumulate, int want_sum,
              float* __restrict__ partial, int M, int C) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float sm[];   // [LN_WARPS][3][C]
    int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float pg[EPL], pb[EPL], ps[EPL], gv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        pg[j] = 0.f;
        pb[j] = 0.f;
        ps[j] = 0.f;
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
                ps[j] += o;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < EPL; j++) {
        int c = lane + 32 * j;
        if (c < C) {
            sm[(warp * 3 + 0) * C + c] = pg[j];
            sm[(warp * 3 + 1) * C + c] = pb[j];
            sm[(warp * 3 + 2) * C + c] = ps[j];
        }
    }
    __syncthreads();
    const int np = want_sum ? 3 : 2;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        for (int k = 0; k < np; k++) {
            float a = 0.f;
            for (int w = 0; w < LN_WARPS; w++) a += sm[(w * 3 + k) * C + c];
            partial[((int64_t)blockIdx.x * 3 + k) * C + c] = a;
        }
    }
}


// ---------------------------------------------------------------- vector path
// C a multiple of 128: lane l owns float4 columns l, l+32, ... (each warp load
// is 512 contiguous bytes); the activation is written 4 values at a time.
template <typename Act>
__device__ __forceinline__ void store4(Act* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) { *(float4*)dst = v; }
template <>
__device__ __forceinline__ void store4<bf16>(bf16* dst, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *(uint32_t*)&lo;
    o.y = *(uint32_t*)&hi;
    *(uint2*)dst = o;
}
template <typename Act>
__device__ __forceinline__ float4 load4(const Act* src);
template <>
__device__ __forceinline__ float4 load4<float>(const float* src) { return *(const float4*)src; }
template <>
__device__ __forceinline__ float4 load4<bf16>(const bf16* src) {
    uint2 w = *(const uint2*)src;
    float2 a = __bfloat1622float2(*(const __nv_bfloat162*)&w.x);
    float2 b = __bfloat1622float2(*(const __nv_bfloat162*)&w.y);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <typename Act, int V4>
__global__ void __launch_bounds__(LN_WARPS * 32)
ln_fwd_vec(const float* __restrict__ x, const Act* __restrict__ y, float* __restrict__ x_out,
           const float* __restrict__ g, const float* __restrict__ b, Act* __restrict__ u,
           float* __restrict__ mu_out, float* __restrict__ rstd_out, int M, int C) {
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x * LN_WARPS + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= M) return;
    const float4* xr = (const float4*)(x + (int64_t)row * C);
    float4 v[V4];
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < V4; j++) v[j] = xr[lane + 32 * j];
    if (y) {
        const Act* yr = y + (int64_t)row * C;
        float4* xo = (float4*)(x_out + (int64_t)row * C);
#pragma unroll
        for (int j = 0; j < V4; j++) {
            const float4 a = load4<Act>(yr + 4 * (lane + 32 * j));
            v[j].x += a.x; v[j].y += a.y; v[j].z += a.z; v[j].w += a.w;
            xo[lane + 32 * j] = v[j];
        }
    }
#pragma unroll
    for (int j = 0; j < V4; j++) s += (v[j].x + v[j].y) + (v[j].z + v[j].w);
    const float mean = warp_sum(s) / (float)C;
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < V4; j++) {
        float a = v[j].x - mean, bq = v[j].y - mean, c = v[j].z - mean, d = v[j].w - mean;
        q += (a * a + bq * bq) + (c * c + d * d);
    }
    const float rstd = 1.0f / sqrtf(warp_sum(q) / (float)C + LN_EPS);
    Act* ur = u + (int64_t)row * C;
#pragma unroll
    for (int j = 0; j < V4; j++) {
        const int c4 = lane + 32 * j;
        const float4 gg = __ldg((const float4*)g + c4), bb = __ldg((const float4*)b + c4);
        float4 y = make_float4((v[j].x - mean) * rstd * gg.x + bb.x, (v[j].y - mean) * rstd * gg.y + bb.y,
                               (v[j].z - mean) * rstd * gg.z + bb.z, (v[j].w - mean) * rstd * gg.w + bb.w);
        store4<Act>(ur + 4 * c4, y);
    }
    if (lane == 0) {
        mu_out[row] = mean;
        rstd_out[row] = rstd;
    }
}

template <typename Act, int V4>
__global__ void __launch_bounds__(LN_WARPS * 32, 2)
ln_bwd_vec(const Act* __restrict__ du, const float* __restrict__ x, const float* __restrict__ g,
           const float* __restrict__ mu, const float* __restrict__ rstd_in,
           float* __restrict__ dres, Act* __restrict__ dres_act, int accumulate, int want_sum,
           float* __restrict__ partial, int M, int C) {
    pdl_wait();
    pdl_trigger();
    // each warp accumulates its partials (dg, db and, if asked, the column sum
    // of the new dres) in its own slice of shared memory ([LN_WARPS][3][C]);
    // slices are combined in warp order at the end
    extern __shared__ float sm[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float4* pgs = (float4*)&sm[(warp * 3 + 0) * C];
    float4* pbs = (float4*)&sm[(warp * 3 + 1) * C];
    float4* pss = (float4*)&sm[(warp * 3 + 2) * C];
#pragma unroll
    for (int j = 0; j < V4; j++) {
        pgs[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
        pbs[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
        pss[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float invC = 1.0f / (float)C;
    const int stride = gridDim.x * LN_WARPS;
    for (int row = blockIdx.x * LN_WARPS + warp; row < M; row += stride) {
        const Act* dur = du + (int64_t)row * C;
        const float4* xr = (const float4*)(x + (int64_t)row * C);
        float4* dr = (float4*)(dres + (int64_t)row * C);
        const float m = mu[row], rs = rstd_in[row];
        float4 dy[V4], xh[V4], prev[V4];
#pragma unroll
        for (int j = 0; j < V4; j++) {
            const int c4 = lane + 32 * j;
            dy[j] = load4<Act>(dur + 4 * c4);
            xh[j] = xr[c4];
            prev[j] = accumulate ? dr[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int j = 0; j < V4; j++) {
            const int c4 = lane + 32 * j;
            xh[j] = make_float4((xh[j].x - m) * rs, (xh[j].y - m) * rs, (xh[j].z - m) * rs, (xh[j].w - m) * rs);
            const float4 gg = __ldg((const float4*)g + c4);
            float a = dy[j].x * gg.x, bq = dy[j].y * gg.y, c = dy[j].z * gg.z, d = dy[j].w * gg.w;
            s1 += (a + bq) + (c + d);
            s2 += (a * xh[j].x + bq * xh[j].y) + (c * xh[j].z + d * xh[j].w);
        }
        s1 = warp_sum(s1) * invC;
        s2 = warp_sum(s2) * invC;
        Act* da = dres_act + (int64_t)row * C;
#pragma unroll
        for (int j = 0; j < V4; j++) {
            const int c4 = lane + 32 * j;
            const float4 gg = __ldg((const float4*)g + c4);
            float4 o = make_float4(prev[j].x + rs * (dy[j].x * gg.x - s1 - xh[j].x * s2),
                                   prev[j].y + rs * (dy[j].y * gg.y - s1 - xh[j].y * s2),
                                   prev[j].z + rs * (dy[j].z * gg.z - s1 - xh[j].z * s2),
                                   prev[j].w + rs * (dy[j].w * gg.w - s1 - xh[j].w * s2));
            dr[c4] = o;
            if ((const void*)da != (const void*)dr) store4<Act>(da + 4 * c4, o);
            float4 pg = pgs[c4], pb = pbs[c4];
            pg.x += dy[j].x * xh[j].x; pg.y += dy[j].y * xh[j].y;
            pg.z += dy[j].z * xh[j].z; pg.w += dy[j].w * xh[j].w;
            pb.x += dy[j].x; pb.y += dy[j].y; pb.z += dy[j].z; pb.w += dy[j].w;
            pgs[c4] = pg;
            pbs[c4] = pb;
            if (want_sum) {
                float4 ps = pss[c4];
                ps.x += o.x; ps.y += o.y; ps.z += o.z; ps.w += o.w;
                pss[c4] = ps;
            }
        }
    }
    __syncthreads();
    const int np = want_sum ? 3 : 2;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        for (int k = 0; k < np; k++) {
            float a = 0.f;
            for (int w = 0; w < LN_WARPS; w++) a += sm[(w * 3 + k) * C + c];
            partial[((int64_t)blockIdx.x * 3 + k) * C + c] = a;
        }
    }
}

// Second stage of the parameter-gradient reduction: block = 32 columns x 32
// slices of the partial rows; slice s sums partial rows s, s+32, ... and the
// slice sums are combined in slice order (fixed order: deterministic).
static constexpr int LNR_SLICES = 32;
__global__ void __launch_bounds__(32 * LNR_SLICES)
ln_param_reduce(const float* __restrict__ partial, int nblocks, int C, float* __restrict__ dg,
                float* __restrict__ db, float* __restrict__ dsum) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sm[3][LNR_SLICES][33];
    const int cx = threadIdx.x & 31, sl = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + cx;
    float a = 0.f, b = 0.f, t = 0.f;
    if (c < C) {
#pragma unroll 4
        for (int k = sl; k < nblocks; k += LNR_SLICES) {
            a += partial[((int64_t)k * 3 + 0) * C + c];
            b += partial[((int64_t)k * 3 + 1) * C + c];
            if (dsum) t += partial[((int64_t)k * 3 + 2) * C + c];
        }
    }
    sm[0][sl][cx] = a;
    sm[1][sl][cx] = b;
    sm[2][sl][cx] = t;
    __syncthreads();
    if (sl < 3 && c < C) {
        float acc = 0.f;
        for (int k = 0; k < LNR_SLICES; k++) acc += sm[sl][k][cx];
        float* dst = sl == 0 ? dg : (sl == 1 ? db : dsum);
        if (dst) dst[c] += acc;
    }
}

static int ln_bwd_blocks(int M) {
    int want = (M + LN_WARPS - 1) / LN_WARPS;
    int cap = num_sms() * 2;
    return want < cap ? want : cap;
}

size_t layernorm_bwd_partial_floats(int M, int C) { return (size_t)ln_bwd_blocks(M) * 3 * C; }

#define LN_DISPATCH(EPLV, CALL)                       \
    if (epl <= EPLV) { CALL(EPLV); return cudaGetLastError(); }

template <typename Act>
cudaError_t layernorm_fwd(const float* x, const Act* y, float* x_out, const float* g,
                          const float* b, Act* u, float* mu, float* rstd, int M, int C,
                          cudaStream_t s) {
    if (y && !x_out) return cudaErrorInvalidValue;
    int epl = (C + 31) / 32;
    int blocks = (M + LN_WARPS - 1) / LN_WARPS;
    if (C % 128 == 0 && C <= 2048) {
        switch (C / 128) {
#define LNV(V)                                                                                      \
    case V:                                                                                         \
        (void)pdl_launch(ln_fwd_vec<Act, V>, blocks, LN_WARPS * 32, 0, s, x, y, x_out, g, b, u, mu, rstd, M, C);            \
        return cudaGetLastError();
            LNV(1) LNV(2) LNV(3) LNV(4) LNV(5) LNV(6) LNV(7) LNV(8)
            LNV(9) LNV(10) LNV(11) LNV(12) LNV(13) LNV(14) LNV(15) LNV(16)
#undef LNV
        }
    }
#define LNF(E) (void)pdl_launch(ln_fwd_kernel<Act, E>, blocks, LN_WARPS * 32, 0, s, x, y, x_out, g, b, u, mu, rstd, M, C)
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

cudaError_t layernorm_bwd_params(const float* partial, int M, int C, float* dg, float* db, float* dsum,
                                 cudaStream_t s) {
    (void)pdl_launch(ln_param_reduce, (C + 31) / 32, 32 * LNR_SLICES, 0, s, partial, ln_bwd_blocks(M), C, dg, db, dsum);
    return cudaGetLastError();
}

template <typename Act>
cudaError_t layernorm_bwd_rows(const Act* du, const float* x, const float* g, const float* mu,
                               const float* rstd, float* dres, Act* dres_act, bool accumulate,
                               bool want_dsum, int M, int C, float* partial, cudaStream_t s) {
    int epl = (C + 31) / 32;
    int blocks = ln_bwd_blocks(M);
    size_t smem = (size_t)LN_WARPS * 3 * C * sizeof(float);
    const int want_sum = want_dsum ? 1 : 0;
    cudaError_t e = cudaErrorInvalidValue;
    if (C % 128 == 0 && C <= 1024) {
        switch (C / 128) {
#define LBV(V)                                                                                     \
    case V:                                                                                        \
        cudaFuncSetAttribute(ln_bwd_vec<Act, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                             (int)smem);                                                           \
        (void)pdl_launch(ln_bwd_vec<Act, V>, blocks, LN_WARPS * 32, smem, s, du, x, g, mu, rstd, dres, dres_act, \
                                                               accumulate ? 1 : 0, want_sum,       \
                                                               partial, M, C);                     \
        e = cudaGetLastError();                                                                    \
        break;
            LBV(1) LBV(2) LBV(3) LBV(4) LBV(5) LBV(6) LBV(7) LBV(8)
#undef LBV
        }
        return e;
    }
#define LNB(E)                                                                                  \
    do {                                                                                        \
        cudaFuncSetAttribute(ln_bwd_kernel<Act, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             (int)smem);                                                        \
        (void)pdl_launch(ln_bwd_kernel<Act, E>, blocks, LN_WARPS * 32, smem, s,                               \
            du, x, g, mu, rstd, dres, dres_act, accumulate ? 1 : 0, want_sum, partial, M, C);   \
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
    return e;
}

template <typename Act>
cudaError_t layernorm_bwd(const Act* du, const float* x, const float* g, const float* mu,
                          const float* rstd, float* dres, Act* dres_act, bool accumulate, float* dg,
                          float* db, float* dsum, int M, int C, float* partial, cudaStream_t s) {
    cudaError_t e = layernorm_bwd_rows<Act>(du, x, g, mu, rstd, dres, dres_act, accumulate,
                                            dsum != nullptr, M, C, partial, s);
    if (e != cudaSuccess) return e;
    return layernorm_bwd_params(partial, M, C, dg, db, dsum, s);
}

template cudaError_t layernorm_fwd<float>(const float*, const float*, float*, const float*,
                                          const float*, float*, float*, float*, int, int,
                                          cudaStream_t);
template cudaError_t layernorm_fwd<bf16>(const float*, const bf16*, float*, const float*,
                                         const float*, bf16*, float*, float*, int, int,
                                         cudaStream_t);
template cudaError_t layernorm_bwd_rows<float>(const float*, const float*, const float*, const float*,
                                               const float*, float*, float*, bool, bool, int, int,
                                               float*, cudaStream_t);
template cudaError_t layernorm_bwd_rows<bf16>(const bf16*, const float*, const float*, const float*,
                                              const float*, float*, bf16*, bool, bool, int, int,
                                              float*, cudaStream_t);
template cudaError_t layernorm_bwd<float>(const float*, const float*, const float*, const float*,
                                          const float*, float*, float*, bool, float*, float*,
                                          float*, int, int, float*, cudaStream_t);
template cudaError_t layernorm_bwd<bf16>(const bf16*, const float*, const float*, const float*,
                                         const float*, float*, bf16*, bool, float*, float*, float*,
                                         int, int, float*, cudaStream_t);

}  // namespace k
