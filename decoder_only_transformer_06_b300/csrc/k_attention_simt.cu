// Causal attention in fp32 for the fp32-math mode (no tensor cores).
// Semantics are the manual path of nanoGPT's CausalSelfAttention (nanoGPT
// guide Deep dive 1): S = q k^T / sqrt(hs), j > i masked to -inf before the
// softmax, o = softmax(S) v. Computed flash-style with an online softmax, so
// the T x T matrix never exists ("Let's reproduce GPT-2" 02:00:18).
//
// Layout: qkv [B*T, 3C] row-major, q at columns [0,C), k at [C,2C), v at
// [2C,3C); head h uses columns h*hs..h*hs+hs-1 of each. out [B*T, C];
// lse [B, H, T] natural-log normaliser of each softmax row.
//
// One warp per query row (forward, dQ) or key row (dK/dV); within a warp
// lanes take 32 consecutive keys (or queries) at a time, and lane l owns the
// output columns l, l+32, ... The backward is deterministic: dQ and dK/dV
// are separate passes with no atomics.
#include "common.cuh"

namespace k {

static constexpr int AW = 8;        // warps per CTA
static constexpr int HS_MAX = 128;

__device__ __forceinline__ float dot_row(const float* a, const float* __restrict__ b, int hs) {
    float s = 0.f;
    for (int c = 0; c < hs; c++) s = fmaf(a[c], b[c], s);
    return s;
}

__global__ void __launch_bounds__(AW * 32)
attn_fwd_f32_kernel(const float* __restrict__ qkv, float* __restrict__ out,
                    float* __restrict__ lse, int B, int T, int H, int hs) {
    pdl_wait();
    pdl_trigger();
    __shared__ float qs[AW][HS_MAX];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t gw = (int64_t)blockIdx.x * AW + warp;
    if (gw >= (int64_t)B * H * T) return;
    const int i = (int)(gw % T);
    const int bh = (int)(gw / T);
    const int h = bh % H, b = bh / H;
    const int C = H * hs;
    const int64_t ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld;
    const float scale = 1.0f / sqrtf((float)hs);
    for (int c = lane; c < hs; c += 32) qs[warp][c] = base[(int64_t)i * ld + h * hs + c];
    __syncwarp();
    float m = -INFINITY, l = 0.f;
    float o[HS_MAX / 32];
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) o[e] = 0.f;
    for (int j0 = 0; j0 <= i; j0 += 32) {
        int j = j0 + lane;
        float s = -INFINITY;
        if (j <= i) s = dot_row(qs[warp], base + (int64_t)j * ld + C + h * hs, hs) * scale;
        float cm = warp_max(s);
        float mn = fmaxf(m, cm);
        float p = (j <= i) ? expf(s - mn) : 0.f;
        float corr = expf(m - mn);
        l = l * corr + warp_sum(p);
        int nj = min(32, i - j0 + 1);
#pragma unroll
        for (int e = 0; e < HS_MAX / 32; e++) o[e] *= corr;
        for (int t = 0; t < nj; t++) {
            float pt = __shfl_sync(0xffffffffu, p, t);
            const float* vr = base + (int64_t)(j0 + t) * ld + 2 * C + h * hs;
#pragma unroll
            for (int e = 0; e < HS_MAX / 32; e++) {
                int c = lane + 32 * e;
                if (c < hs) o[e] = fmaf(pt, vr[c], o[e]);
            }
        }
        m = mn;
    }
    float* orow = out + ((int64_t)b * T + i) * C + h * hs;
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) {
        int c = lane + 32 * e;
        if (c < hs) orow[c] = o[e] / l;
    }
    if (lane == 0) lse[gw] = m + logf(l);
}

// D[b,h,i] = sum_c dout[i, h*hs+c] * out[i, h*hs+c]  (= rowsum(dP * P))
__global__ void attn_bwd_d_f32(const float* __restrict__ out, const float* __restrict__ dout,
                               float* __restrict__ D, int B, int T, int H, int hs) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t gw = (int64_t)blockIdx.x * AW + warp;
    if (gw >= (int64_t)B * H * T) return;
    const int i = (int)(gw % T);
    const int bh = (int)(gw / T);
    const int h = bh % H, b = bh / H;
    const int C = H * hs;
    const int64_t off = ((int64_t)b * T + i) * C + h * hs;
    float s = 0.f;
    for (int c = lane; c < hs; c += 32) s = fmaf(dout[off + c], out[off + c], s);
    s = warp_sum(s);
    if (lane == 0) D[gw] = s;
}

// dQ_i = scale * sum_{j<=i} P_ij (dP_ij - D_i) k_j, dP_ij = dO_i . v_j
__global__ void __launch_bounds__(AW * 32)
attn_bwd_dq_f32(const float* __restrict__ qkv, const float* __restrict__ lse,
                const float* __restrict__ dout, const float* __restrict__ D,
                float* __restrict__ dqkv, int B, int T, int H, int hs) {
    pdl_wait();
    pdl_trigger();
    __shared__ float qs[AW][HS_MAX];
    __shared__ float ds_[AW][HS_MAX];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t gw = (int64_t)blockIdx.x * AW + warp;
    if (gw >= (int64_t)B * H * T) return;
    const int i = (int)(gw % T);
    const int bh = (int)(gw / T);
    const int h = bh % H, b = bh / H;
    const int C = H * hs;
    const int64_t ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld;
    const float scale = 1.0f / sqrtf((float)hs);
    for (int c = lane; c < hs; c += 32) {
        qs[warp][c] = base[(int64_t)i * ld + h * hs + c];
        ds_[warp][c] = dout[((int64_t)b * T + i) * C + h * hs + c];
    }
    __syncwarp();
    const float li = lse[gw], Di = D[gw];
    float dq[HS_MAX / 32];
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) dq[e] = 0.f;
    for (int j0 = 0; j0 <= i; j0 += 32) {
        int j = j0 + lane;
        float ds = 0.f;
        if (j <= i) {
            float s = dot_row(qs[warp], base + (int64_t)j * ld + C + h * hs, hs) * scale;
            float p = expf(s - li);
            float dp = dot_row(ds_[warp], base + (int64_t)j * ld + 2 * C + h * hs, hs);
            ds = p * (dp - Di);
        }
        int nj = min(32, i - j0 + 1);
        for (int t = 0; t < nj; t++) {
            float dt = __shfl_sync(0xffffffffu, ds, t);
            const float* kr = base + (int64_t)(j0 + t) * ld + C + h * hs;
#pragma unroll
            for (int e = 0; e < HS_MAX / 32; e++) {
                int c = lane + 32 * e;
                if (c < hs) dq[e] = fmaf(dt, kr[c], dq[e]);
            }
        }
    }
    float* dqr = dqkv + ((int64_t)b * T + i) * ld + h * hs;
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) {
        int c = lane + 32 * e;
        if (c < hs) dqr[c] = dq[e] * scale;
    }
}

// dV_j = sum_{i>=j} P_ij dO_i ; dK_j = scale * sum_{i>=j} P_ij (dP_ij - D_i) q_i
__global__ void __launch_bounds__(AW * 32)
attn_bwd_dkv_f32(const float* __restrict__ qkv, const float* __restrict__ lse,
                 const float* __restrict__ dout, const float* __restrict__ D,
                 float* __restrict__ dqkv, int B, int T, int H, int hs) {
    pdl_wait();
    pdl_trigger();
    __shared__ float ks[AW][HS_MAX];
    __shared__ float vs[AW][HS_MAX];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t gw = (int64_t)blockIdx.x * AW + warp;
    if (gw >= (int64_t)B * H * T) return;
    const int j = (int)(gw % T);
    const int bh = (int)(gw / T);
    const int h = bh % H, b = bh / H;
    const int C = H * hs;
    const int64_t ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld;
    const float* dbase = dout + (int64_t)b * T * C;
    const float* lrow = lse + (int64_t)bh * T;
    const float* Drow = D + (int64_t)bh * T;
    const float scale = 1.0f / sqrtf((float)hs);
    for (int c = lane; c < hs; c += 32) {
        ks[warp][c] = base[(int64_t)j * ld + C + h * hs + c];
        vs[warp][c] = base[(int64_t)j * ld + 2 * C + h * hs + c];
    }
    __syncwarp();
    float dk[HS_MAX / 32], dv[HS_MAX / 32];
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) { dk[e] = 0.f; dv[e] = 0.f; }
    for (int i0 = j; i0 < T; i0 += 32) {
        int i = i0 + lane;
        float p = 0.f, ds = 0.f;
        if (i < T) {
            float s = dot_row(ks[warp], base + (int64_t)i * ld + h * hs, hs) * scale;
            p = expf(s - lrow[i]);
            float dp = dot_row(vs[warp], dbase + (int64_t)i * C + h * hs, hs);
            ds = p * (dp - Drow[i]);
        }
        int ni = min(32, T - i0);
        for (int t = 0; t < ni; t++) {
            float pt = __shfl_sync(0xffffffffu, p, t);
            float dt = __shfl_sync(0xffffffffu, ds, t);
            const float* qr = base + (int64_t)(i0 + t) * ld + h * hs;
            const float* dor = dbase + (int64_t)(i0 + t) * C + h * hs;
#pragma unroll
            for (int e = 0; e < HS_MAX / 32; e++) {
                int c = lane + 32 * e;
                if (c < hs) {
                    dv[e] = fmaf(pt, dor[c], dv[e]);
                    dk[e] = fmaf(dt, qr[c], dk[e]);
                }
            }
        }
    }
    float* row = dqkv + ((int64_t)b * T + j) * ld + h * hs;
#pragma unroll
    for (int e = 0; e < HS_MAX / 32; e++) {
        int c = lane + 32 * e;
        if (c < hs) {
            row[C + c] = dk[e] * scale;
            row[2 * C + c] = dv[e];
        }
    }
}

cudaError_t attention_fwd_f32(const float* qkv, float* out, float* lse, int B, int T, int H, int hs,
                              cudaStream_t s) {
    if (hs > HS_MAX) return cudaErrorInvalidValue;
    int64_t rows = (int64_t)B * H * T;
    (void)pdl_launch(attn_fwd_f32_kernel, (unsigned)((rows + AW - 1) / AW), AW * 32, 0, s, qkv, out, lse, B, T,
                                                                           H, hs);
    return cudaGetLastError();
}

cudaError_t attention_bwd_f32(const float* qkv, const float* out, const float* lse,
                              const float* dout, float* dqkv, float* Dbuf, int B, int T, int H,
                              int hs, cudaStream_t s) {
    if (hs > HS_MAX) return cudaErrorInvalidValue;
    int64_t rows = (int64_t)B * H * T;
    unsigned g = (unsigned)((rows + AW - 1) / AW);
    (void)pdl_launch(attn_bwd_d_f32, g, AW * 32, 0, s, out, dout, Dbuf, B, T, H, hs);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(attn_bwd_dq_f32, g, AW * 32, 0, s, qkv, lse, dout, Dbuf, dqkv, B, T, H, hs);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(attn_bwd_dkv_f32, g, AW * 32, 0, s, qkv, lse, dout, Dbuf, dqkv, B, T, H, hs);
    return cudaGetLastError();
}

}  // namespace k
