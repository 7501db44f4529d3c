// Kernels of one decoding step with the key/value cache: the forward of a
// single new position p per sequence, whose query attends to the keys and
// values of positions 0..p that earlier steps left in the layer's qkv buffer.
// The pages' generation loop ("Let's reproduce GPT-2", 00:37:02 the sampling
// loop; nanoGPT guide, sample.py) recomputes the whole context for every new
// token; with absolute position embeddings the cached keys and values of
// positions 0..p-1 are exactly what that recomputation would produce, so the
// step gives the same logits with work proportional to one position.
#include "common.cuh"

namespace k {

namespace {

constexpr int DEC_THREADS = 128;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float& d, float x) { d = x; }
__device__ __forceinline__ void from_f(bf16& d, float x) { d = __float2bfloat16_rn(x); }

// x[b] = wte[tok[b]] + wpe[p] (fp32 rows of width C); an id outside [0, V) is
// clamped and flagged, as the training forward's input check does.
__global__ void embed_rows_kernel(const int32_t* __restrict__ tok, const float* __restrict__ wte,
                                  const float* __restrict__ wpe, float* __restrict__ x, int p, int C, int V,
                                  DevState* st) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    int t = tok[b];
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0 && st) atomicOr(&st->err, ERR_TOKEN_RANGE);
        t = t < 0 ? 0 : V - 1;
    }
    for (int c = threadIdx.x; c < C; c += blockDim.x)
        x[(int64_t)b * C + c] = wte[(int64_t)t * C + c] + wpe[(int64_t)p * C + c];
}

// Block-wide reductions over DEC_THREADS threads in a fixed order.
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < DEC_THREADS / 32; i++) r = fmaxf(r, red[i]);
    return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < DEC_THREADS / 32; i++) r += red[i];
    return r;
}

// Split decoding attention: the keys 0..p of a (b, h) are cut into spans of
// DEC_SPAN; CTA (span, b*H + h) computes, for its span, the maximum m of the
// scaled scores q.k_j / sqrt(hs), l = sum_j exp(s_j - m) and
// o = sum_j exp(s_j - m) v_j, and the combine kernel merges the spans of a
// head exactly: M = max m_i, o = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i
// (the online-softmax identity, in span order). Warp w takes the keys
// w, w + 4, ... of the span; lane d handles dimensions d, d + 32, ... (loads of
// one key row are coalesced across the warp).
constexpr int DEC_SPAN = 64;

template <typename Act>
__global__ void __launch_bounds__(DEC_THREADS)
attention_decode_span_kernel(const Act* __restrict__ qkv, float* __restrict__ part, int T, int H, int hs, int p,
                             int nspan) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sw[DEC_SPAN];
    __shared__ float so[DEC_THREADS / 32][128];
    __shared__ float red[DEC_THREADS / 32];
    const int span = blockIdx.x, bh = blockIdx.y, b = bh / H, h = bh % H, C = H * hs;
    const int64_t row = 3ll * C;
    const Act* base = qkv + (int64_t)b * T * row;
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int j0 = span * DEC_SPAN, j1 = min(p + 1, j0 + DEC_SPAN);
    const int nd = (hs + 31) / 32;                 // dimensions per lane (hs <= 128)
    float q[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int d = lane + 32 * i;
        q[i] = (i < nd && d < hs) ? to_f(base[(int64_t)p * row + h * hs + d]) : 0.f;
    }
    const float scale = 1.0f / sqrtf((float)hs);
    float lmax = -INFINITY;
    // keys in groups of DEC_KG per warp, their loads issued before any reduction
    constexpr int DEC_KG = 4;
    for (int jb = j0 + w; jb < j1; jb += DEC_KG * (DEC_THREADS / 32)) {
        float s[DEC_KG];
#pragma unroll
        for (int u = 0; u < DEC_KG; u++) {
            const int j = jb + u * (DEC_THREADS / 32);
            s[u] = 0.f;
            if (j < j1) {
                const Act* kr = base + (int64_t)j * row + C + h * hs;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int d = lane + 32 * i;
                    if (i < nd && d < hs) s[u] = fmaf(q[i], to_f(kr[d]), s[u]);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < DEC_KG; u++) s[u] += __shfl_xor_sync(0xffffffffu, s[u], o);
#pragma unroll
        for (int u = 0; u < DEC_KG; u++) {
            const int j = jb + u * (DEC_THREADS / 32);
            if (j < j1) {
                const float sc = s[u] * scale;
                if (lane == 0) sw[j - j0] = sc;
                lmax = fmaxf(lmax, sc);
            }
        }
    }
    const float m = block_max(lmax, red);          // barriers: every score is in sw
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float lsum = 0.f;
#pragma unroll 4
    for (int j = j0 + w; j < j1; j += DEC_THREADS / 32) {
        const float e = expf(sw[j - j0] - m);
        lsum += e;
        const Act* vr = base + (int64_t)j * row + 2 * C + h * hs;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int d = lane + 32 * i;
            if (i < nd && d < hs) acc[i] = fmaf(e, to_f(vr[d]), acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) so[w][lane + 32 * i] = acc[i];
    const float l = block_sum(lane == 0 ? lsum : 0.f, red);   // ends with a barrier
    float* out = part + ((int64_t)bh * nspan + span) * (hs + 2);
    for (int d = threadIdx.x; d < hs; d += DEC_THREADS) {
        float o = 0.f;
#pragma unroll
        for (int ww = 0; ww < DEC_THREADS / 32; ww++) o += so[ww][d];
        out[2 + d] = o;
    }
    if (threadIdx.x == 0) {
        out[0] = m;
        out[1] = l;
    }
}

// One CTA per (b, h): merge the spans in order into out [B, C].
template <typename Act>
__global__ void __launch_bounds__(DEC_THREADS)
attention_decode_combine_kernel(const float* __restrict__ part, Act* __restrict__ out, int H, int hs, int nspan) {
    pdl_wait();
    pdl_trigger();
    const int bh = blockIdx.x, b = bh / H, h = bh % H, C = H * hs;
    const float* pp = part + (int64_t)bh * nspan * (hs + 2);
    float M = -INFINITY;
    for (int i = 0; i < nspan; i++) M = fmaxf(M, pp[(int64_t)i * (hs + 2)]);
    for (int d = threadIdx.x; d < hs; d += DEC_THREADS) {
        float o = 0.f, l = 0.f;
        for (int i = 0; i < nspan; i++) {
            const float* q = pp + (int64_t)i * (hs + 2);
            const float f = expf(q[0] - M);
            l = fmaf(f, q[1], l);
            o = fmaf(f, q[2 + d], o);
        }
        from_f(out[(int64_t)b * C + h * hs + d], o / l);
    }
}

}  // namespace

cudaError_t embed_rows(const int32_t* tok, const float* wte, const float* wpe, float* x, int B, int p, int C,
                       int V, DevState* st, cudaStream_t s) {
    if (B < 1 || C < 1 || p < 0) return cudaErrorInvalidValue;
    (void)pdl_launch(embed_rows_kernel, B, 256, 0, s, tok, wte, wpe, x, p, C, V, st);
    return cudaGetLastError();
}

size_t attention_decode_workspace_floats(int B, int T, int H, int hs) {
    return (size_t)B * H * ((T + DEC_SPAN - 1) / DEC_SPAN) * (hs + 2);
}

template <typename Act>
cudaError_t attention_decode(const Act* qkv, Act* out, float* part, int B, int T, int H, int hs, int p,
                             cudaStream_t s) {
    if (B < 1 || H < 1 || hs < 1 || hs > 128 || p < 0 || p >= T || !part) return cudaErrorInvalidValue;
    const int nspan = (p + 1 + DEC_SPAN - 1) / DEC_SPAN;
    (void)pdl_launch(attention_decode_span_kernel<Act>, dim3(nspan, B * H), DEC_THREADS, 0, s, qkv, part, T, H, hs, p, nspan);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(attention_decode_combine_kernel<Act>, B * H, DEC_THREADS, 0, s, part, out, H, hs, nspan);
    return cudaGetLastError();
}

template cudaError_t attention_decode<float>(const float*, float*, float*, int, int, int, int, int, cudaStream_t);
template cudaError_t attention_decode<bf16>(const bf16*, bf16*, float*, int, int, int, int, int, cudaStream_t);

}  // namespace k
