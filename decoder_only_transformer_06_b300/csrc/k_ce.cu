// Fused softmax cross-entropy forward + backward over the padded vocabulary
// (F.cross_entropy with ignore_index = -1, nanoGPT guide Part IV Stage 4;
// vocabulary padded 50257 -> 50304, "Let's reproduce GPT-2" 02:06:54).
//
// One CTA per row. The row (Vp values) is loaded once into registers with
// 16-byte loads, max and sum-of-exp are block-reduced over the real columns
// j < V only (pad columns are masked), then d loss / d z =
// (softmax - onehot(y)) / (n_valid * accum) is written over the logits in
// place (0 on pad columns and on ignored rows). HBM traffic: one read and one
// write of the logits. Math in fp32.
#include "common.cuh"

namespace k {

static constexpr int CE_THREADS = 256;

template <typename Act>
struct Vec16;
template <>
struct Vec16<bf16> {
    static constexpr int N = 8;
};
template <>
struct Vec16<float> {
    static constexpr int N = 4;
};

template <typename Act>
__device__ __forceinline__ void unpack16(const uint4& r, float* f) {
    if constexpr (sizeof(Act) == 2) {
        const __nv_bfloat162* h = (const __nv_bfloat162*)&r;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            float2 t = __bfloat1622float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    } else {
        const float* p = (const float*)&r;
#pragma unroll
        for (int i = 0; i < 4; i++) f[i] = p[i];
    }
}

template <typename Act>
__device__ __forceinline__ uint4 pack16(const float* f) {
    uint4 r;
    if constexpr (sizeof(Act) == 2) {
        __nv_bfloat162* h = (__nv_bfloat162*)&r;
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    } else {
        float* p = (float*)&r;
#pragma unroll
        for (int i = 0; i < 4; i++) p[i] = f[i];
    }
    return r;
}

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* sm) {
    v = is_max ? warp_max(v) : warp_sum(v);
    int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) sm[w] = v;
    __syncthreads();
    float r = sm[0];
    for (int i = 1; i < CE_THREADS / 32; i++) r = is_max ? fmaxf(r, sm[i]) : r + sm[i];
    return r;
}

template <typename Act, int NCH>
__global__ void __launch_bounds__(CE_THREADS)
ce_kernel(Act* __restrict__ logits, const int32_t* __restrict__ tgt, float* __restrict__ row_loss,
          int V, int Vp, const DevState* __restrict__ st) {
    constexpr int VEC = Vec16<Act>::N;
    __shared__ float sm[CE_THREADS / 32];
    const int row = blockIdx.x;
    Act* z = logits + (int64_t)row * Vp;
    const int nvec = Vp / VEC;
    int y = tgt[row];
    const bool ignore = (y == -1);
    y = (y < 0 || y >= V) ? 0 : y;
    const float zy = to_f(z[y]);
    uint4 r[NCH];
#pragma unroll
    for (int c = 0; c < NCH; c++) {
        int vi = c * CE_THREADS + threadIdx.x;
        if (vi < nvec) r[c] = ((const uint4*)z)[vi];
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < NCH; c++) {
        int vi = c * CE_THREADS + threadIdx.x;
        if (vi < nvec) {
            float f[VEC];
            unpack16<Act>(r[c], f);
#pragma unroll
            for (int e = 0; e < VEC; e++)
                if (vi * VEC + e < V) mx = fmaxf(mx, f[e]);
        }
    }
    mx = block_reduce(mx, true, sm);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; c++) {
        int vi = c * CE_THREADS + threadIdx.x;
        if (vi < nvec) {
            float f[VEC];
            unpack16<Act>(r[c], f);
#pragma unroll
            for (int e = 0; e < VEC; e++)
                if (vi * VEC + e < V) sum += __expf(f[e] - mx);
        }
    }
    sum = block_reduce(sum, false, sm);
    const float lse = mx + logf(sum);
    const float scale = ignore ? 0.f : st->inv_count;
#pragma unroll
    for (int c = 0; c < NCH; c++) {
        int vi = c * CE_THREADS + threadIdx.x;
        if (vi < nvec) {
            float f[VEC];
            unpack16<Act>(r[c], f);
#pragma unroll
            for (int e = 0; e < VEC; e++) {
                int j = vi * VEC + e;
                float d = 0.f;
                if (j < V) {
                    float p = __expf(f[e] - lse);
                    d = (p - (j == y ? 1.f : 0.f)) * scale;
                }
                f[e] = d;
            }
            ((uint4*)z)[vi] = pack16<Act>(f);
        }
    }
    if (threadIdx.x == 0) row_loss[row] = ignore ? 0.f : (lse - zy);
}

template <typename Act>
cudaError_t cross_entropy(Act* logits, const int32_t* tgt, float* row_loss, int M, int V, int Vp,
                          const DevState* st, cudaStream_t s) {
    constexpr int VEC = Vec16<Act>::N;
    if (Vp % VEC) return cudaErrorInvalidValue;
    int nch = (Vp / VEC + CE_THREADS - 1) / CE_THREADS;
#define CE_CASE(NC)                                                                     \
    if (nch <= NC) {                                                                    \
        ce_kernel<Act, NC><<<M, CE_THREADS, 0, s>>>(logits, tgt, row_loss, V, Vp, st); \
        return cudaGetLastError();                                                      \
    }
    CE_CASE(1)
    CE_CASE(2)
    CE_CASE(4)
    CE_CASE(8)
    CE_CASE(16)
    CE_CASE(25)
    CE_CASE(32)
    CE_CASE(50)
#undef CE_CASE
    return cudaErrorInvalidValue;
}

template cudaError_t cross_entropy<float>(float*, const int32_t*, float*, int, int, int,
                                          const DevState*, cudaStream_t);
template cudaError_t cross_entropy<bf16>(bf16*, const int32_t*, float*, int, int, int,
                                         const DevState*, cudaStream_t);

}  // namespace k
