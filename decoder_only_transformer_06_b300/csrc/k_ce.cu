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
#include "ptx.cuh"

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
    pdl_wait();
    pdl_trigger();
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


// ------------------------------------------------------------------ bf16 rows
// Persistent variant for bf16 logits whose row fits in shared memory (Vp <=
// 110000): two CTAs per SM, each walking rows blockIdx.x, +gridDim.x, ...
// with one row buffer: a row arrives by one TMA bulk copy and the gradient row
// leaves by one bulk store, while the other CTA on the SM computes. Per row:
//   pass 1  max over j < V (packed bf16x2 max);
//   pass 2  e_j = exp(z_j - max) in fp32, sum in fp32, e_j kept as bf16 in place;
//   pass 3  dz_j = (e_j / sum - [j == y]) * scale, 0 on pad columns.
// Storing e_j in bf16 rounds it once more at the precision the gradient is
// written in anyway.
static constexpr int CEB_THREADS = 512;

__device__ __forceinline__ float block_reduce_n(float v, bool is_max, float* sm) {
    v = is_max ? warp_max(v) : warp_sum(v);
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) sm[w] = v;
    __syncthreads();
    float r = sm[0];
    for (int i = 1; i < CEB_THREADS / 32; i++) r = is_max ? fmaxf(r, sm[i]) : r + sm[i];
    return r;
}

__global__ void __launch_bounds__(CEB_THREADS, 2)
ce_bulk_kernel(bf16* __restrict__ logits, const int32_t* __restrict__ tgt,
               float* __restrict__ row_loss, int M, int V, int Vp, DevState* st) {
    extern __shared__ __align__(128) uint8_t ce_smem[];
    const uint32_t rowbytes = (uint32_t)Vp * 2;
    const uint32_t padbytes = (rowbytes + 127) & ~127u;
    bf16* cur = (bf16*)ce_smem;
    uint64_t* bar = (uint64_t*)(ce_smem + padbytes);   // [2]: the row's two halves
    float* red = (float*)(bar + 2);
    const int tid = threadIdx.x;
    if (tid == 0) {
        ptx::mbar_init(&bar[0], 1);
        ptx::mbar_init(&bar[1], 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();                       // the previous kernel's outputs are visible
    pdl_trigger();
    const int nvec = Vp / 8;          // 16-byte chunks per row
    const int nfull = V / 8;          // chunks entirely below V
    // The row moves in two halves (chunks [0, nh) and [nh, nvec)), each with its
    // own barrier and bulk copies: the maximum pass starts on the first half
    // while the second is arriving, and the first half's gradients leave while
    // the second half's are computed.
    const int nh = nvec / 2;
    const uint32_t h0 = (uint32_t)nh * 16u, h1 = rowbytes - h0;
    const float L2E = 1.4426950408889634f;
    const float scale_valid = st->inv_count;
    uint32_t par = 0;
    for (int row = blockIdx.x; row < M; row += gridDim.x, par ^= 1) {
        if (tid == 0) {
            const bf16* src = logits + (int64_t)row * Vp;
            ptx::bulk_wait_read_1();              // the previous row's first-half store has read it
            ptx::mbar_arrive_expect_tx(&bar[0], h0);
            ptx::bulk_g2s(cur, src, h0, &bar[0]);
            ptx::bulk_wait_read_all();            // and the second half's
            ptx::mbar_arrive_expect_tx(&bar[1], h1);
            ptx::bulk_g2s((uint8_t*)cur + h0, (const uint8_t*)src + h0, h1, &bar[1]);
        }
        int y = tgt[row];
        const bool ignore = (y == -1);
        y = (y < 0 || y >= V) ? 0 : y;
        const uint4* cv = (const uint4*)cur;
        // pass 1: max, first half as soon as it has landed, then the second
        __nv_bfloat162 mx2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
        bool ok = ptx::mbar_wait_bounded(&bar[0], par);
        const int e0 = nh < nfull ? nh : nfull;
        if (ok) {
#pragma unroll 4
            for (int vi = tid; vi < e0; vi += CEB_THREADS) {
                uint4 w = cv[vi];
                const __nv_bfloat162* h = (const __nv_bfloat162*)&w;
                mx2 = __hmax2(mx2, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
            }
            ok = ptx::mbar_wait_bounded(&bar[1], par);
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(&st->err, ERR_TIMEOUT);
                st->timeout_site = 2;
            }
            break;
        }
#pragma unroll 4
        for (int vi = e0 + tid; vi < nfull; vi += CEB_THREADS) {
            uint4 w = cv[vi];
            const __nv_bfloat162* h = (const __nv_bfloat162*)&w;
            mx2 = __hmax2(mx2, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
        }
        const float zy = __bfloat162float(cur[y]);
        float mx = fmaxf(__low2float(mx2), __high2float(mx2));
        if (tid == 0) {
            for (int j = nfull * 8; j < V; j++) mx = fmaxf(mx, __bfloat162float(cur[j]));
        }
        mx = block_reduce_n(mx, true, red);
        const float mxl = mx * L2E;
        // pass 2: e = exp(z - max), sum; e kept in place as bf16
        float sum = 0.f;
#pragma unroll 2
        for (int vi = tid; vi < nfull; vi += CEB_THREADS) {
            uint4 w = cv[vi];
            const __nv_bfloat162* h = (const __nv_bfloat162*)&w;
            uint4 o;
            uint32_t* op = (uint32_t*)&o;
#pragma unroll
            for (int t = 0; t < 4; t++) {
                float2 f = __bfloat1622float2(h[t]);
                float e0f = ptx::ex2(fmaf(f.x, L2E, -mxl)), e1f = ptx::ex2(fmaf(f.y, L2E, -mxl));
                sum += e0f + e1f;
                __nv_bfloat162 p = __floats2bfloat162_rn(e0f, e1f);
                op[t] = *(uint32_t*)&p;
            }
            ((uint4*)cur)[vi] = o;
        }
        if (tid == 0) {
            for (int j = nfull * 8; j < V; j++) {
                float e = ptx::ex2(fmaf(__bfloat162float(cur[j]), L2E, -mxl));
                sum += e;
                cur[j] = __float2bfloat16_rn(e);
            }
        }
        sum = block_reduce_n(sum, false, red);
        const float inv = 1.0f / sum;
        const float scale = ignore ? 0.f : scale_valid;
        // pass 3: gradient in place, half by half; each half leaves by one bulk store
        for (int hh = 0; hh < 2; hh++) {
            const int v0 = hh == 0 ? 0 : nh, v1 = hh == 0 ? nh : nvec;
#pragma unroll 2
            for (int vi = v0 + tid; vi < v1; vi += CEB_THREADS) {
                uint4 o;
                uint32_t* op = (uint32_t*)&o;
                if (vi < nfull) {
                    uint4 w = cv[vi];
                    const __nv_bfloat162* h = (const __nv_bfloat162*)&w;
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        float2 f = __bfloat1622float2(h[t]);
                        const int j = vi * 8 + 2 * t;
                        float d0 = (f.x * inv - (j == y ? 1.f : 0.f)) * scale;
                        float d1 = (f.y * inv - (j + 1 == y ? 1.f : 0.f)) * scale;
                        __nv_bfloat162 p = __floats2bfloat162_rn(d0, d1);
                        op[t] = *(uint32_t*)&p;
                    }
                } else {
                    const bf16* e = cur + vi * 8;
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        const int j = vi * 8 + 2 * t;
                        float d0 = j < V ? (__bfloat162float(e[2 * t]) * inv - (j == y ? 1.f : 0.f)) * scale : 0.f;
                        float d1 = j + 1 < V ? (__bfloat162float(e[2 * t + 1]) * inv - (j + 1 == y ? 1.f : 0.f)) * scale : 0.f;
                        __nv_bfloat162 p = __floats2bfloat162_rn(d0, d1);
                        op[t] = *(uint32_t*)&p;
                    }
                }
                ((uint4*)cur)[vi] = o;
            }
            ptx::fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                ptx::bulk_s2g((uint8_t*)(logits + (int64_t)row * Vp) + (hh == 0 ? 0u : h0),
                              (const uint8_t*)cur + (hh == 0 ? 0u : h0), hh == 0 ? h0 : h1);
                ptx::bulk_commit();
            }
        }
        if (tid == 0) row_loss[row] = ignore ? 0.f : (mx + logf(sum) - zy);
    }
    if (tid == 0) ptx::bulk_wait_all();
}

template <typename Act>
cudaError_t cross_entropy(Act* logits, const int32_t* tgt, float* row_loss, int M, int V, int Vp,
                          DevState* st, cudaStream_t s) {
    constexpr int VEC = Vec16<Act>::N;
    if (Vp % VEC) return cudaErrorInvalidValue;
    if constexpr (sizeof(Act) == 2) {
        const size_t pad = ((size_t)Vp * 2 + 127) & ~(size_t)127;
        const size_t smem = pad + 16 + CEB_THREADS / 32 * sizeof(float);
        if (Vp >= 1024 && smem <= 110 * 1024) {
            CUDA_OK(cudaFuncSetAttribute(ce_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem));
            CUDA_OK(cudaFuncSetAttribute(ce_bulk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         100));
            int grid = M < 2 * num_sms() ? M : 2 * num_sms();
            (void)pdl_launch(ce_bulk_kernel, grid, CEB_THREADS, smem, s, (bf16*)logits, tgt, row_loss, M, V, Vp, st);
            return cudaGetLastError();
        }
    }
    int nch = (Vp / VEC + CE_THREADS - 1) / CE_THREADS;
#define CE_CASE(NC)                                                                     \
    if (nch <= NC) {                                                                    \
        (void)pdl_launch(ce_kernel<Act, NC>, M, CE_THREADS, 0, s, logits, tgt, row_loss, V, Vp, st); \
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

template cudaError_t cross_entropy<float>(float*, const int32_t*, float*, int, int, int, DevState*,
                                          cudaStream_t);
template cudaError_t cross_entropy<bf16>(bf16*, const int32_t*, float*, int, int, int, DevState*,
                                         cudaStream_t);

}  // namespace k
