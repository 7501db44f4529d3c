// One sampling step of generation ("Let's reproduce GPT-2", 00:37:02 the
// sampling loop; nanoGPT guide, sample.py): per row of last-position logits,
// divide by the temperature, keep the top k (every entry >= the k-th largest,
// ties included, as the pages' topk mask does), softmax, and draw the token by
// inverse CDF from a uniform the caller supplies; optionally append the token
// to the row's context (shifting the context left by one once it is full, the
// pages' crop to the block size).
//
// One 1024-thread CTA per row. Every reduction has a fixed order, so a call is
// deterministic: thread t owns the contiguous column chunk
// [t*chunk, (t+1)*chunk) and the block combines the per-thread results in
// thread order. The top-k threshold is the k-th largest value found by a
// bitwise search over the order-preserving 32-bit keys of the floats (32
// block-wide counting passes over keys cached in shared memory, no sort).
#include "common.cuh"

namespace k {

namespace {

constexpr int SMP_THREADS = 1024;
constexpr int SMP_WARPS = SMP_THREADS / 32;
constexpr int SMP_KEYS_MAX = 56 * 1024;          // keys cached in shared memory up to this V

// Order-preserving key of a float: a < b (as floats, no NaN) <=> key(a) < key(b).
__device__ __forceinline__ uint32_t fkey(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide sum of an int (fixed order); every thread gets the result.
__device__ __forceinline__ int block_sum_int(int v, int* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) sh[w] = v;
    __syncthreads();
    int r = l < SMP_WARPS ? sh[l] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Block-wide maximum of (value, -index): the largest value, lowest index on
// ties. Every thread gets both.
__device__ __forceinline__ void block_argmax(float v, int i, float* shv, int* shi, float& bv, int& bi) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
    const int w = threadIdx.x / 32, l = threadIdx.x % 32;
    __syncthreads();
    if (l == 0) { shv[w] = v; shi[w] = i; }
    __syncthreads();
    v = l < SMP_WARPS ? shv[l] : -INFINITY;
    i = l < SMP_WARPS ? shi[l] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
    bv = v;
    bi = i;
}

}  // namespace

__global__ void __launch_bounds__(SMP_THREADS)
sample_kernel(const float* __restrict__ logits, int V, int64_t ld, float temperature, int top_k,
              const float* __restrict__ uni, int32_t* __restrict__ out, int32_t* __restrict__ ctx, int T,
              int t) {
    pdl_wait();
    pdl_trigger();
    __shared__ float shv[SMP_WARPS];
    __shared__ int shi[SMP_WARPS];
    __shared__ float sh_scan[SMP_WARPS];
    __shared__ int sh_tok;
    extern __shared__ uint32_t skey[];               // [V] keys of x when V <= SMP_KEYS_MAX
    const int row = blockIdx.x, tid = threadIdx.x;
    const float* z = logits + (int64_t)row * ld;
    const int chunk = (V + SMP_THREADS - 1) / SMP_THREADS;
    const int c0 = min(V, tid * chunk), c1 = min(V, c0 + chunk);
    const bool greedy = !(temperature > 0.f);
    // x_j = z_j / temperature (IEEE division; greedy uses z itself)
    auto xval = [&](int j) { return greedy ? z[j] : z[j] / temperature; };

    // the largest x (lowest index on ties)
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = c0; j < c1; j++) {
        const float x = xval(j);
        if (x > bv) { bv = x; bi = j; }
    }
    float xmax;
    int amax;
    block_argmax(bv, bi, shv, shi, xmax, amax);
    int token = amax;
    if (!greedy) {
        // top-k threshold: the largest key K with #{key >= K} >= k
        uint32_t thr = 0u;
        if (top_k > 0 && top_k < V) {
            const bool cached = V <= SMP_KEYS_MAX;
            if (cached)
                for (int j = c0; j < c1; j++) skey[j] = fkey(xval(j));
            __syncthreads();
            for (int bit = 31; bit >= 0; bit--) {
                const uint32_t cand = thr | (1u << bit);
                int cnt = 0;
                for (int j = c0; j < c1; j++) cnt += (cached ? skey[j] : fkey(xval(j))) >= cand ? 1 : 0;
                if (block_sum_int(cnt, shi) >= top_k) thr = cand;
            }
        }
        // w_j = exp(x_j - max) on the kept entries; chunk sums; exclusive scan in
        // thread order
        float s = 0.f;
        int lastk = -1;                                  // last kept column of the chunk
        for (int j = c0; j < c1; j++) {
            const float x = xval(j);
            if (fkey(x) >= thr) {
                s += expf(x - xmax);
                lastk = j;
            }
        }
        // the last kept column of the row (exact in fp32: V < 2^24)
        float lastf;
        int unused;
        block_argmax((float)lastk, 0, shv, shi, lastf, unused);
        const int w = tid / 32, l = tid % 32;
        float inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, inc, o);
            if (l >= o) inc += y;
        }
        __syncthreads();
        if (l == 31) sh_scan[w] = inc;
        __syncthreads();
        if (w == 0) {
            float v = l < SMP_WARPS ? sh_scan[l] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, v, o);
                if (l >= o) v += y;
            }
            if (l < SMP_WARPS) sh_scan[l] = v;            // inclusive warp totals
        }
        __syncthreads();
        const float excl = (w > 0 ? sh_scan[w - 1] : 0.f) + (inc - s);
        const float total = sh_scan[SMP_WARPS - 1];
        const float target = uni[row] * total;
        // the first thread whose chunk ends above the target walks its chunk
        const int first = (excl + s > target && s > 0.f) ? tid : 0x7fffffff;
        float dummy;
        int owner;
        block_argmax(0.f, first, shv, shi, dummy, owner);
        if (tid == owner) {
            float acc = excl;
            int pick = -1, last = -1;
            for (int j = c0; j < c1; j++) {
                const float x = xval(j);
                if (fkey(x) < thr) continue;
                last = j;
                acc += expf(x - xmax);
                if (acc > target) { pick = j; break; }
            }
            sh_tok = pick >= 0 ? pick : last;
        }
        __syncthreads();
        // a target at or above the rounded total (no owner) takes the last kept column
        token = owner == 0x7fffffff ? (int)lastf : sh_tok;
    }
    if (tid == 0) out[row] = token;
    if (ctx) {
        int32_t* c = ctx + (int64_t)row * T;
        if (t < T) {
            if (tid == 0) c[t] = token;
        } else {
            // full context: shift left by one (read everything, then write)
            int32_t v[(1024 + SMP_THREADS - 1) / SMP_THREADS + 1];
            int n = 0;
            for (int i = tid + 1; i < T; i += SMP_THREADS) v[n++] = c[i];
            __syncthreads();
            n = 0;
            for (int i = tid + 1; i < T; i += SMP_THREADS) c[i - 1] = v[n++];
            if (tid == 0) c[T - 1] = token;
        }
    }
}

cudaError_t sample(const float* logits, int rows, int V, int64_t ld, float temperature, int top_k,
                   const float* u, int32_t* out, int32_t* ctx, int T, int t, cudaStream_t s) {
    if (rows <= 0 || V <= 0 || ld < V || !logits || !u || !out) return cudaErrorInvalidValue;
    if (ctx && (T < 1 || T > 1024 || t < 1 || t > T)) return cudaErrorInvalidValue;
    const bool cache = temperature > 0.f && top_k > 0 && top_k < V && V <= SMP_KEYS_MAX;
    const size_t smem = cache ? (size_t)V * 4 : 0;
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        CUDA_OK(cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SMP_KEYS_MAX * 4));
        attr_done.fetch_or(dbit);
    }
    (void)pdl_launch(sample_kernel, rows, SMP_THREADS, smem, s, logits, V, ld, temperature, top_k, u, out, ctx, T, t);
    return cudaGetLastError();
}

}  // namespace k
