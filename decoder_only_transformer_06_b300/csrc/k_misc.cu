// Memory-bound kernels of the step: input validation, embedding forward and
// deterministic backward, bias-gradient column sums, split-K reduction,
// global grad norm + clip coefficient, fused AdamW.
#include "common.cuh"

namespace k {

int num_sms() {
    static std::atomic<int> cached[64];     // per device; 0 = not queried yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    std::atomic<int>& slot = cached[dev & 63];
    int n = slot.load();
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        slot.store(n);
    }
    return n;
}

// ---------------------------------------------------------------- validation
// Token ids must lie in [0, V), targets in [0, V) or -1 (ignore_index,
// nanoGPT guide Part IV Stage 4). Counts the valid targets and sets the
// cross-entropy gradient scale 1 / (n_valid * grad_accum_steps).
__global__ void validate_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ tgt,
                                int M, int V, DevState* st, int accum) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_cnt[32];
    __shared__ unsigned s_err[32];
    int cnt = 0;
    unsigned err = 0;
    for (int m = threadIdx.x; m < M; m += blockDim.x) {
        int t = tok[m];
        if (t < 0 || t >= V) err |= ERR_TOKEN_RANGE;
        if (tgt) {
            int y = tgt[m];
            if (y != -1) {
                if (y < 0 || y >= V) err |= ERR_TARGET_RANGE;
                else cnt++;
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        err |= __shfl_xor_sync(0xffffffffu, err, o);
    }
    int w = threadIdx.x / 32, l = threadIdx.x % 32;
    if (l == 0) { s_cnt[w] = cnt; s_err[w] = err; }
    __syncthreads();
    if (threadIdx.x == 0) {
        int c = 0;
        unsigned e = 0;
        for (int i = 0; i < (int)(blockDim.x / 32); i++) { c += s_cnt[i]; e |= s_err[i]; }
        st->n_valid = c;
        st->inv_count = c > 0 ? 1.0f / ((float)c * (float)accum) : 0.0f;
        if (e) atomicOr(&st->err, e);
    }
}

cudaError_t validate_inputs(const int32_t* tok, const int32_t* tgt, int M, int V, DevState* st,
                            int accum, cudaStream_t s) {
    (void)pdl_launch(validate_kernel, 1, 1024, 0, s, tok, tgt, M, V, st, accum);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- embedding
// x[m, :] = wte[tok[m], :] + wpe[m % T, :]  (nanoGPT guide Part IV Stage 4).
// Out-of-range ids are clamped here (the validation kernel records them).
__global__ void embed_fwd_kernel(const int32_t* __restrict__ tok, const float4* __restrict__ wte,
                                 const float4* __restrict__ wpe, float4* __restrict__ x, int M,
                                 int T, int C4, int V) {
    pdl_wait();
    pdl_trigger();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t n = (int64_t)M * C4;
    if (i >= n) return;
    int m = (int)(i / C4), c = (int)(i % C4);
    int t = tok[m];
    t = t < 0 ? 0 : (t >= V ? V - 1 : t);
    float4 a = wte[(int64_t)t * C4 + c], b = wpe[(int64_t)(m % T) * C4 + c];
    x[i] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

cudaError_t embed_fwd(const int32_t* tok, const float* wte, const float* wpe, float* x, int M,
                      int T, int C, int V, cudaStream_t s) {
    int C4 = C / 4;
    int64_t n = (int64_t)M * C4;
    (void)pdl_launch(embed_fwd_kernel, (unsigned)((n + 255) / 256), 256, 0, s, 
        tok, (const float4*)wte, (const float4*)wpe, (float4*)x, M, T, C4, V);
    return cudaGetLastError();
}

// Embedding backward, deterministic (no floating-point atomics):
//  1. one CTA sorts the entries by (token, position) in shared memory (a
//     stable radix sort on the token id; a bitonic sort of tok*M + m for
//     larger M or V), so equal tokens form contiguous segments ordered by
//     position;
//  2. fixed chunks of R sorted entries are summed in order; a segment wholly
//     inside its chunk is added to dwte directly, otherwise the chunk's partial
//     goes to a carry slot at the segment's first index in that chunk;
//  3. the chunk in which a spanning segment starts adds its carries in order.
static constexpr int EMB_R = 32;

__global__ void __launch_bounds__(1024) embed_sort_kernel(const int32_t* __restrict__ tok, int M,
                                                          int V, int P2, int* __restrict__ s_tok,
                                                          int* __restrict__ s_pos) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint32_t keys[];
    for (int i = threadIdx.x; i < P2; i += blockDim.x) {
        if (i < M) {
            int t = tok[i];
            t = t < 0 ? 0 : (t >= V ? V - 1 : t);
            keys[i] = (uint32_t)t * (uint32_t)M + (uint32_t)i;
        } else {
            keys[i] = 0xffffffffu;
        }
    }
    __syncthreads();
    for (int kk = 2; kk <= P2; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < P2; i += blockDim.x) {
                int ixj = i ^ j;
                if (ixj > i) {
                    uint32_t a = keys[i], b = keys[ixj];
                    bool up = (i & kk) == 0;
                    if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
        uint32_t kv = keys[i];
        s_tok[i] = (int)(kv / (uint32_t)M);
        s_pos[i] = (int)(kv % (uint32_t)M);
    }
}

// The same order (token, then position) by a stable LSD radix sort over the
// token id, for V <= 65536 and M <= EMB_RADIX_MAX_M: keys token << 16 | position
// start in position order; each pass ranks one 8-bit digit of the token.
// Warp w takes a contiguous slice of the keys in rounds of 32 (lanes in key
// order, equal digits of a round found with __match_any_sync), so equal digits
// keep their order within a round, across rounds and across warps: every pass
// is stable. Also writes, for every chunk of EMB_R sorted entries, the end of
// the segment that holds the chunk's last entry (seg_end), so that the carry
// pass needs no search.
static constexpr int RS_THREADS = 1024, RS_WARPS = RS_THREADS / 32;
static constexpr int EMB_RADIX_MAX_M = 24576;

__global__ void __launch_bounds__(RS_THREADS) embed_radix_kernel(const int32_t* __restrict__ tok, int M, int V,
                                                                 int passes, int* __restrict__ s_tok,
                                                                 int* __restrict__ s_pos,
                                                                 int* __restrict__ seg_end) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint32_t rs_sm[];
    uint32_t* a = rs_sm;                         // [M]
    uint32_t* b = rs_sm + M;                     // [M]
    uint32_t* cnt = rs_sm + 2 * M;               // [RS_WARPS][256]: counts, then running bases
    __shared__ uint32_t wsum[RS_WARPS];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int i = threadIdx.x; i < M; i += RS_THREADS) {
        int t = tok[i];
        t = t < 0 ? 0 : (t >= V ? V - 1 : t);
        a[i] = ((uint32_t)t << 16) | (uint32_t)i;
    }
    const int per = (M + RS_WARPS - 1) / RS_WARPS;
    const int w0 = min(M, warp * per), w1 = min(M, w0 + per);
    const unsigned lt = (1u << lane) - 1u;
    for (int pass = 0; pass < passes; pass++) {
        const int shift = 16 + 8 * pass;
        for (int i = threadIdx.x; i < 256 * RS_WARPS; i += RS_THREADS) cnt[i] = 0u;
        __syncthreads();
        for (int r = w0; r < w1; r += 32) {
            const int i = r + lane;
            const bool v = i < w1;
            const uint32_t d = v ? (a[i] >> shift) & 255u : 256u;
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            if (v && (peers & lt) == 0u) cnt[warp * 256 + d] += (uint32_t)__popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // exclusive scan over (digit, warp) in digit-major order: logical index
        // j = d * RS_WARPS + w at cnt[w * 256 + d]; thread t owns j = 8t .. 8t+7
        {
            uint32_t loc[8], sum = 0u;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int j = threadIdx.x * 8 + k;
                loc[k] = cnt[(j % RS_WARPS) * 256 + j / RS_WARPS];
                sum += loc[k];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) wsum[warp] = incl;
            __syncthreads();
            uint32_t before = 0u;
            for (int w = 0; w < warp; w++) before += wsum[w];
            uint32_t ex = before + incl - sum;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int j = threadIdx.x * 8 + k;
                cnt[(j % RS_WARPS) * 256 + j / RS_WARPS] = ex;
                ex += loc[k];
            }
        }
        __syncthreads();
        for (int r = w0; r < w1; r += 32) {
            const int i = r + lane;
            const bool v = i < w1;
            const uint32_t key = v ? a[i] : 0u;
            const uint32_t d = v ? (key >> shift) & 255u : 256u;
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            const uint32_t base = v ? cnt[warp * 256 + d] : 0u;
            __syncwarp();
            if (v) {
                b[base + (uint32_t)__popc(peers & lt)] = key;
                if ((peers & lt) == 0u) cnt[warp * 256 + d] = base + (uint32_t)__popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        uint32_t* t = a;
        a = b;
        b = t;
    }
    for (int i = threadIdx.x; i < M; i += RS_THREADS) {
        s_tok[i] = (int)(a[i] >> 16);
        s_pos[i] = (int)(a[i] & 0xffffu);
    }
    const int chunks = (M + EMB_R - 1) / EMB_R;
    for (int c = threadIdx.x; c < chunks; c += RS_THREADS) {
        const int last = min(M, (c + 1) * EMB_R) - 1;
        const uint32_t t = a[last] >> 16;
        int lo = last + 1, hi = M;                  // first entry after last with another token
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if ((a[mid] >> 16) == t) lo = mid + 1;
            else hi = mid;
        }
        seg_end[c] = lo;
    }
}

// seg_end for the bitonic path: per chunk, the end of the segment that holds
// its last sorted entry (binary search over the sorted tokens).
__global__ void embed_seg_end_kernel(const int* __restrict__ s_tok, int M, int* __restrict__ seg_end) {
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= (M + EMB_R - 1) / EMB_R) return;
    const int last = min(M, (c + 1) * EMB_R) - 1;
    const int t = s_tok[last];
    int lo = last + 1, hi = M;
    while (lo < hi) {
        const int mid = (lo + hi) / 2;
        if (s_tok[mid] == t) lo = mid + 1;
        else hi = mid;
    }
    seg_end[c] = lo;
}

__global__ void embed_chunk_kernel(const int* __restrict__ s_tok, const int* __restrict__ s_pos,
                                   const float4* __restrict__ dx, float4* __restrict__ dwte,
                                   float4* __restrict__ carry, int M, int C4) {
    pdl_wait();
    pdl_trigger();
    // the chunk's entries, with the tokens just before and after it, staged in
    // shared memory so that the row loads below do not wait on index loads
    __shared__ int st[EMB_R + 2], sp[EMB_R];
    const int i0 = blockIdx.x * EMB_R;
    const int i1 = min(i0 + EMB_R, M);
    const int n = i1 - i0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        st[j + 1] = s_tok[i0 + j];
        sp[j] = s_pos[i0 + j];
    }
    if (threadIdx.x == 0) {
        st[0] = i0 > 0 ? s_tok[i0 - 1] : -1;
        st[n + 1] = i1 < M ? s_tok[i1] : -1;
    }
    __syncthreads();
    const int c = threadIdx.x;
    if (c >= C4) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int seg = 0;
#pragma unroll 8
    for (int j = 0; j < n; j++) {
        const int t = st[j + 1];
        const float4 v = dx[(int64_t)sp[j] * C4 + c];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        if (st[j + 2] != t || j + 1 == n) {
            const bool from_before = seg == 0 && st[0] == t;
            const bool to_after = j + 1 == n && st[n + 1] == t;
            if (!from_before && !to_after) {
                float4* w = dwte + (int64_t)t * C4 + c;
                const float4 o = *w;
                *w = make_float4(o.x + acc.x, o.y + acc.y, o.z + acc.z, o.w + acc.w);
            } else {
                carry[(int64_t)(i0 + seg) * C4 + c] = acc;
            }
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
            seg = j + 1;
        }
    }
}

__global__ void embed_carry_kernel(const int* __restrict__ s_tok, const int* __restrict__ seg_end,
                                   const float4* __restrict__ carry, float4* __restrict__ dwte, int M, int C4) {
    pdl_wait();
    pdl_trigger();
    int c = threadIdx.x;
    if (c >= C4) return;
    int i0 = blockIdx.x * EMB_R;
    int i1 = min(i0 + EMB_R, M);
    if (i1 >= M) return;                     // nothing extends past the last chunk
    int t = s_tok[i1 - 1];
    if (s_tok[i1] != t) return;              // last segment ends inside this chunk
    int s = i1 - 1;
    while (s > i0 && s_tok[s - 1] == t) s--;
    if (s == i0 && i0 > 0 && s_tok[i0 - 1] == t) return;   // owned by an earlier chunk
    float4 acc = carry[(int64_t)s * C4 + c];
    // the later chunks' pieces start at their first entry, up to the segment's end
    const int e = seg_end[blockIdx.x];
#pragma unroll 4
    for (int b = i1; b < e; b += EMB_R) {
        const float4 v = carry[(int64_t)b * C4 + c];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    float4* w = dwte + (int64_t)t * C4 + c;
    float4 o = *w;
    *w = make_float4(o.x + acc.x, o.y + acc.y, o.z + acc.z, o.w + acc.w);
}

// dwpe[t, :] += sum over b of dx[b*T + t, :], b in increasing order.
__global__ void embed_pos_kernel(const float4* __restrict__ dx, float4* __restrict__ dwpe, int B,
                                 int T, int C4) {
    pdl_wait();
    pdl_trigger();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * C4) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b = 0; b < B; b++) {
        float4 v = dx[(int64_t)b * T * C4 + i];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    float4 o = dwpe[i];
    dwpe[i] = make_float4(o.x + acc.x, o.y + acc.y, o.z + acc.z, o.w + acc.w);
}

static int pow2_at_least(int m) {
    int p = 1;
    while (p < m) p <<= 1;
    return p;
}

// workspace: s_tok [M], s_pos [M], one spare word and seg_end [chunks] (ints),
// then the carries (fp32 [M, C], 256-byte aligned)
static int emb_chunks(int M) { return (M + EMB_R - 1) / EMB_R; }
size_t embed_bwd_workspace(int M, int C) {
    return (size_t)(2 * M + 1 + emb_chunks(M)) * sizeof(int) + (size_t)M * C * sizeof(float) + 256;
}

cudaError_t embed_bwd_sort(const int32_t* tok, int M, int V, void* workspace, cudaStream_t s) {
    int* s_tok = (int*)workspace;
    int* s_pos = s_tok + M;
    int* seg_end = s_pos + M + 1;
    if (V <= 65536 && M <= EMB_RADIX_MAX_M) {
        const size_t smem = ((size_t)2 * M + 256 * RS_WARPS) * sizeof(uint32_t);
        CUDA_OK(cudaFuncSetAttribute(embed_radix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem));
        (void)pdl_launch(embed_radix_kernel, 1, RS_THREADS, smem, s, tok, M, V, V <= 256 ? 1 : 2, s_tok,
                         s_pos, seg_end);
        return cudaGetLastError();
    }
    int P2 = pow2_at_least(M);
    size_t smem = (size_t)P2 * sizeof(uint32_t);
    CUDA_OK(cudaFuncSetAttribute(embed_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem));
    (void)pdl_launch(embed_sort_kernel, 1, 1024, smem, s, tok, M, V, P2, s_tok, s_pos);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(embed_seg_end_kernel, (emb_chunks(M) + 255) / 256, 256, 0, s, s_tok, M, seg_end);
    return cudaGetLastError();
}

cudaError_t embed_bwd_apply(const float* dx, float* dwte, float* dwpe, int M, int T, int C,
                            void* workspace, cudaStream_t s) {
    int* s_tok = (int*)workspace;
    int* s_pos = s_tok + M;
    float* carry = (float*)(((uintptr_t)(s_pos + M + 1 + emb_chunks(M)) + 255) & ~(uintptr_t)255);
    int C4 = C / 4;
    int chunks = (M + EMB_R - 1) / EMB_R;
    (void)pdl_launch(embed_chunk_kernel, chunks, C4, 0, s, s_tok, s_pos, (const float4*)dx, (float4*)dwte,
                                             (float4*)carry, M, C4);
    CUDA_OK(cudaGetLastError());
    const int* seg_end = s_pos + M + 1;      // written by embed_bwd_sort
    (void)pdl_launch(embed_carry_kernel, chunks, C4, 0, s, s_tok, seg_end, (const float4*)carry, (float4*)dwte,
                     M, C4);
    CUDA_OK(cudaGetLastError());
    int B = M / T;
    int64_t n = (int64_t)T * C4;
    (void)pdl_launch(embed_pos_kernel, (unsigned)((n + 255) / 256), 256, 0, s, (const float4*)dx, (float4*)dwpe,
                                                                 B, T, C4);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- column sums
// db[n] += sum_m dy[m, n], as a fixed-order two-stage reduction. Stage 1: a
// CTA of 32 x 8 threads covers 32 16-byte column vectors and one split of
// CS_ROWS_PER_SPLIT rows; threadIdx.y takes every 8th row, the 8 row phases
// are combined in order through shared memory. Stage 2 adds the split
// partials in split order.
static constexpr int CS_ROWS_PER_SPLIT = 256;

template <typename T>
__global__ void __launch_bounds__(256)
colsum_stage1(const T* __restrict__ dy, int64_t ld, int M, int N, float* __restrict__ partial) {
    pdl_wait();
    pdl_trigger();
    constexpr int VEC = 16 / sizeof(T);
    __shared__ float sm[8][32 * VEC + 1];
    const int n = (blockIdx.x * 32 + threadIdx.x) * VEC;
    const int r0 = blockIdx.y * CS_ROWS_PER_SPLIT;
    const int r1 = min(r0 + CS_ROWS_PER_SPLIT, M);
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; e++) acc[e] = 0.f;
    if (n < N) {
#pragma unroll 4
        for (int r = r0 + threadIdx.y; r < r1; r += 8) {
            uint4 w = *(const uint4*)(dy + (int64_t)r * ld + n);
            if constexpr (sizeof(T) == 2) {
                const __nv_bfloat162* h = (const __nv_bfloat162*)&w;
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    float2 f = __bfloat1622float2(h[t]);
                    acc[2 * t] += f.x;
                    acc[2 * t + 1] += f.y;
                }
            } else {
                const float* f = (const float*)&w;
#pragma unroll
                for (int t = 0; t < 4; t++) acc[t] += f[t];
            }
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; e++) sm[threadIdx.y][threadIdx.x * VEC + e] = acc[e];
    __syncthreads();
    for (int c = threadIdx.y * 32 + threadIdx.x; c < 32 * VEC; c += 256) {
        const int col = blockIdx.x * 32 * VEC + c;
        if (col < N) {
            float s = 0.f;
#pragma unroll
            for (int y = 0; y < 8; y++) s += sm[y][c];
            partial[(int64_t)blockIdx.y * N + col] = s;
        }
    }
}

// Second stage: block = 32 columns x 8 slices of the partial rows, slices
// combined in slice order (deterministic).
__global__ void __launch_bounds__(256)
colsum_stage2(const float* __restrict__ partial, int splits, int N, float* __restrict__ db) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sm[8][33];
    const int cx = threadIdx.x & 31, sl = threadIdx.x >> 5;
    const int n = blockIdx.x * 32 + cx;
    float s = 0.f;
    if (n < N)
        for (int k = sl; k < splits; k += 8) s += partial[(int64_t)k * N + n];
    sm[sl][cx] = s;
    __syncthreads();
    if (sl == 0 && n < N) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; k++) t += sm[k][cx];
        db[n] += t;
    }
}

cudaError_t colsum_partials_add(const float* partial, int groups, int N, float* db, cudaStream_t s) {
    if (groups < 1 || N < 1) return cudaErrorInvalidValue;
    (void)pdl_launch(colsum_stage2, (N + 31) / 32, 256, 0, s, partial, groups, N, db);
    return cudaGetLastError();
}

size_t colsum_partial_floats(int M, int N) {
    return (size_t)((M + CS_ROWS_PER_SPLIT - 1) / CS_ROWS_PER_SPLIT) * N;
}

template <typename T>
cudaError_t colsum_add(const T* dy, int64_t ld, int M, int N, float* db, float* partial,
                       cudaStream_t s) {
    constexpr int VEC = 16 / sizeof(T);
    if ((N % VEC) || (ld % VEC) || ((uintptr_t)dy & 15)) return cudaErrorInvalidValue;
    int splits = (M + CS_ROWS_PER_SPLIT - 1) / CS_ROWS_PER_SPLIT;
    dim3 grid((N / VEC + 31) / 32, splits);
    (void)pdl_launch(colsum_stage1<T>, grid, dim3(32, 8), 0, s, dy, ld, M, N, partial);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(colsum_stage2, (N + 31) / 32, 256, 0, s, partial, splits, N, db);
    return cudaGetLastError();
}
template cudaError_t colsum_add<float>(const float*, int64_t, int, int, float*, float*,
                                       cudaStream_t);
template cudaError_t colsum_add<bf16>(const bf16*, int64_t, int, int, float*, float*,
                                      cudaStream_t);

// ---------------------------------------------------------------- split-K
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int64_t n,
                                     float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int64_t n4 = n / 4;
    if (i >= n4) return;
    const float4* p = (const float4*)partial;
    float4 a = p[i];
    for (int k = 1; k < splits; k++) {
        float4 b = p[(int64_t)k * n4 + i];
        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    float4* o = (float4*)out;
    float4 c = o[i];
    o[i] = make_float4(c.x + a.x, c.y + a.y, c.z + a.z, c.w + a.w);
}

cudaError_t splitk_reduce_add(const float* partial, int splits, int64_t n, float* out,
                              cudaStream_t s) {
    int64_t n4 = n / 4;
    (void)pdl_launch(splitk_reduce_kernel, (unsigned)((n4 + 255) / 256), 256, 0, s, partial, splits, n, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- conversion
__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                   int64_t n4) {
    pdl_wait();
    pdl_trigger();
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 v = src[i];
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *(uint32_t*)&lo;
    o.y = *(uint32_t*)&hi;
    dst[i] = o;
}

cudaError_t f32_to_bf16(const float* src, bf16* dst, int64_t n, cudaStream_t s) {
    int64_t n4 = n / 4;
    if (n4 == 0) return cudaSuccess;
    (void)pdl_launch(f32_to_bf16_kernel, (unsigned)((n4 + 255) / 256), 256, 0, s, (const float4*)src,
                                                                     (uint2*)dst, n4);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- loss mean
__global__ void loss_reduce_kernel(const float* __restrict__ row_loss, int M, DevState* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ double sm[32];
    double acc = 0.0;
    for (int i = threadIdx.x; i < M; i += blockDim.x) acc += (double)row_loss[i];
    acc = warp_sum_d(acc);
    if (threadIdx.x % 32 == 0) sm[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int i = 0; i < (int)(blockDim.x / 32); i++) s += sm[i];
        st->loss_sum = s;
        st->loss = (float)(s / (double)(st->n_valid > 0 ? st->n_valid : 1));
    }
}

cudaError_t loss_reduce(const float* row_loss, int M, DevState* st, cudaStream_t s) {
    (void)pdl_launch(loss_reduce_kernel, 1, 1024, 0, s, row_loss, M, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- grad norm
// Sum of squares over the flat gradient arena: each CTA owns a fixed
// contiguous range, fp32 per thread, fp64 across the CTA; partials are
// combined in order by step_finalize.
__global__ void grad_norm_kernel(const float4* __restrict__ g, int64_t n4, int64_t per_block,
                                 double* __restrict__ partial) {
    pdl_wait();
    pdl_trigger();
    __shared__ double sm[32];
    int64_t b0 = (int64_t)blockIdx.x * per_block;
    int64_t b1 = min(b0 + per_block, n4);
    float acc = 0.f;
    for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x) {
        float4 v = g[i];
        acc += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    double d = warp_sum_d((double)acc);
    if (threadIdx.x % 32 == 0) sm[threadIdx.x / 32] = d;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int i = 0; i < (int)(blockDim.x / 32); i++) s += sm[i];
        partial[blockIdx.x] = s;
    }
}

cudaError_t grad_norm(const float* g, int64_t n, double* partial, int nparts, cudaStream_t s) {
    int64_t n4 = n / 4;
    int64_t per_block = (n4 + nparts - 1) / nparts;
    (void)pdl_launch(grad_norm_kernel, nparts, 512, 0, s, (const float4*)g, n4, per_block, partial);
    return cudaGetLastError();
}

// norm = sqrt(sum); clip coefficient min(1, clip/(norm + 1e-6)) (PyTorch
// clip_grad_norm_ reading of "rescales if it exceeds 1.0", nanoGPT guide
// Stage 5); a non-finite norm skips the update and leaves t unchanged.
__global__ void step_finalize_kernel(const double* __restrict__ partial, int nparts, float clip,
                                     float beta1, float beta2, DevState* st) {
    pdl_wait();
    pdl_trigger();
    __shared__ double sm[32];
    double acc = 0.0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) acc += partial[i];
    acc = warp_sum_d(acc);
    if (threadIdx.x % 32 == 0) sm[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int i = 0; i < (int)(blockDim.x / 32); i++) s += sm[i];
        double norm = sqrt(s);
        st->grad_norm = (float)norm;
        if (isfinite(norm)) {
            double c = (double)clip / (norm + 1e-6);
            st->clip_coef = (float)(c < 1.0 ? c : 1.0);
            int t = st->step_t + 1;
            st->step_t = t;
            st->bc1 = (float)(1.0 - pow((double)beta1, (double)t));
            st->bc2 = (float)(1.0 - pow((double)beta2, (double)t));
            st->skip = 0;
        } else {
            st->clip_coef = 0.f;
            st->skip = 1;
        }
    }
}

cudaError_t step_finalize(const double* partial, int nparts, float clip, float beta1, float beta2,
                          DevState* st, cudaStream_t s) {
    (void)pdl_launch(step_finalize_kernel, 1, 256, 0, s, partial, nparts, clip, beta1, beta2, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- AdamW
// Decoupled decay on elements below decay_end (the arena keeps every 2-D
// tensor first), bias-corrected moments, eps outside the sqrt; the bf16 copy
// of elements below bf16_end is refreshed for the tensor cores.
__global__ void adamw_kernel(float4* __restrict__ p, const float4* __restrict__ g,
                             float4* __restrict__ m, float4* __restrict__ v,
                             uint2* __restrict__ pb, int64_t n4, int64_t decay_end4,
                             int64_t bf16_end4, float lr, float beta1, float beta2, float eps,
                             float wd, const DevState* __restrict__ st) {
    pdl_wait();
    pdl_trigger();
    if (st->skip) return;
    const float c = st->clip_coef;
    const float inv_bc1 = 1.0f / st->bc1;
    const float inv_sqrt_bc2 = 1.0f / sqrtf(st->bc2);
    const float step = lr * inv_bc1;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 pp = p[i], gg = g[i], mm = m[i], vv = v[i];
        float decay = (i < decay_end4) ? (1.0f - lr * wd) : 1.0f;
        float* pa = &pp.x; float* ga = &gg.x; float* ma = &mm.x; float* va = &vv.x;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float gj = ga[j] * c;
            float pj = pa[j] * decay;
            float mj = beta1 * ma[j] + (1.0f - beta1) * gj;
            float vj = beta2 * va[j] + (1.0f - beta2) * gj * gj;
            pj -= step * mj / (sqrtf(vj) * inv_sqrt_bc2 + eps);
            pa[j] = pj; ma[j] = mj; va[j] = vj;
        }
        p[i] = pp; m[i] = mm; v[i] = vv;
        if (i < bf16_end4) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pp.x, pp.y), hi = __floats2bfloat162_rn(pp.z, pp.w);
            uint2 o;
            o.x = *(uint32_t*)&lo;
            o.y = *(uint32_t*)&hi;
            pb[i] = o;
        }
    }
}

cudaError_t adamw(float* p, const float* g, float* m, float* v, bf16* p_bf16, int64_t n,
                  int64_t decay_end, int64_t bf16_end, float lr, float beta1, float beta2, float eps,
                  float wd, const DevState* st, cudaStream_t s) {
    int64_t n4 = n / 4;
    const int64_t want = (n4 + 511) / 512;
    int blocks = want < num_sms() * 4 ? (int)(want > 0 ? want : 1) : num_sms() * 4;
    (void)pdl_launch(adamw_kernel, blocks, 512, 0, s, (float4*)p, (const float4*)g, (float4*)m, (float4*)v,
                                        (uint2*)p_bf16, n4, decay_end / 4,
                                        p_bf16 ? bf16_end / 4 : 0, lr, beta1, beta2, eps, wd, st);
    return cudaGetLastError();
}

}  // namespace k
