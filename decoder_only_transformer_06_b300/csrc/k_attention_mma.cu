// Causal flash attention BACKWARD, bf16 operands / fp32 softmax and
// accumulation, head size 64, on warp-level mma.sync (m16n8k16) tensor-core
// instructions (the forward runs on tcgen05: k_attention_tc.cu).
//
// Semantics: the manual attention of nanoGPT's CausalSelfAttention (nanoGPT
// guide Deep dive 1): S = q k^T / sqrt(hs), keys j > i masked to -inf before
// the softmax, o = softmax(S) v. The probabilities are recomputed from the
// forward's per-row lse ("Let's reproduce GPT-2" 02:00:18, Flash Attention;
// nixfred "Flash attention"), so the T x T matrices never leave the chip.
//
// K/V and Q/dO blocks of 64 rows are double-buffered through 128B-XOR-swizzled
// shared memory with cp.async; 4 warps x 16 rows per CTA.
// Deterministic (no atomics): rowsum(dO*O) pre-pass; one kernel
// accumulates dK/dV per 64-key block over the query blocks that see it;
// another accumulates dQ per 64-query block over the key blocks it sees.
// Layout as in the fp32 kernels: qkv [B*T, 3C], out [B*T, C], lse [B,H,T].
#include "common.cuh"

namespace k {

static constexpr int FA_BLK = 64;
static constexpr int FA_HS = 64;
static constexpr int FA_THREADS = 128;
static constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ uint32_t s_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(uint32_t*)&h;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// Address of 16-byte chunk `chunk` of row `row` in a 64x64 bf16 tile whose
// chunks are XOR-swizzled by the row (conflict-free ldmatrix).
__device__ __forceinline__ uint32_t tile_addr(const bf16* tile, int row, int chunk) {
    return s_u32(tile + row * FA_HS + ((chunk ^ (row & 7)) << 3));
}

// Rows [row0, row0+64) of a [*, ld] bf16 matrix (columns col0..col0+63) into a
// swizzled tile; rows >= nvalid are zero-filled.
__device__ __forceinline__ void load_tile(bf16* tile, const bf16* g, int64_t ld, int row0,
                                          int nvalid) {
    for (int i = threadIdx.x; i < FA_BLK * 8; i += FA_THREADS) {
        int r = i >> 3, c = i & 7;
        bool ok = row0 + r < nvalid;
        const bf16* src = ok ? g + (int64_t)(row0 + r) * ld + c * 8 : g;
        cp_async16(tile_addr(tile, r, c), src, ok ? 16 : 0);
    }
}

// A fragments (16 rows starting at r0, all 64 columns = 4 k-steps) from a tile.
__device__ __forceinline__ void load_a_frags(const bf16* tile, int r0, uint32_t (&a)[4][4]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        int row = r0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        int chunk = 2 * ks + (lane >> 4);
        ldsm_x4(tile_addr(tile, row, chunk), a[ks][0], a[ks][1], a[ks][2], a[ks][3]);
    }
}

// acc[16 x 64] += A[16 x 64 (k)] * X^T where X is a 64x64 tile stored
// [n][k] (n = rows of the tile): B fragments via plain ldmatrix.
__device__ __forceinline__ void mma_a_xt(float (&acc)[8][4], const uint32_t (&a)[4][4],
                                         const bf16* tile) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
#pragma unroll
        for (int np = 0; np < 4; np++) {
            uint32_t b0, b1, b2, b3;
            int row = np * 16 + (lane & 7) + 8 * (lane >> 4);
            int chunk = 2 * ks + ((lane >> 3) & 1);
            ldsm_x4(tile_addr(tile, row, chunk), b0, b1, b2, b3);
            mma16816(acc[2 * np], a[ks], b0, b1);
            mma16816(acc[2 * np + 1], a[ks], b2, b3);
        }
    }
}

// acc[16 x 64] += P[16 x 64 (k)] * X where X is a 64x64 tile stored [k][n]:
// B fragments via ldmatrix.trans. P given as fp32 accumulator layout.
__device__ __forceinline__ void mma_p_x(float (&acc)[8][4], const float (&p)[8][4],
                                        const bf16* tile) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {
        uint32_t a[4];
        a[0] = pack2(p[2 * ks][0], p[2 * ks][1]);
        a[1] = pack2(p[2 * ks][2], p[2 * ks][3]);
        a[2] = pack2(p[2 * ks + 1][0], p[2 * ks + 1][1]);
        a[3] = pack2(p[2 * ks + 1][2], p[2 * ks + 1][3]);
#pragma unroll
        for (int np = 0; np < 4; np++) {
            uint32_t b0, b1, b2, b3;
            int row = ks * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            int chunk = 2 * np + (lane >> 4);
            ldsm_x4_t(tile_addr(tile, row, chunk), b0, b1, b2, b3);
            mma16816(acc[2 * np], a, b0, b1);
            mma16816(acc[2 * np + 1], a, b2, b3);
        }
    }
}

__device__ __forceinline__ void zero8x4(float (&a)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) a[i][j] = 0.f;
}

// Store a 16x64 fp32 accumulator (rows r0.., scaled) as bf16 into rows of a
// [*, ld] matrix, skipping rows >= nvalid.
__device__ __forceinline__ void store_acc(const float (&acc)[8][4], bf16* g, int64_t ld, int r0,
                                          int nvalid, float scale) {
    const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
        int col = nt * 8 + 2 * t;
        int ra = r0 + gq, rb = r0 + gq + 8;
        if (ra < nvalid)
            *(uint32_t*)(g + (int64_t)ra * ld + col) = pack2(acc[nt][0] * scale, acc[nt][1] * scale);
        if (rb < nvalid)
            *(uint32_t*)(g + (int64_t)rb * ld + col) = pack2(acc[nt][2] * scale, acc[nt][3] * scale);
    }
}

// ------------------------------------------------------------------ backward
// D[b,h,i] = sum_c dO[i, h*64+c] * O[i, h*64+c]; one thread per (row, head).
__global__ void fa_bwd_d_kernel(const bf16* __restrict__ out, const bf16* __restrict__ dout,
                                float* __restrict__ D, int B, int T, int H) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)B * T * H) return;
    int h = (int)(idx % H);
    int64_t row = idx / H;             // b*T + t
    int64_t b = row / T, tt = row % T;
    const int C = H * FA_HS;
    const uint4* o4 = (const uint4*)(out + row * C + h * FA_HS);
    const uint4* d4 = (const uint4*)(dout + row * C + h * FA_HS);
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        uint4 a = o4[q], c = d4[q];
        const __nv_bfloat162* ha = (const __nv_bfloat162*)&a;
        const __nv_bfloat162* hc = (const __nv_bfloat162*)&c;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 fa = __bfloat1622float2(ha[j]), fc = __bfloat1622float2(hc[j]);
            s += fa.x * fc.x + fa.y * fc.y;
        }
    }
    D[(b * H + h) * T + tt] = s;
}

// dK, dV for 64 keys of one (b, h): loop over query blocks at or after them.
__global__ void __launch_bounds__(FA_THREADS)
fa_bwd_dkv_kernel(const bf16* __restrict__ qkv, const bf16* __restrict__ dout,
                  const float* __restrict__ lse, const float* __restrict__ D,
                  bf16* __restrict__ dqkv, int T, int H) {
    extern __shared__ __align__(128) uint8_t fa_smem[];
    bf16* sK = (bf16*)fa_smem;
    bf16* sV = sK + FA_BLK * FA_HS;
    bf16* sQ = sV + FA_BLK * FA_HS;               // [2][64*64]
    bf16* sdO = sQ + 2 * FA_BLK * FA_HS;          // [2][64*64]
    float* sL = (float*)(sdO + 2 * FA_BLK * FA_HS);  // [2][64]
    float* sD = sL + 2 * FA_BLK;                  // [2][64]

    const int nb = (T + FA_BLK - 1) / FA_BLK;
    const int kb = blockIdx.x;
    const int bh = blockIdx.y, h = bh % H, b = bh / H;
    const int C = H * FA_HS;
    const int64_t ld = 3 * C;
    const bf16* base = qkv + (int64_t)b * T * ld;
    const bf16* qg = base + h * FA_HS;
    const bf16* kg = base + C + h * FA_HS;
    const bf16* vg = base + 2 * C + h * FA_HS;
    const bf16* dog = dout + (int64_t)b * T * C + h * FA_HS;
    const float* lg = lse + (int64_t)bh * T;
    const float* Dg = D + (int64_t)bh * T;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
    const float scale = 1.f / sqrtf((float)FA_HS);
    const float sl2 = LOG2E * scale;

    load_tile(sK, kg, ld, kb * FA_BLK, T);
    load_tile(sV, vg, ld, kb * FA_BLK, T);
    auto load_q = [&](int qb, int buf) {
        load_tile(sQ + buf * FA_BLK * FA_HS, qg, ld, qb * FA_BLK, T);
        load_tile(sdO + buf * FA_BLK * FA_HS, dog, C, qb * FA_BLK, T);
        for (int i = threadIdx.x; i < FA_BLK; i += FA_THREADS) {
            int q = qb * FA_BLK + i;
            sL[buf * FA_BLK + i] = q < T ? lg[q] : 0.f;
            sD[buf * FA_BLK + i] = q < T ? Dg[q] : 0.f;
        }
    };
    load_q(kb, 0);
    cp_commit();

    uint32_t kf[4][4], vf[4][4];
    float dk[8][4], dv[8][4];
    zero8x4(dk);
    zero8x4(dv);
    const int key0 = kb * FA_BLK + warp * 16 + gq;   // keys of this thread: key0, key0+8

    for (int qb = kb; qb < nb; qb++) {
        const int buf = (qb - kb) & 1;
        __syncthreads();   // previous iteration done with buf^1
        if (qb + 1 < nb) load_q(qb + 1, buf ^ 1);
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (qb == kb) {
            load_a_frags(sK, warp * 16, kf);
            load_a_frags(sV, warp * 16, vf);
        }
        const bf16* q_t = sQ + buf * FA_BLK * FA_HS;
        const bf16* do_t = sdO + buf * FA_BLK * FA_HS;
        const float* Ls = sL + buf * FA_BLK;
        const float* Ds = sD + buf * FA_BLK;

        // S^T = K Q^T ; P^T = exp(S^T * scale - lse_q)
        float pt[8][4];
        zero8x4(pt);
        mma_a_xt(pt, kf, q_t);
        const bool need_mask = (qb == kb) || ((qb + 1) * FA_BLK > T);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int ql = nt * 8 + 2 * t + (e & 1);
                int q = qb * FA_BLK + ql;
                int key = key0 + ((e >> 1) << 3);
                float p = exp2f(pt[nt][e] * sl2 - Ls[ql] * LOG2E);
                if (need_mask && (q < key || q >= T)) p = 0.f;
                pt[nt][e] = p;
            }
        }
        // dV += P^T dO
        mma_p_x(dv, pt, do_t);
        // dP^T = V dO^T ; dS^T = P^T (dP^T - D_q)
        float dpt[8][4];
        zero8x4(dpt);
        mma_a_xt(dpt, vf, do_t);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int ql = nt * 8 + 2 * t + (e & 1);
                dpt[nt][e] = pt[nt][e] * (dpt[nt][e] - Ds[ql]);
            }
        }
        // dK += dS^T Q
        mma_p_x(dk, dpt, q_t);
    }
    bf16* drow = dqkv + (int64_t)b * T * ld + h * FA_HS;
    store_acc(dk, drow + C, ld, kb * FA_BLK + warp * 16, T, scale);
    store_acc(dv, drow + 2 * C, ld, kb * FA_BLK + warp * 16, T, 1.f);
}

// dQ for 64 queries of one (b, h): loop over the key blocks they see.
__global__ void __launch_bounds__(FA_THREADS)
fa_bwd_dq_kernel(const bf16* __restrict__ qkv, const bf16* __restrict__ dout,
                 const float* __restrict__ lse, const float* __restrict__ D,
                 bf16* __restrict__ dqkv, int T, int H) {
    __shared__ __align__(128) bf16 sQ[FA_BLK * FA_HS];
    __shared__ __align__(128) bf16 sdO[FA_BLK * FA_HS];
    __shared__ __align__(128) bf16 sK[2][FA_BLK * FA_HS];
    __shared__ __align__(128) bf16 sV[2][FA_BLK * FA_HS];
    const int nqb = (T + FA_BLK - 1) / FA_BLK;
    const int qb = nqb - 1 - blockIdx.x;
    const int bh = blockIdx.y, h = bh % H, b = bh / H;
    const int C = H * FA_HS;
    const int64_t ld = 3 * C;
    const bf16* base = qkv + (int64_t)b * T * ld;
    const bf16* qg = base + h * FA_HS;
    const bf16* kg = base + C + h * FA_HS;
    const bf16* vg = base + 2 * C + h * FA_HS;
    const bf16* dog = dout + (int64_t)b * T * C + h * FA_HS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
    const float scale = 1.f / sqrtf((float)FA_HS);
    const float sl2 = LOG2E * scale;
    const int qrow0 = qb * FA_BLK + warp * 16 + gq;
    float Lr[2], Dr[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
        int q = qrow0 + 8 * r;
        Lr[r] = q < T ? lse[(int64_t)bh * T + q] * LOG2E : 0.f;
        Dr[r] = q < T ? D[(int64_t)bh * T + q] : 0.f;
    }

    load_tile(sQ, qg, ld, qb * FA_BLK, T);
    load_tile(sdO, dog, C, qb * FA_BLK, T);
    load_tile(sK[0], kg, ld, 0, T);
    load_tile(sV[0], vg, ld, 0, T);
    cp_commit();

    uint32_t qf[4][4], dof[4][4];
    float dq[8][4];
    zero8x4(dq);
    for (int kb = 0; kb <= qb; kb++) {
        const int buf = kb & 1;
        if (kb + 1 <= qb) {
            load_tile(sK[buf ^ 1], kg, ld, (kb + 1) * FA_BLK, T);
            load_tile(sV[buf ^ 1], vg, ld, (kb + 1) * FA_BLK, T);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        if (kb == 0) {
            load_a_frags(sQ, warp * 16, qf);
            load_a_frags(sdO, warp * 16, dof);
        }
        float p[8][4];
        zero8x4(p);
        mma_a_xt(p, qf, sK[buf]);
        const bool need_mask = (kb == qb) || ((kb + 1) * FA_BLK > T);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                int key = kb * FA_BLK + nt * 8 + 2 * t + (e & 1);
                int row = qrow0 + ((e >> 1) << 3);
                float v = exp2f(p[nt][e] * sl2 - Lr[e >> 1]);
                if (need_mask && (key > row || key >= T)) v = 0.f;
                p[nt][e] = v;
            }
        }
        float dp[8][4];
        zero8x4(dp);
        mma_a_xt(dp, dof, sV[buf]);
#pragma unroll
        for (int nt = 0; nt < 8; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) dp[nt][e] = p[nt][e] * (dp[nt][e] - Dr[e >> 1]);
        mma_p_x(dq, dp, sK[buf]);
        __syncthreads();
    }
    store_acc(dq, dqkv + (int64_t)b * T * ld + h * FA_HS, ld, qb * FA_BLK + warp * 16, T, scale);
}

bool attention_bf16_supported(int T, int hs) { return hs == FA_HS && T >= 1; }

cudaError_t attention_bwd_bf16(const bf16* qkv, const bf16* out, const float* lse,
                               const bf16* dout, bf16* dqkv, float* Dbuf, int B, int T, int H,
                               int hs, cudaStream_t s) {
    if (!attention_bf16_supported(T, hs)) return cudaErrorInvalidValue;
    int64_t n = (int64_t)B * T * H;
    fa_bwd_d_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(out, dout, Dbuf, B, T, H);
    CUDA_OK(cudaGetLastError());
    dim3 grid((T + FA_BLK - 1) / FA_BLK, B * H);
    size_t smem = (size_t)6 * FA_BLK * FA_HS * sizeof(bf16) + 4 * FA_BLK * sizeof(float);
    static bool attr = false;
    if (!attr) {
        CUDA_OK(cudaFuncSetAttribute(fa_bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem));
        attr = true;
    }
    fa_bwd_dkv_kernel<<<grid, FA_THREADS, smem, s>>>(qkv, dout, lse, Dbuf, dqkv, T, H);
    CUDA_OK(cudaGetLastError());
    fa_bwd_dq_kernel<<<grid, FA_THREADS, 0, s>>>(qkv, dout, lse, Dbuf, dqkv, T, H);
    return cudaGetLastError();
}

}  // namespace k
