// bf16 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   D[m,n] = sum_k A(m,k) B(n,k), fp32 accumulation in tensor memory (TMEM),
//   followed by a fused epilogue (bias, tanh-GELU, residual add, GELU
//   backward, fp32 gradient accumulation).
//
// Every Linear of the step maps onto this one routine (PyTorch layout
// W[out,in], nanoGPT guide Deep dive 1):
//   forward   y  = x W^T  : A = x  (K-major),  B = W (K-major)
//   backward  dx = dy W   : A = dy (K-major),  B = W viewed [in, out] (MN-major)
//   backward  dW += dy^T x: A = dy^T (MN-major), B = x^T (MN-major)
// so operands are consumed in either major order straight from memory.
//
// Structure: persistent CTAs (one per SM), 320 threads.
//   warp 0      TMA producer: 128B-swizzled tiles into a STAGES-deep ring
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=BN, K=16)
//               and tcgen05.commit to free ring slots / publish accumulators
//   warps 2..9  epilogue: two warps per TMEM lane quarter, each taking half
//               the columns: tcgen05.ld 32 at a time, fused math, stores
// Two TMEM accumulators (2*BN columns) let the epilogue of one tile overlap
// the main loop of the next. Every mbarrier wait is bounded: on expiry the
// CTA records ERR_TIMEOUT in the device status word, drains its in-flight
// copies and MMAs (again bounded), frees TMEM and returns.
#include "common.cuh"
#include "tc.cuh"
#include <cuda.h>

namespace k {

using namespace tc;

static constexpr int TC_BM = 128, TC_BK = 64;

// Grouped tile order: 16 m-tiles per group, m fastest inside a group, so a
// wave of CTAs shares A and B tiles through L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mt, int& nt) {
    const int G = 16;
    int group = t / (G * num_n);
    int first = group * G;
    int gm = min(num_m - first, G);
    int r = t - group * G * num_n;
    mt = first + r % gm;
    nt = r / gm;
}

// ------------------------------------------------------------------ epilogue
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(uint32_t*)&h;
}

// Hardware tanh (MUFU, max relative error about 2^-11): ample for values that
// are rounded to bf16 right after.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float gelu_hw(float x) {
    const float a = 0.7978845608028654f, c = 0.044715f;
    return 0.5f * x * (1.0f + tanh_hw(a * (x + c * x * x * x)));
}
__device__ __forceinline__ float gelu_grad_hw(float x) {
    const float a = 0.7978845608028654f, c = 0.044715f;
    float t = tanh_hw(a * (x + c * x * x * x));
    return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * a * (1.0f + 3.0f * c * x * x);
}

__device__ __forceinline__ void store_bf16_32(bf16* dst, const float (&v)[32]) {
    uint4* d = (uint4*)dst;
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        d[q] = w;
    }
}

// The epilogue works on 32 x 32 chunks per warp (32 TMEM lanes = rows, 32
// fp32 columns). The chunk is staged through a 4 KB per-warp shared-memory
// tile (16-byte groups XOR-swizzled by row, conflict-free both ways) so that
// the fused math and every global load/store run in a coalesced layout: lane
// l handles columns 4*(l%8)..+3 of rows l/8, l/8+4, ..., i.e. each warp
// instruction covers 4 rows x 32 columns.
__device__ __forceinline__ void stage_write(float* st, int lane, const uint32_t (&r)[32]) {
#pragma unroll
    for (int c = 0; c < 8; c++)
        *(uint4*)&st[lane * 32 + ((c ^ (lane & 7)) << 2)] =
            make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
}
__device__ __forceinline__ float4 stage_read(const float* st, int row, int q) {
    return *(const float4*)&st[row * 32 + ((q ^ (row & 7)) << 2)];
}

__device__ __forceinline__ uint2 pack4_bf16(float4 v) {
    return make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// Operand the epilogue reads besides the accumulator (residual fp32, GELU
// pre-activation bf16, or the fp32 gradient it accumulates into): for one
// chunk, lane l's 8 groups of 4 columns. Loaded one chunk ahead of its use.
struct AuxBuf {
    float4 f[8];
};

__device__ __forceinline__ void aux_load(const GemmEpi& e, int64_t m_base, int M, int n, int N,
                                         int rsub, AuxBuf& a) {
    const bool ncol = n < N;
    if (e.kind == EPI_RESID || e.kind == EPI_ACCUM_F32) {
        const float* src = (e.kind == EPI_RESID) ? (const float*)e.aux : (const float*)e.out;
        const int64_t ld = (e.kind == EPI_RESID) ? e.ld_aux : e.ldo;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int64_t m = m_base + it * 4 + rsub;
            a.f[it] = (ncol && m < M) ? *(const float4*)(src + m * ld + n) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else if (e.kind == EPI_GELU_BWD) {
        const bf16* src = (const bf16*)e.aux;
#pragma unroll
        for (int it = 0; it < 8; it++) {
            const int64_t m = m_base + it * 4 + rsub;
            uint2 w = (ncol && m < M) ? *(const uint2*)(src + m * e.ld_aux + n) : make_uint2(0u, 0u);
            a.f[it] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), 0.f, 0.f);
        }
    }
}

// Apply the epilogue to one staged chunk: rows m_base..m_base+31, columns
// n..n+3 for this lane (n = chunk start + 4*(lane%8)); N % 4 == 0.
__device__ __forceinline__ void epilogue_chunk(const GemmEpi& e, const float* st, int64_t m_base,
                                               int M, int n, int N, int rsub, int q,
                                               const AuxBuf& a, int64_t split_off) {
    if (n >= N) return;
    float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e.bias && e.kind != EPI_ACCUM_F32 && e.kind != EPI_GELU_BWD) bias = __ldg((const float4*)(e.bias + n));
#pragma unroll
    for (int it = 0; it < 8; it++) {
        const int row = it * 4 + rsub;
        const int64_t m = m_base + row;
        if (m >= M) continue;
        float4 v = stage_read(st, row, q);
        v.x += bias.x; v.y += bias.y; v.z += bias.z; v.w += bias.w;
        switch (e.kind) {
            case EPI_STORE_ACT:
                *(uint2*)((bf16*)e.out + m * e.ldo + n) = pack4_bf16(v);
                break;
            case EPI_GELU: {
                *(uint2*)((bf16*)e.out + m * e.ldo + n) = pack4_bf16(v);
                float4 g = make_float4(gelu_hw(v.x), gelu_hw(v.y), gelu_hw(v.z), gelu_hw(v.w));
                *(uint2*)((bf16*)e.out2 + m * e.ldo2 + n) = pack4_bf16(g);
                break;
            }
            case EPI_RESID:
            case EPI_ACCUM_F32: {
                const float4 r = a.f[it];
                v.x += r.x; v.y += r.y; v.z += r.z; v.w += r.w;
                *(float4*)((float*)e.out + m * e.ldo + n) = v;
                break;
            }
            case EPI_GELU_BWD: {
                const uint32_t w0 = __float_as_uint(a.f[it].x), w1 = __float_as_uint(a.f[it].y);
                float2 p0 = __bfloat1622float2(*(const __nv_bfloat162*)&w0);
                float2 p1 = __bfloat1622float2(*(const __nv_bfloat162*)&w1);
                v.x *= gelu_grad_hw(p0.x); v.y *= gelu_grad_hw(p0.y);
                v.z *= gelu_grad_hw(p1.x); v.w *= gelu_grad_hw(p1.y);
                *(uint2*)((bf16*)e.out + m * e.ldo + n) = pack4_bf16(v);
                break;
            }
            case EPI_STORE_F32:
                *(float4*)((float*)e.out + split_off + m * e.ldo + n) = v;
                break;
        }
    }
}

// ------------------------------------------------------------------ kernel
template <int BN, bool A_MN, bool B_MN>
struct TcCfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = BN * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int STAGING_BYTES = 8 * 32 * 32 * 4;   // 4 KB per epilogue warp
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + 256;
};

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(320, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               int M, int N, int K, int splits, GemmEpi epi, DevState* st) {
    using Cfg = TcCfg<BN, A_MN, B_MN>;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    float* staging = (float*)(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t* full = (uint64_t*)(smem + STAGES * Cfg::STAGE_BYTES + Cfg::STAGING_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = (uint32_t*)(drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_m = (M + TC_BM - 1) / TC_BM;
    const int num_n = (N + BN - 1) / BN;
    const int tiles = num_m * num_n;
    const int kblocks = (K + TC_BK - 1) / TC_BK;
    const int kpb = (kblocks + splits - 1) / splits;
    const int total = tiles * splits;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            long issued = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                int split = w / tiles, mt, nt;
                tile_coords(w - split * tiles, num_m, num_n, mt, nt);
                int kb0 = split * kpb, kb1 = min(kb0 + kpb, kblocks);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
                    uint8_t* a = sA + stage * Cfg::A_BYTES;
                    uint8_t* b = sB + stage * Cfg::B_BYTES;
                    const int k0 = kb * TC_BK;
                    if (!A_MN) {
                        tma_load_2d(a, &tmA, &full[stage], k0, mt * TC_BM);
                    } else {
                        tma_load_2d(a, &tmA, &full[stage], mt * TC_BM, k0);
                        tma_load_2d(a + 8192, &tmA, &full[stage], mt * TC_BM + 64, k0);
                    }
                    if (!B_MN) {
                        tma_load_2d(b, &tmB, &full[stage], k0, nt * BN);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; j++)
                            tma_load_2d(b + j * 8192, &tmB, &full[stage], nt * BN + 64 * j, k0);
                    }
                    issued++;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok || *abort_flag) {
                // drain: wait (bounded, ignoring the abort flag) for our last copies
                long first = issued > STAGES ? issued - STAGES : 0;
                for (long i = first; i < issued; i++) {
                    int s = (int)(i % STAGES);
                    uint32_t par = (uint32_t)((i / STAGES) & 1);
                    const long long t0 = wait_clock();
                    while (!mbar_try_wait(&full[s], par) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = make_idesc(TC_BM, BN, A_MN, B_MN);
            constexpr uint32_t A_LBO = A_MN ? 8192 : 16, B_LBO = B_MN ? 8192 : 16;
            constexpr uint32_t KSTEP_A = A_MN ? 2048 : 32, KSTEP_B = B_MN ? 2048 : 32;
            const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                int split = w / tiles;
                int kb0 = split * kpb, kb1 = min(kb0 + kpb, kblocks);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = sA0 + stage * Cfg::A_BYTES;
                    const uint32_t b_addr = sB0 + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; kk++) {
                        uint64_t ad = smem_desc(a_addr + kk * KSTEP_A, A_LBO, 1024);
                        uint64_t bd = smem_desc(b_addr + kk * KSTEP_B, B_LBO, 1024);
                        mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            if (any) {
                // all MMAs of this CTA complete before TMEM is released
                mma_commit(drain);
                const long long t0 = wait_clock();
                while (!mbar_try_wait(drain, 0) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
            }
        }
    } else {
        // ---------------- epilogue warps 2..9. TMEM lane quarter = warp % 4 (the
        // hardware's access rule); the two warps of a quarter split the columns.
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;
        constexpr int HCH = BN / 64;                 // 32-column chunks per half
        float* st_w = staging + (warp - 2) * 32 * 32;
        const int rsub = lane >> 3, qc = lane & 7;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int w = blockIdx.x; w < total; w += gridDim.x) {
            int split = w / tiles, mt, nt;
            tile_coords(w - split * tiles, num_m, num_n, mt, nt);
            const int64_t m_base = (int64_t)mt * TC_BM + q4 * 32;
            const int64_t split_off = (int64_t)split * M * N;
            const int nbase = nt * BN + half * HCH * 32;
            AuxBuf cur;
            aux_load(epi, m_base, M, nbase + 4 * qc, N, rsub, cur);   // overlaps the main loop
            bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < HCH; cc++) {
                const int c = half * HCH + cc;
                const int n0 = nt * BN + c * 32;
                AuxBuf nxt;
                if (cc + 1 < HCH) aux_load(epi, m_base, M, n0 + 32 + 4 * qc, N, rsub, nxt);
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                stage_write(st_w, lane, r);
                __syncwarp();
                epilogue_chunk(epi, st_w, m_base, M, n0 + 4 * qc, N, rsub, qc, cur, split_off);
                __syncwarp();
                if (cc + 1 < HCH) cur = nxt;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 1;
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// 2-D bf16 tensor map: `inner` contiguous elements per line, `outer` lines
// `ld` elements apart; boxes of box_inner x box_outer with 128B swizzle.
static bool make_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, int64_t ld,
                     uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool gemm_bf16_tc_supported(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi) {
    if (M <= 0 || N <= 0 || K <= 0) return false;
    if ((A.ld % 8) || (B.ld % 8)) return false;
    if (((uintptr_t)A.ptr | (uintptr_t)B.ptr) & 15) return false;
    if (epi.ldo % 8) return false;
    if (N % 4) return false;
    if (!get_encode()) return false;
    return true;
}

template <int BN, bool A_MN, bool B_MN>
static cudaError_t launch_tc(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                             int splits, DevState* st, cudaStream_t s) {
    using Cfg = TcCfg<BN, A_MN, B_MN>;
    CUtensorMap ta, tb;
    bool ok = A_MN ? make_map(&ta, A.ptr, (uint64_t)M, (uint64_t)K, A.ld, 64, 64)
                   : make_map(&ta, A.ptr, (uint64_t)K, (uint64_t)M, A.ld, 64, TC_BM);
    ok = ok && (B_MN ? make_map(&tb, B.ptr, (uint64_t)N, (uint64_t)K, B.ld, 64, 64)
                     : make_map(&tb, B.ptr, (uint64_t)K, (uint64_t)N, B.ld, 64, BN));
    if (!ok) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        CUDA_OK(cudaFuncSetAttribute(gemm_tc_kernel<BN, A_MN, B_MN>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM));
        attr_set = true;
    }
    const int tiles = ((M + TC_BM - 1) / TC_BM) * ((N + BN - 1) / BN);
    const int total = tiles * splits;
    const int grid = total < num_sms() ? total : num_sms();
    gemm_tc_kernel<BN, A_MN, B_MN><<<grid, 320, Cfg::SMEM, s>>>(ta, tb, M, N, K, splits, epi, st);
    return cudaGetLastError();
}

cudaError_t gemm_bf16_tc(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                         int splits, DevState* st, cudaStream_t s) {
    if (!gemm_bf16_tc_supported(M, N, K, A, B, epi)) return cudaErrorInvalidValue;
    const int kblocks = (K + TC_BK - 1) / TC_BK;
    if (splits < 1) splits = 1;
    if (splits > kblocks) splits = kblocks;
    if (splits > 1) {
        // every split must own at least one k-block
        int kpb = (kblocks + splits - 1) / splits;
        splits = (kblocks + kpb - 1) / kpb;
        if (epi.kind != EPI_STORE_F32 || epi.bias) return cudaErrorInvalidValue;
        if (epi.ldo != N) return cudaErrorInvalidValue;
    }
    const bool a_mn = !A.kmajor, b_mn = !B.kmajor;
    const bool wide = (N % 256 == 0) || N > 2048;
#define TC_CASE(BNV, AM, BM_)                                                   \
    if (a_mn == AM && b_mn == BM_)                                              \
        return launch_tc<BNV, AM, BM_>(M, N, K, A, B, epi, splits, st, s);
    if (wide) {
        TC_CASE(256, false, false)
        TC_CASE(256, false, true)
        TC_CASE(256, true, false)
        TC_CASE(256, true, true)
    } else {
        TC_CASE(128, false, false)
        TC_CASE(128, false, true)
        TC_CASE(128, true, false)
        TC_CASE(128, true, true)
    }
#undef TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace k
