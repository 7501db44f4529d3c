// Causal flash attention forward on the 5th-generation tensor cores (tcgen05,
// sm_103a): bf16 q, k, v, fp32 scores and output accumulation in tensor memory.
//
// Semantics: the manual attention of nanoGPT's CausalSelfAttention (nanoGPT
// guide Deep dive 1): S = q k^T / sqrt(hs), keys j > i masked to -inf before
// the softmax, o = softmax(S) v; the T x T scores never leave the chip (online
// softmax over key blocks: "Let's reproduce GPT-2" 02:00:18, Flash Attention).
// Also writes lse = log sum_j exp(S_ij) per query for the backward.
//
// Work item = (128-query block, b, h); persistent CTAs, 192 threads:
//   warps 0..3  softmax: one thread per query row (= its TMEM lane). Reads the
//               row of S from TMEM, masks, tracks the running max, writes
//               P = exp(S - max) in bf16 back to TMEM, where the P V product
//               reads it as its A operand (keeping P out of shared memory,
//               whose bandwidth the S and P V operand reads and the K/V
//               copies already use up), rescales the O row in TMEM when the max grew
//               by more than 2^8 (otherwise P may exceed 1 by up to 2^8, which
//               the final division by the row sum absorbs exactly). The item's
//               O / l leaves through a 4 KB shared-memory slab per warp and one
//               TMA store (per-lane row stores cost 14% of the kernel).
//   warp 4      TMA producer: Q once per item, then K and V of each block of
//               128 keys into one slot of a three-slot ring.
//   warp 5      allocates 512 TMEM columns (S double buffer, O double buffer,
//               P double buffer); lane 0 issues S_j = Q K_j^T (M=128, N=128,
//               K=64) into S[j%2].
//   warp 6      lane 0 issues O += P_j V_j (M=128, N=64, K=128; A = P from
//               TMEM), so the tensor core computes S_{j+1} and P_j V_j while
//               the softmax works on S_{j+1}.
// Every mbarrier wait is bounded; on expiry the CTA records ERR_TIMEOUT,
// drains its copies and MMAs (bounded), frees TMEM and returns.
#include "common.cuh"
#include "tc.cuh"
#include <cuda.h>
#include <cstring>

namespace k {

using namespace tc;

namespace {

constexpr int AT_BQ = 128;                     // queries per CTA
constexpr int AT_BK = 128;                     // keys per block
constexpr int AT_HS = 64;                      // head size
constexpr int AT_SLOTS = 3;                    // K and V ring depth
constexpr int AT_TILE = AT_BQ * AT_HS * 2;     // 16 KB: 128 rows x 128 B
constexpr int FW_THREADS = 224;                // forward: 4 softmax warps, producer, two MMA issuers
constexpr int OFF_Q = 0;                       // Q double buffer
constexpr int OFF_K = OFF_Q + 2 * AT_TILE;
constexpr int OFF_V = OFF_K + AT_SLOTS * AT_TILE;
constexpr int OUT_SLAB = 32 * AT_HS * 2;       // one warp's 32 output rows, 4 KB
constexpr int OFF_OUT = OFF_V + AT_SLOTS * AT_TILE;   // [4 softmax warps] O slabs
constexpr int OFF_BAR = OFF_OUT + 4 * OUT_SLAB;
constexpr size_t AT_SMEM = OFF_BAR + 256 + 1024;
// forward TMEM columns: S[0] 0..127, S[1] 128..255, O[0] 256..319, O[1]
// 320..383, P[0] 384..447, P[1] 448..511 (P: bf16 pairs, the A operand of P V)
constexpr uint32_t TM_O = 256, TM_P = 384;
constexpr uint32_t AT_TMEM_COLS = 512;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(uint32_t*)&h;
}
__device__ __forceinline__ void wait_bounded(uint64_t* bar, uint32_t parity) {
    const long long t0 = wait_clock();
    while (!mbar_try_wait(bar, parity) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
}
// max(a, b, c) in one instruction (three-input max.f32, sm_100 family)
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// A warp's 32 rows x 64 columns of an output tile (fp32 accumulator values
// times `scale`) as bf16 into a 128B-swizzled 4 KB slab: lane = row, 16-byte
// piece q of row r at r*128 + ((q ^ (r & 7)) << 4), the layout the TMA store
// of a 64 x 32 box expects.
__device__ __forceinline__ void stage_out_slab(uint8_t* slab, int lane, const uint32_t (&a)[64], float scale) {
#pragma unroll
    for (int q = 0; q < 8; q++) {
        const float* f = (const float*)&a[8 * q];
        *(uint4*)(slab + lane * 128 + ((q ^ (lane & 7)) << 4)) =
            make_uint4(pack2_bf16(f[0] * scale, f[1] * scale), pack2_bf16(f[2] * scale, f[3] * scale),
                       pack2_bf16(f[4] * scale, f[5] * scale), pack2_bf16(f[6] * scale, f[7] * scale));
    }
}

}  // namespace

// Persistent: one CTA per SM walks work items w = blockIdx.x, +gridDim.x, ...
// ordered heaviest first (query block qb = nqb-1 - w / (B*H)). Barrier phases
// run on counters that every role advances identically: g counts key blocks
// over all items (K/V ring slots, S and P buffers), `it` counts items (Q and O
// double buffers), so the next item's Q, K and V load and its first S product
// runs while the softmax warps finish the previous item. Two threads issue the
// tensor-core work, one the S products and one the P V products, so that
// neither chain of barrier waits delays the other.
__global__ void __launch_bounds__(FW_THREADS, 1)
fa_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_out,
                 float* __restrict__ lse, int T, int H, int BH, DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + OFF_Q;
    uint8_t* sK = smem + OFF_K;
    uint8_t* sV = smem + OFF_V;
    uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
    uint64_t* q_full = bars;           // [2]
    uint64_t* q_empty = bars + 2;      // [2]
    uint64_t* kv_full = bars + 4;      // [3] K and V block j
    uint64_t* kv_empty = bars + 7;     // [3]
    uint64_t* s_full = bars + 10;      // [2]
    uint64_t* s_empty = bars + 12;
    uint64_t* p_full = bars + 14;
    uint64_t* pv_done = bars + 16;
    uint64_t* o_free = bars + 18;      // [2]
    uint64_t* drain = bars + 20;       // [2] one per issuing thread
    uint32_t* tmem_slot = (uint32_t*)(bars + 22);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nqb = (T + AT_BQ - 1) / AT_BQ;
    const int items = nqb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
            mbar_init(&o_free[i], 4);
            mbar_init(&drain[i], 1);
        }
        for (int s = 0; s < AT_SLOTS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 4) {
        if (lane == 0) {
            // ---------------- TMA producer
            int g = 0, it = 0, nq = 0, nkv_l = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH, bh = w % BH, h = bh % H, b = bh / H;
                const int nkv = qb + 1;
                const int qs = it & 1;
                if (!mbar_wait(&q_empty[qs], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&q_full[qs], AT_TILE);
                tma_load_3d(sQ + qs * AT_TILE, &tm_qkv, &q_full[qs], h * AT_HS, qb * AT_BQ, b);
                nq++;
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % AT_SLOTS;
                    if (!mbar_wait(&kv_empty[s], (uint32_t)(((G / AT_SLOTS) & 1) ^ 1), abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&kv_full[s], 2 * AT_TILE);
                    tma_load_3d(sK + s * AT_TILE, &tm_qkv, &kv_full[s], C + h * AT_HS, j * AT_BK, b);
                    tma_load_3d(sV + s * AT_TILE, &tm_qkv, &kv_full[s], 2 * C + h * AT_HS, j * AT_BK, b);
                    nkv_l++;
                }
                g += nkv;
            }
            if (!ok || *abort_flag) {
                // wait (bounded) for every copy still in flight before the CTA exits
                for (int i = (nq > 2 ? nq - 2 : 0); i < nq; i++) wait_bounded(&q_full[i & 1], (uint32_t)((i >> 1) & 1));
                for (int i = (nkv_l > AT_SLOTS ? nkv_l - AT_SLOTS : 0); i < nkv_l; i++)
                    wait_bounded(&kv_full[i % AT_SLOTS], (uint32_t)((i / AT_SLOTS) & 1));
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ---------------- S = Q K^T issuer
            constexpr uint32_t id_s = make_idesc(AT_BQ, AT_BK, false, false);
            const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024), dk0 = smem_desc(smem_u32(sK), 16, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH;
                const int nkv = qb + 1;
                const int qs = it & 1;
                if (!mbar_wait(&q_full[qs], (uint32_t)((it >> 1) & 1), abort_flag)) { ok = false; break; }
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % AT_SLOTS, sb = G & 1;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / AT_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&s_empty[sb], (uint32_t)(((G >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dq = desc_adv(dq0, qs * AT_TILE), dk = desc_adv(dk0, s * AT_TILE);
#pragma unroll
                    for (int kk = 0; kk < AT_HS / 16; kk++)
                        mma_bf16(tmem_base + (uint32_t)(sb * AT_BK), desc_adv(dq, 32 * kk), desc_adv(dk, 32 * kk),
                                 id_s, kk > 0 ? 1u : 0u);
                    mma_commit(&s_full[sb]);
                    if (j == nkv - 1) mma_commit(&q_empty[qs]);
                    any = true;
                }
                g += nkv;
            }
            if (any) {
                mma_commit(&drain[0]);
                wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == 6) {
        if (lane == 0) {
            // ---------------- O += P V issuer (P read from TMEM, V MN-major)
            constexpr uint32_t id_o = make_idesc(AT_BQ, AT_HS, false, true);
            const uint64_t dv0 = smem_desc(smem_u32(sV), 8192, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH;
                const int nkv = qb + 1;
                const int ob = it & 1;
                if (!mbar_wait(&o_free[ob], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % AT_SLOTS, pb = G & 1;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / AT_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&p_full[pb], (uint32_t)((G >> 1) & 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dv = desc_adv(dv0, s * AT_TILE);
                    const uint32_t tp = tmem_base + TM_P + pb * (AT_BK / 2);
#pragma unroll
                    for (int kk = 0; kk < AT_BK / 16; kk++)
                        mma_bf16_ta(tmem_base + TM_O + ob * AT_HS, tp + kk * 8, desc_adv(dv, kk * 2048), id_o,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&pv_done[pb]);
                    mma_commit(&kv_empty[s]);
                    any = true;
                }
                g += nkv;
            }
            if (any) {
                mma_commit(&drain[1]);
                wait_bounded(&drain[1], 0);
            }
        }
    } else {
        // ---------------- softmax warps 0..3: thread r owns query row r (TMEM lane r)
        const int r = threadIdx.x;
        const float sl2 = 1.4426950408889634f * 0.125f;   // log2(e) / sqrt(64)
        const uint32_t lane_base = tmem_base + ((uint32_t)(warp * 32) << 16);
        uint8_t* slab = smem + OFF_OUT + warp * OUT_SLAB;
        bool ok = true;
        int g = 0, it = 0;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int qb = nqb - 1 - w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int nkv = qb + 1;
            const int q = qb * AT_BQ + r;
            const int ob = it & 1;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nkv; j++) {
                const int G = g + j, sb = G & 1;
                ok = mbar_wait(&s_full[sb], (uint32_t)((G >> 1) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[128];
#pragma unroll
                for (int c = 0; c < 4; c++) tmem_ld32_nowait(lane_base + (uint32_t)(sb * AT_BK + 32 * c), sr + 32 * c);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                // mask (raw scores; the scale is applied in the exponent), row max
                // as eight independent partial maxima
                const int key0 = j * AT_BK;
                const bool edge = (j == qb) || (key0 + AT_BK > T);
                if (edge) {
#pragma unroll
                    for (int i = 0; i < 128; i++)
                        if (key0 + i > q || key0 + i >= T) sr[i] = __float_as_uint(-INFINITY);
                }
                float pm[8];
#pragma unroll
                for (int t = 0; t < 8; t++) pm[t] = __uint_as_float(sr[t]);
#pragma unroll
                for (int i = 8; i < 120; i += 16)
#pragma unroll
                    for (int t = 0; t < 8; t++)
                        pm[t] = fmax3f(pm[t], __uint_as_float(sr[i + t]), __uint_as_float(sr[i + 8 + t]));
#pragma unroll
                for (int t = 0; t < 8; t++) pm[t] = fmaxf(pm[t], __uint_as_float(sr[120 + t]));
                const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                       fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * sl2;
                const float m_new = fmaxf(m_run, mx);
                const bool resc = (j > 0) && (m_new > m_run + 8.f);
                if (j == 0) m_run = m_new;
                if (__any_sync(0xffffffffu, resc)) {
                    // rescale the O row once the previous P V product has landed
                    ok = mbar_wait(&pv_done[(G - 1) & 1], (uint32_t)(((G - 1) >> 1) & 1), abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    const float f = resc ? ex2f(m_run - m_new) : 1.f;
                    const uint32_t oaddr = lane_base + TM_O + ob * AT_HS;
                    uint32_t o[64];
                    tmem_ld32_nowait(oaddr, o);
                    tmem_ld32_nowait(oaddr + 32, o + 32);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 64; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                    tmem_st32(oaddr, o);
                    tmem_st32(oaddr + 32, o + 32);
                    if (resc) {
                        l_run *= f;
                        m_run = m_new;
                    }
                }
                // the P buffer is free once the product that read it (two blocks ago) is done
                if (G >= 2) {
                    ok = mbar_wait(&pv_done[sb], (uint32_t)(((G - 2) >> 1) & 1), abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                }
                float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                const uint32_t prow = lane_base + TM_P + sb * (AT_BK / 2);
#pragma unroll
                for (int hf = 0; hf < 2; hf++) {
                    uint32_t pk[32];                    // 64 probabilities as bf16 pairs
#pragma unroll
                    for (int c = 0; c < 32; c++) {
                        const float e0 = ex2f(fmaf(__uint_as_float(sr[hf * 64 + 2 * c]), sl2, -m_run));
                        const float e1 = ex2f(fmaf(__uint_as_float(sr[hf * 64 + 2 * c + 1]), sl2, -m_run));
                        ps[(2 * c) & 7] += e0;
                        ps[(2 * c + 1) & 7] += e1;
                        pk[c] = pack2_bf16(e0, e1);
                    }
                    tmem_st32(prow + 32 * hf, pk);
                }
                l_run += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
            }
            if (!ok) break;
            // the item's output: O / l and lse, once its last P V product is done
            const int GL = g + nkv - 1;
            ok = mbar_wait(&pv_done[GL & 1], (uint32_t)((GL >> 1) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t o[64];
            tmem_ld32_nowait(lane_base + TM_O + ob * AT_HS, o);
            tmem_ld32_nowait(lane_base + TM_O + ob * AT_HS + 32, o + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&o_free[ob]);
                tma_wait_read<0>();             // the previous item's store has read the slab
            }
            __syncwarp();
            // O / l through this warp's slab and one TMA store (rows beyond T clipped)
            stage_out_slab(slab, lane, o, 1.f / l_run);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&tm_out, slab, h * AT_HS, qb * AT_BQ + warp * 32, b);
                tma_commit();
            }
            if (q < T) lse[(int64_t)bh * T + q] = (m_run + log2f(l_run)) * LN2;
            g += nkv;
        }
        if (lane == 0) tma_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 3;
    }
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem_base, AT_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFnA)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnA encode_fn() {
    static EncodeTiledFnA fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFnA)p;
    }
    return fn;
}

// qkv [B, T, 3C] bf16 as a 3-D map {3C, T, B}: rows beyond T of a sequence
// read as zeros (never the next sequence's rows). Boxes of 64 x 128 x 1 with
// 128B swizzle: the K-major operand layout of the tcgen05 descriptors.
static bool make_qkv_map(CUtensorMap* map, const bf16* qkv, int B, int T, int C) {
    EncodeTiledFnA enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)3 * C * 2 * T};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(qkv), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [B, T, width] bf16 tensor as the target of per-warp output stores: 3-D map
// {width, T, B}, boxes of 64 x 32 x 1 with 128B swizzle (rows beyond T clipped).
static bool make_rows_out_map(CUtensorMap* map, bf16* ptr, int B, int T, int width) {
    EncodeTiledFnA enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * T};
    cuuint32_t box[3] = {64, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t attention_fwd_bf16(const bf16* qkv, bf16* out, float* lse, int B, int T, int H, int hs,
                               DevState* st, cudaStream_t s) {
    if (hs != AT_HS || T < 1 || B < 1 || H < 1 || !st) return cudaErrorInvalidValue;
    if (((uintptr_t)qkv & 15) || ((uintptr_t)out & 15)) return cudaErrorInvalidValue;
    CUtensorMap map, omap;
    memset(&map, 0, sizeof map);
    memset(&omap, 0, sizeof omap);
    if (!make_qkv_map(&map, qkv, B, T, H * hs) || !make_rows_out_map(&omap, out, B, T, H * hs))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        CUDA_OK(cudaFuncSetAttribute(fa_tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AT_SMEM));
        attr_done.fetch_or(dbit);
    }
    const int items = ((T + AT_BQ - 1) / AT_BQ) * B * H;
    const int grid = items < num_sms() ? items : num_sms();
    fa_tc_fwd_kernel<<<grid, FW_THREADS, AT_SMEM, s>>>(map, omap, lse, T, H, B * H, st);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ backward
// Deterministic (no atomics) backward in two kernels; the probabilities are
// recomputed from the forward's lse; the dQ kernel (run first) also computes
// D = rowsum(dO * O) per query row and stores it for the dK/dV kernel.
// With s the raw score q.k, p = exp(s/sqrt(hs) - lse), dP = dO V^T,
// dS = P * (dP - D) (the gradient of the scaled scores):
//   dK = dS^T Q / sqrt(hs), dV = P^T dO   (work item: one 128-key block)
//   dQ = dS K / sqrt(hs)                  (work item: one 128-query block)
// Both kernels keep the two 128x128 products (S and dP, or their transposes)
// in TMEM, write the bf16 operands of the accumulating products (P^T and
// dS^T, or dS) to shared memory in the K-major 128B-swizzled layout, and
// accumulate dK, dV (or dQ) in TMEM across the blocks of the other operand.

namespace {

constexpr int BW_THREADS = 352;                 // 8 softmax warps, producer, two MMA issuers
constexpr int BW_PRODUCER = 8, BW_ISSUE_A = 9, BW_ISSUE_B = 10;
constexpr int BW_SLOTS = 3;
// dK/dV kernel: K and V double buffered per item, Q and dO in a 3-slot ring,
// per-warp staging of the dK and dV rows for their TMA stores
constexpr int KV_OFF_K = 0;                                  // [2]
constexpr int KV_OFF_V = KV_OFF_K + 2 * AT_TILE;             // [2]
constexpr int KV_OFF_Q = KV_OFF_V + 2 * AT_TILE;             // [3]
constexpr int KV_OFF_DO = KV_OFF_Q + BW_SLOTS * AT_TILE;     // [3]
constexpr int KV_OFF_OUT = KV_OFF_DO + BW_SLOTS * AT_TILE;   // [8 warps] dK or dV slab
constexpr int KV_OFF_LD = KV_OFF_OUT + 8 * OUT_SLAB;         // [3 slots] lse2[128], D[128]
constexpr int KV_OFF_BAR = KV_OFF_LD + BW_SLOTS * 2 * 128 * 4;
constexpr size_t KV_SMEM = KV_OFF_BAR + 256 + 1024;
// dQ kernel: Q and dO double buffered per item, K and V in a 3-slot ring
constexpr int DQ_OFF_Q = 0;                                  // [2]
constexpr int DQ_OFF_DO = DQ_OFF_Q + 2 * AT_TILE;            // [2]
constexpr int DQ_OFF_K = DQ_OFF_DO + 2 * AT_TILE;            // [3]
constexpr int DQ_OFF_V = DQ_OFF_K + BW_SLOTS * AT_TILE;      // [3]
constexpr int DQ_OFF_OUT = DQ_OFF_V + BW_SLOTS * AT_TILE;    // [4 quarters] dQ slabs
constexpr int DQ_OFF_O = DQ_OFF_OUT + 4 * OUT_SLAB;          // [2] forward output tile (for D)
constexpr int DQ_OFF_BAR = DQ_OFF_O + 2 * AT_TILE;
constexpr size_t DQ_SMEM = DQ_OFF_BAR + 256 + 1024;
// TMEM columns. dK/dV: S^T 0..127, dP^T 128..255, dV 256..319, dK 320..383,
// P^T 384..447 and dS^T 448..511 (bf16 pairs, the A operands of dV and dK).
// dQ: S 0..127, dP 128..255, dQ[2] 256..383, dS 384..447.
constexpr uint32_t TM_S = 0, TM_DP = 128, TM_ACC = 256, TM_PT = 384, TM_DST = 448;
constexpr float LOG2E_F = 1.4426950408889634f;


}  // namespace

// Persistent like the forward: work items (key block kb, b, h), fewest key
// blocks last (kb = w / (B*H)); g counts query blocks over all items, `it`
// counts items. Warp 9 issues S^T = K Q^T and dP^T = V dO^T, warp 10 the
// accumulating dV += P^T dO and dK += dS^T Q with P^T, dS^T read from TMEM;
// warp 8 loads; warps 0..7 compute P^T and dS^T, two warps per TMEM lane
// quarter (no row reductions are needed here, so the columns split freely).
__global__ void __launch_bounds__(BW_THREADS, 1)
fa_tc_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ lse,
                     const float* __restrict__ Dg, int T, int H, int BH, DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sK = smem + KV_OFF_K;
    uint8_t* sV = smem + KV_OFF_V;
    uint8_t* sQ = smem + KV_OFF_Q;
    uint8_t* sDO = smem + KV_OFF_DO;
    uint8_t* sOut = smem + KV_OFF_OUT;
    float* sLD = (float*)(smem + KV_OFF_LD);         // [3][lse (log2 units) 128, D 128]
    uint64_t* bars = (uint64_t*)(smem + KV_OFF_BAR);
    uint64_t* kv_full = bars;                          // [2]
    uint64_t* kv_empty = bars + 2;                     // [2]
    uint64_t* qd_full = bars + 4;                      // [3]
    uint64_t* qd_empty = bars + 7;                     // [3]
    uint64_t* st_full = bars + 10;
    uint64_t* st_free = bars + 11;
    uint64_t* ps_full = bars + 12;
    uint64_t* ps_free = bars + 13;
    uint64_t* acc_full = bars + 14;
    uint64_t* acc_free = bars + 15;
    uint64_t* ld_full = bars + 16;                     // [3] lse/D of the Q/dO slot staged
    uint64_t* drain = bars + 19;                       // [2]
    uint32_t* tmem_slot = (uint32_t*)(bars + 21);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nb = (T + AT_BK - 1) / AT_BK;
    const int items = nb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&drain[i], 1);
        }
        for (int s = 0; s < BW_SLOTS; s++) {
            mbar_init(&qd_full[s], 1);
            mbar_init(&qd_empty[s], 1);
            mbar_init(&ld_full[s], 1);
        }
        mbar_init(st_full, 1);
        mbar_init(st_free, 8);
        mbar_init(ps_full, 8);
        mbar_init(ps_free, 1);
        mbar_init(acc_full, 1);
        mbar_init(acc_free, 8);
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == BW_ISSUE_A) tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == BW_PRODUCER) {
        // ---------------- producer warp: lane 0 issues the TMA copies; all lanes stage
        // the lse (log2 units) and D values of each query block beside its Q/dO slot
        int g = 0, it = 0, nkvl = 0, nql = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int kb = w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int n = nb - kb;
            const int ks = it & 1;
            if (lane == 0) {
                ok = mbar_wait(&kv_empty[ks], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag);
                if (ok) {
                    mbar_arrive_expect_tx(&kv_full[ks], 2 * AT_TILE);
                    tma_load_3d(sK + ks * AT_TILE, &tm_qkv, &kv_full[ks], C + h * AT_HS, kb * AT_BK, b);
                    tma_load_3d(sV + ks * AT_TILE, &tm_qkv, &kv_full[ks], 2 * C + h * AT_HS, kb * AT_BK, b);
                    nkvl++;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
            for (int i = 0; i < n; i++) {
                const int G = g + i, qs = G % BW_SLOTS;
                const int q0 = (kb + i) * AT_BQ;
                ok = mbar_wait(&qd_empty[qs], (uint32_t)(((G / BW_SLOTS) & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&qd_full[qs], 2 * AT_TILE);
                    tma_load_3d(sQ + qs * AT_TILE, &tm_qkv, &qd_full[qs], h * AT_HS, q0, b);
                    tma_load_3d(sDO + qs * AT_TILE, &tm_do, &qd_full[qs], h * AT_HS, q0, b);
                    nql++;
                }
                float* ldst = sLD + qs * 256;
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int qq = u * 32 + lane, q = q0 + qq;
                    ldst[qq] = q < T ? lse[(int64_t)bh * T + q] * LOG2E_F : INFINITY;
                    ldst[128 + qq] = q < T ? Dg[(int64_t)bh * T + q] : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ld_full[qs]);
            }
            g += n;
        }
        if (lane == 0 && (!ok || *abort_flag)) {
            for (int i = (nkvl > 2 ? nkvl - 2 : 0); i < nkvl; i++) wait_bounded(&kv_full[i & 1], (uint32_t)((i >> 1) & 1));
            for (int i = (nql > BW_SLOTS ? nql - BW_SLOTS : 0); i < nql; i++)
                wait_bounded(&qd_full[i % BW_SLOTS], (uint32_t)((i / BW_SLOTS) & 1));
        }
    } else if (warp == BW_ISSUE_A) {
        if (lane == 0) {
            // ---------------- S^T = K Q^T, dP^T = V dO^T (M = keys, N = queries, K = head dim)
            constexpr uint32_t id_s = make_idesc(AT_BK, AT_BQ, false, false);
            const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 1024), dv0 = smem_desc(smem_u32(sV), 16, 1024),
                           dq0 = smem_desc(smem_u32(sQ), 16, 1024), ddo0 = smem_desc(smem_u32(sDO), 16, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int n = nb - w / BH;
                const int ks = it & 1;
                if (!mbar_wait(&kv_full[ks], (uint32_t)((it >> 1) & 1), abort_flag)) { ok = false; break; }
                const uint64_t dk = desc_adv(dk0, ks * AT_TILE), dv = desc_adv(dv0, ks * AT_TILE);
                for (int i = 0; i < n; i++) {
                    const int G = g + i, qs = G % BW_SLOTS;
                    if (!mbar_wait(&qd_full[qs], (uint32_t)((G / BW_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(st_free, (uint32_t)((G & 1) ^ 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dq = desc_adv(dq0, qs * AT_TILE), ddo = desc_adv(ddo0, qs * AT_TILE);
#pragma unroll
                    for (int kk = 0; kk < AT_HS / 16; kk++) {
                        mma_bf16(tmem_base + TM_S, desc_adv(dk, 32 * kk), desc_adv(dq, 32 * kk), id_s, kk > 0 ? 1u : 0u);
                        mma_bf16(tmem_base + TM_DP, desc_adv(dv, 32 * kk), desc_adv(ddo, 32 * kk), id_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(st_full);
                    if (i == n - 1) mma_commit(&kv_empty[ks]);
                    any = true;
                }
                g += n;
            }
            if (any) {
                mma_commit(&drain[0]);
                wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == BW_ISSUE_B) {
        if (lane == 0) {
            // ---------------- dV += P^T dO, dK += dS^T Q (A from TMEM; dO, Q read MN-major)
            constexpr uint32_t id_a = make_idesc(AT_BK, AT_HS, false, true);
            const uint64_t dqm0 = smem_desc(smem_u32(sQ), 8192, 1024), ddom0 = smem_desc(smem_u32(sDO), 8192, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int n = nb - w / BH;
                if (!mbar_wait(acc_free, (uint32_t)((it & 1) ^ 1), abort_flag)) { ok = false; break; }
                for (int i = 0; i < n; i++) {
                    const int G = g + i, qs = G % BW_SLOTS;
                    if (!mbar_wait(&qd_full[qs], (uint32_t)((G / BW_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(ps_full, (uint32_t)(G & 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dqm = desc_adv(dqm0, qs * AT_TILE), ddom = desc_adv(ddom0, qs * AT_TILE);
#pragma unroll
                    for (int kk = 0; kk < AT_BQ / 16; kk++) {
                        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                        mma_bf16_ta(tmem_base + TM_ACC, tmem_base + TM_PT + kk * 8, desc_adv(ddom, kk * 2048), id_a, acc);
                        mma_bf16_ta(tmem_base + TM_ACC + AT_HS, tmem_base + TM_DST + kk * 8, desc_adv(dqm, kk * 2048),
                                    id_a, acc);
                    }
                    mma_commit(ps_free);
                    mma_commit(&qd_empty[qs]);
                    if (i == n - 1) mma_commit(acc_full);
                    any = true;
                }
                g += n;
            }
            if (any) {
                mma_commit(&drain[1]);
                wait_bounded(&drain[1], 0);
            }
        }
    } else {
        // ---------------- warps 0..7: warp w reads TMEM lane quarter w % 4 (thread
        // row r = its lane there: key row r) and query columns 64*(w/4)..+63
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = q4 * 32 + lane;
        const float sl2 = LOG2E_F * 0.125f;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q4 * 32) << 16);
        uint8_t* slab = sOut + warp * OUT_SLAB;            // dK (hf 0) or dV (hf 1) of these 32 rows
        bool ok = true;
        int g = 0, it = 0;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int kb = w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int n = nb - kb;
            for (int i = 0; i < n; i++) {
                const int G = g + i, qs = G % BW_SLOTS;
                ok = mbar_wait(&ld_full[qs], (uint32_t)((G / BW_SLOTS) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ok = mbar_wait(st_full, (uint32_t)(G & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                // P^T / dS^T in TMEM are free once the previous block's products read them
                ok = mbar_wait(ps_free, (uint32_t)((G & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const float* L = sLD + qs * 256;
                const float* Dq = L + 128;
#pragma unroll 1
                for (int c = 2 * hf; c < 2 * hf + 2; c++) {
                    uint32_t sr[32], dr[32];
                    tmem_ld32_nowait(lane_base + TM_S + 32 * c, sr);
                    tmem_ld32_nowait(lane_base + TM_DP + 32 * c, dr);
                    tmem_wait_ld();
                    if (c == 2 * hf + 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(st_free);
                    }
                    uint32_t pp[16], pd[16];
#pragma unroll
                    for (int t4 = 0; t4 < 8; t4++) {
                        const float4 l4 = *(const float4*)&L[32 * c + 4 * t4];     // broadcast reads
                        const float4 d4 = *(const float4*)&Dq[32 * c + 4 * t4];
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                        float p[4], d[4];
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const int qq = 32 * c + 4 * t4 + u;
                            float e = ex2f(fmaf(__uint_as_float(sr[4 * t4 + u]), sl2, -lv[u]));
                            if (i == 0 && qq < r) e = 0.f;          // query before key: masked
                            p[u] = e;
                            d[u] = e * (__uint_as_float(dr[4 * t4 + u]) - dv4[u]);
                        }
                        pp[2 * t4] = pack2_bf16(p[0], p[1]);
                        pp[2 * t4 + 1] = pack2_bf16(p[2], p[3]);
                        pd[2 * t4] = pack2_bf16(d[0], d[1]);
                        pd[2 * t4 + 1] = pack2_bf16(d[2], d[3]);
                    }
                    tmem_st16(lane_base + TM_PT + 16 * c, pp);
                    tmem_st16(lane_base + TM_DST + 16 * c, pd);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ps_full);
            }
            if (!ok) break;
            // the item's dK, dV rows: out of TMEM, staged, one TMA store per warp and tensor
            ok = mbar_wait(acc_full, (uint32_t)(it & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // lower-half warps take dK (TMEM columns 320..383), upper-half ones dV (256..319)
            uint32_t acc[64];
            const uint32_t tacc = lane_base + TM_ACC + (hf == 0 ? AT_HS : 0);
            tmem_ld32_nowait(tacc, acc);
            tmem_ld32_nowait(tacc + 32, acc + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            if (lane == 0) tma_wait_read<0>();               // the previous item's store has read the slab
            __syncwarp();
            stage_out_slab(slab, lane, acc, hf == 0 ? 0.125f : 1.f);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int row0 = kb * AT_BK + q4 * 32;
                if (row0 < T) tma_store_3d(&tm_out, slab, (hf == 0 ? C : 2 * C) + h * AT_HS, row0, b);
                tma_commit();
            }
            g += n;
        }
        if (lane == 0) tma_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 4;
    }
    if (warp == BW_ISSUE_A) {
        tc_fence_after();
        tmem_dealloc(tmem_base, AT_TMEM_COLS);
    }
}

// Persistent: work items (query block qb, b, h), heaviest first. Warp 9 issues
// S = Q K^T and dP = dO V^T, warp 10 the accumulating dQ += dS K (dS from
// TMEM); warp 8 loads; warps 0..7 compute dS, two per TMEM lane quarter.
__global__ void __launch_bounds__(BW_THREADS, 1)
fa_tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_o,
                    const float* __restrict__ lse, float* __restrict__ Dg, int T, int H, int BH,
                    DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + DQ_OFF_Q;
    uint8_t* sDO = smem + DQ_OFF_DO;
    uint8_t* sK = smem + DQ_OFF_K;
    uint8_t* sV = smem + DQ_OFF_V;
    uint8_t* sOut = smem + DQ_OFF_OUT;
    uint8_t* sO = smem + DQ_OFF_O;
    uint64_t* bars = (uint64_t*)(smem + DQ_OFF_BAR);
    uint64_t* qd_full = bars;                          // [2]
    uint64_t* qd_empty = bars + 2;                     // [2]
    uint64_t* kv_full = bars + 4;                      // [3]
    uint64_t* kv_empty = bars + 7;                     // [3]
    uint64_t* st_full = bars + 10;
    uint64_t* st_free = bars + 11;
    uint64_t* ds_full = bars + 12;
    uint64_t* ds_free = bars + 13;
    uint64_t* acc_full = bars + 14;                    // [2]
    uint64_t* acc_free = bars + 16;                    // [2]
    uint64_t* drain = bars + 18;                       // [2]
    uint32_t* tmem_slot = (uint32_t*)(bars + 20);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nqb = (T + AT_BQ - 1) / AT_BQ;
    const int items = nqb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&qd_full[i], 1);
            // released by the item's last S/dP products and by the eight softmax
            // warps once they have read their dO rows (for D)
            mbar_init(&qd_empty[i], 9);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], 8);
            mbar_init(&drain[i], 1);
        }
        for (int s = 0; s < BW_SLOTS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        mbar_init(st_full, 1);
        mbar_init(st_free, 8);
        mbar_init(ds_full, 8);
        mbar_init(ds_free, 1);
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == BW_ISSUE_A) tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == BW_PRODUCER) {
        if (lane == 0) {
            // ---------------- TMA producer
            int g = 0, it = 0, nql = 0, nkvl = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH, bh = w % BH, h = bh % H, b = bh / H;
                const int nkv = qb + 1;
                const int qs = it & 1;
                if (!mbar_wait(&qd_empty[qs], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&qd_full[qs], 3 * AT_TILE);
                tma_load_3d(sQ + qs * AT_TILE, &tm_qkv, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                tma_load_3d(sDO + qs * AT_TILE, &tm_do, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                tma_load_3d(sO + qs * AT_TILE, &tm_o, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                nql++;
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % BW_SLOTS;
                    if (!mbar_wait(&kv_empty[s], (uint32_t)(((G / BW_SLOTS) & 1) ^ 1), abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&kv_full[s], 2 * AT_TILE);
                    tma_load_3d(sK + s * AT_TILE, &tm_qkv, &kv_full[s], C + h * AT_HS, j * AT_BK, b);
                    tma_load_3d(sV + s * AT_TILE, &tm_qkv, &kv_full[s], 2 * C + h * AT_HS, j * AT_BK, b);
                    nkvl++;
                }
                g += nkv;
            }
            if (!ok || *abort_flag) {
                for (int i = (nql > 2 ? nql - 2 : 0); i < nql; i++) wait_bounded(&qd_full[i & 1], (uint32_t)((i >> 1) & 1));
                for (int i = (nkvl > BW_SLOTS ? nkvl - BW_SLOTS : 0); i < nkvl; i++)
                    wait_bounded(&kv_full[i % BW_SLOTS], (uint32_t)((i / BW_SLOTS) & 1));
            }
        }
    } else if (warp == BW_ISSUE_A) {
        if (lane == 0) {
            // ---------------- S = Q K^T, dP = dO V^T (M = queries, N = keys, K = head dim)
            constexpr uint32_t id_s = make_idesc(AT_BQ, AT_BK, false, false);
            const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024), ddo0 = smem_desc(smem_u32(sDO), 16, 1024),
                           dk0 = smem_desc(smem_u32(sK), 16, 1024), dv0 = smem_desc(smem_u32(sV), 16, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int nkv = nqb - w / BH;
                const int qs = it & 1;
                if (!mbar_wait(&qd_full[qs], (uint32_t)((it >> 1) & 1), abort_flag)) { ok = false; break; }
                const uint64_t dq = desc_adv(dq0, qs * AT_TILE), ddo = desc_adv(ddo0, qs * AT_TILE);
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % BW_SLOTS;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / BW_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(st_free, (uint32_t)((G & 1) ^ 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dk = desc_adv(dk0, s * AT_TILE), dv = desc_adv(dv0, s * AT_TILE);
#pragma unroll
                    for (int kk = 0; kk < AT_HS / 16; kk++) {
                        mma_bf16(tmem_base + TM_S, desc_adv(dq, 32 * kk), desc_adv(dk, 32 * kk), id_s, kk > 0 ? 1u : 0u);
                        mma_bf16(tmem_base + TM_DP, desc_adv(ddo, 32 * kk), desc_adv(dv, 32 * kk), id_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(st_full);
                    if (j == nkv - 1) mma_commit(&qd_empty[qs]);
                    any = true;
                }
                g += nkv;
            }
            if (any) {
                mma_commit(&drain[0]);
                wait_bounded(&drain[0], 0);
            }
        }
    } else if (warp == BW_ISSUE_B) {
        if (lane == 0) {
            // ---------------- dQ += dS K (A = dS from TMEM, K read MN-major)
            constexpr uint32_t id_a = make_idesc(AT_BQ, AT_HS, false, true);
            const uint64_t dkm0 = smem_desc(smem_u32(sK), 8192, 1024);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int nkv = nqb - w / BH;
                const int ab = it & 1;
                if (!mbar_wait(&acc_free[ab], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % BW_SLOTS;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / BW_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(ds_full, (uint32_t)(G & 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dkm = desc_adv(dkm0, s * AT_TILE);
#pragma unroll
                    for (int kk = 0; kk < AT_BK / 16; kk++)
                        mma_bf16_ta(tmem_base + TM_ACC + ab * AT_HS, tmem_base + TM_PT + kk * 8,
                                    desc_adv(dkm, kk * 2048), id_a, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(ds_free);
                    mma_commit(&kv_empty[s]);
                    if (j == nkv - 1) mma_commit(&acc_full[ab]);
                    any = true;
                }
                g += nkv;
            }
            if (any) {
                mma_commit(&drain[1]);
                wait_bounded(&drain[1], 0);
            }
        }
    } else {
        // ---------------- warps 0..7: warp w reads TMEM lane quarter w % 4 (thread
        // row r = its lane there: query row r) and key columns 64*(w/4)..+63
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = q4 * 32 + lane;
        const float sl2 = LOG2E_F * 0.125f;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q4 * 32) << 16);
        uint8_t* slab = sOut + q4 * OUT_SLAB;
        // this row's lse (log2 units) and D for an item, loaded one item ahead
        // this row's lse (log2 units) for an item, loaded one item ahead
        auto fetch = [&](int w_, float& l_) {
            l_ = INFINITY;
            if (w_ < items) {
                const int qb_ = nqb - 1 - w_ / BH, bh_ = w_ % BH, q_ = qb_ * AT_BQ + r;
                if (q_ < T) l_ = lse[(int64_t)bh_ * T + q_] * LOG2E_F;
            }
        };
        float nl;
        fetch(blockIdx.x, nl);
        bool ok = true;
        int g = 0, it = 0;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int qb = nqb - 1 - w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int nkv = qb + 1;
            const int q = qb * AT_BQ + r;
            const int ab = it & 1, qs = it & 1;
            const float lse2 = nl;
            fetch(w + gridDim.x, nl);
            // D = rowsum(dO * O) from this row of the dO and O tiles (128B-swizzled);
            // written once for the dK/dV kernel
            ok = mbar_wait(&qd_full[qs], (uint32_t)((it >> 1) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            float Dq = 0.f;
            {
                const uint8_t* drow = sDO + qs * AT_TILE + r * 128;
                const uint8_t* orow = sO + qs * AT_TILE + r * 128;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const uint4 dv = *(const uint4*)(drow + ((c ^ (r & 7)) << 4));
                    const uint4 ov = *(const uint4*)(orow + ((c ^ (r & 7)) << 4));
                    const uint32_t du[4] = {dv.x, dv.y, dv.z, dv.w};
                    const uint32_t ou[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
                    for (int k2 = 0; k2 < 4; k2++) {
                        const float2 a2 = __bfloat1622float2(*(const __nv_bfloat162*)&du[k2]);
                        const float2 o2 = __bfloat1622float2(*(const __nv_bfloat162*)&ou[k2]);
                        Dq = fmaf(a2.x, o2.x, fmaf(a2.y, o2.y, Dq));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qd_empty[qs]);
            if (hf == 0 && q < T) Dg[(int64_t)bh * T + q] = Dq;
            for (int j = 0; j < nkv; j++) {
                const int G = g + j;
                ok = mbar_wait(st_full, (uint32_t)(G & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ok = mbar_wait(ds_free, (uint32_t)((G & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const int key0 = j * AT_BK;
                const bool edge = (j == qb) || (key0 + AT_BK > T);
#pragma unroll 1
                for (int c = 2 * hf; c < 2 * hf + 2; c++) {
                    uint32_t sr[32], dr[32];
                    tmem_ld32_nowait(lane_base + TM_S + 32 * c, sr);
                    tmem_ld32_nowait(lane_base + TM_DP + 32 * c, dr);
                    tmem_wait_ld();
                    if (c == 2 * hf + 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(st_free);
                    }
                    uint32_t pd[16];
#pragma unroll
                    for (int t = 0; t < 16; t++) {
                        float d[2];
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            const int kk = key0 + 32 * c + 2 * t + u;
                            float e = ex2f(fmaf(__uint_as_float(sr[2 * t + u]), sl2, -lse2));
                            if (edge && (kk > q || kk >= T)) e = 0.f;
                            d[u] = e * (__uint_as_float(dr[2 * t + u]) - Dq);
                        }
                        pd[t] = pack2_bf16(d[0], d[1]);
                    }
                    tmem_st16(lane_base + TM_PT + 16 * c, pd);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
            }
            if (!ok) break;
            ok = mbar_wait(&acc_full[ab], (uint32_t)((it >> 1) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // the lower-half warp of each quarter writes the dQ rows
            uint32_t dq[64];
            if (hf == 0) {
                tmem_ld32_nowait(lane_base + TM_ACC + ab * AT_HS, dq);
                tmem_ld32_nowait(lane_base + TM_ACC + ab * AT_HS + 32, dq + 32);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[ab]);
            if (hf == 0) {
                if (lane == 0) tma_wait_read<0>();
                __syncwarp();
                stage_out_slab(slab, lane, dq, 0.125f);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int row0 = qb * AT_BQ + q4 * 32;
                    if (row0 < T) tma_store_3d(&tm_out, slab, h * AT_HS, row0, b);
                    tma_commit();
                }
            }
            g += nkv;
        }
        if (lane == 0) tma_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 5;
    }
    if (warp == BW_ISSUE_A) {
        tc_fence_after();
        tmem_dealloc(tmem_base, AT_TMEM_COLS);
    }
}

// dout (or the forward output) [B, T, C] bf16 as a 3-D map {C, T, B}, boxes
// 64 x 128 x 1, 128B swizzle.
static bool make_do_map(CUtensorMap* map, const bf16* dout, int B, int T, int C) {
    EncodeTiledFnA enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)C * 2 * T};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(dout), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// dqkv [B, T, 3C] bf16 as the target of the per-warp output stores: 3-D map
// {3C, T, B}, boxes of 64 x 32 x 1 with 128B swizzle (rows beyond T clipped).
static bool make_dqkv_map(CUtensorMap* map, bf16* dqkv, int B, int T, int C) {
    EncodeTiledFnA enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)3 * C * 2 * T};
    cuuint32_t box[3] = {64, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dqkv, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t attention_bwd_tc(const bf16* qkv, const bf16* out, const bf16* dout, const float* lse,
                             float* D, bf16* dqkv, int B, int T, int H, int hs, DevState* st,
                             cudaStream_t s) {
    if (hs != AT_HS || T < 1 || B < 1 || H < 1 || !st) return cudaErrorInvalidValue;
    if (((uintptr_t)qkv & 15) || ((uintptr_t)dout & 15) || ((uintptr_t)dqkv & 15) || ((uintptr_t)out & 15))
        return cudaErrorInvalidValue;
    CUtensorMap mq, md, mo, mf;
    memset(&mq, 0, sizeof mq);
    memset(&md, 0, sizeof md);
    memset(&mo, 0, sizeof mo);
    memset(&mf, 0, sizeof mf);
    if (!make_qkv_map(&mq, qkv, B, T, H * hs) || !make_do_map(&md, dout, B, T, H * hs) ||
        !make_dqkv_map(&mo, dqkv, B, T, H * hs) || !make_do_map(&mf, out, B, T, H * hs))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        CUDA_OK(cudaFuncSetAttribute(fa_tc_bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)KV_SMEM));
        CUDA_OK(cudaFuncSetAttribute(fa_tc_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DQ_SMEM));
        attr_done.fetch_or(dbit);
    }
    const int items = ((T + AT_BQ - 1) / AT_BQ) * B * H;
    const int grid = items < num_sms() ? items : num_sms();
    // the dQ kernel also computes D = rowsum(dO * O), which the dK/dV kernel reads
    fa_tc_bwd_dq_kernel<<<grid, BW_THREADS, DQ_SMEM, s>>>(mq, md, mo, mf, lse, D, T, H, B * H, st);
    CUDA_OK(cudaGetLastError());
    fa_tc_bwd_dkv_kernel<<<grid, BW_THREADS, KV_SMEM, s>>>(mq, md, mo, lse, D, T, H, B * H, st);
    return cudaGetLastError();
}

bool attention_bf16_supported(int T, int hs) { return hs == AT_HS && T >= 1; }

cudaError_t attention_bwd_bf16(const bf16* qkv, const bf16* out, const float* lse,
                               const bf16* dout, bf16* dqkv, float* Dbuf, int B, int T, int H,
                               int hs, DevState* st, cudaStream_t s) {
    if (!attention_bf16_supported(T, hs)) return cudaErrorInvalidValue;
    return attention_bwd_tc(qkv, out, dout, lse, Dbuf, dqkv, B, T, H, hs, st, s);
}

}  // namespace k
