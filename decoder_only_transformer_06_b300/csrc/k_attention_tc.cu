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
#include "attn_tc.cuh"

namespace k {

using namespace tc;

using namespace attn;

namespace {

constexpr int AT_SLOTS = 3;                    // K and V ring depth
constexpr int FW_THREADS = 224;                // forward: 4 softmax warps, producer, two MMA issuers
constexpr int OFF_Q = 0;                       // Q double buffer
constexpr int OFF_K = OFF_Q + 2 * AT_TILE;
constexpr int OFF_V = OFF_K + AT_SLOTS * AT_TILE;
constexpr int OFF_OUT = OFF_V + AT_SLOTS * AT_TILE;   // [4 softmax warps] O slabs
constexpr int OFF_BAR = OFF_OUT + 4 * OUT_SLAB;
constexpr size_t AT_SMEM = OFF_BAR + 256 + 1024;
// forward TMEM columns: S[0] 0..127, S[1] 128..255, O[0] 256..319, O[1]
// 320..383, P[0] 384..447, P[1] 448..511 (P: bf16 pairs, the A operand of P V)
constexpr uint32_t TM_O = 256, TM_P = 384;
constexpr uint32_t AT_TMEM_COLS = 512;

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
cudaError_t attention_fwd_bf16(const bf16* qkv, bf16* out, float* lse, int B, int T, int H, int hs,
                               DevState* st, cudaStream_t s) {
    if (hs != AT_HS || T < 1 || B < 1 || H < 1 || !st) return cudaErrorInvalidValue;
    if (((uintptr_t)qkv & 15) || ((uintptr_t)out & 15)) return cudaErrorInvalidValue;
    CUtensorMap map, omap;
    // qkv [B, T, 3C] read in 128-row boxes; out written by per-warp 32-row stores
    if (!make_rows_map(&map, qkv, B, T, 3 * H * hs, AT_BQ, true) ||
        !make_rows_map(&omap, out, B, T, H * hs, 32, false))
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

}  // namespace k
