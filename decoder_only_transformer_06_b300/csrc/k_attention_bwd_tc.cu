// Causal flash attention backward on the 5th-generation tensor cores (tcgen05,
// sm_103a): bf16 operands, fp32 products and accumulators in tensor memory.
//
// Semantics: the gradient of nanoGPT's manual causal attention (nanoGPT guide
// Deep dive 1; the pages give no backward, autograd computes it): with the raw
// score s = q.k, p = exp(s/sqrt(hs) - lse) (lse saved by the forward),
// dP = dO V^T, D = rowsum(dO * O) and dS = P * (dP - D) (the gradient of the
// scaled scores):
//   dQ = dS K / sqrt(hs)                  (kernel 1, one work item per 128 queries)
//   dK = dS^T Q / sqrt(hs), dV = P^T dO   (kernel 2, one work item per 128 keys)
// The probabilities are recomputed from lse in both kernels; nothing is
// accumulated with atomics, so the result is deterministic. Kernel 1 also
// writes D for kernel 2.
//
// Structure shared by both kernels (persistent, one CTA per SM):
//   warps 0..15 elementwise work: warp w reads TMEM lane quarter w % 4 (32
//               rows) and columns 16 (w / 4) .. +15 of each 64-column step;
//               writes the bf16 A operands of the accumulating products back
//               into TMEM (two buffers)
//   warp 16     TMA producer: the item's 128-row tiles once, then the other
//               operand in 64-row sub-blocks through a ring of slots
//   warps 17..  one warp per product, lane 0 issuing it: the score-like
//               products of a step (S and dP, or their transposes) into one of
//               two TMEM buffers, and the accumulating products (dQ, or dV and
//               dK) whose A operands (dS, or P^T and dS^T) are read from TMEM.
//               Warp 17 allocates the 512 TMEM columns.
// One issuing thread sustains about one tcgen05.mma per hundred cycles
// whatever its size (measured on B300), so each product has its own issuing
// warp and the tensor core interleaves their instruction streams; 16
// elementwise warps (four per SM sub-partition) hide the latency of the
// exponentials and TMEM copies. The 64-row sub-blocks make every per-step
// buffer double-buffered inside the 512 TMEM columns, so the products of step
// j+1 run while the elementwise warps work on step j. In the dQ kernel the
// producer/issuer warpgroup (warps 16..19) gives up registers to the four
// elementwise warpgroups (setmaxnreg), which then run without spills. Every
// mbarrier wait is bounded; on expiry the CTA records ERR_TIMEOUT, drains its
// copies and products (bounded), frees TMEM and returns.
#include "attn_tc.cuh"

namespace k {

using namespace tc;
using namespace attn;

namespace {

constexpr int NEW = 16;                         // elementwise warps
constexpr int BW_PRODUCER = 16;
constexpr int BW_ISSUE0 = 17;                   // first issuing warp
constexpr int KV_THREADS = 32 * (NEW + 1 + 4);  // dK/dV: S^T, dP^T, dV, dK issuers
constexpr int DQ_THREADS = 32 * (NEW + 1 + 3);  // dQ: S, dP, dQ issuers
constexpr int SUB = 64;                         // rows of a streamed sub-block
constexpr int SUB_TILE = SUB * AT_HS * 2;       // 8 KB
constexpr int OUT32 = 32 * 32 * 2;              // one warp's 32 x 32 output slab, 2 KB

// dK/dV kernel: K and V of the item double buffered (by item), Q and dO in a
// ring of 64-query sub-blocks with their lse and D values staged beside them
constexpr int KV_NS = 7;
constexpr int KV_OFF_K = 0;                                  // [2] 16 KB
constexpr int KV_OFF_V = KV_OFF_K + 2 * AT_TILE;             // [2]
constexpr int KV_OFF_Q = KV_OFF_V + 2 * AT_TILE;             // [NS] 8 KB
constexpr int KV_OFF_DO = KV_OFF_Q + KV_NS * SUB_TILE;       // [NS]
constexpr int KV_OFF_OUT = KV_OFF_DO + KV_NS * SUB_TILE;     // [16 warps] dK or dV slab
constexpr int KV_OFF_LD = KV_OFF_OUT + NEW * OUT32;          // [NS] lse2[64], D[64]
constexpr int KV_OFF_BAR = KV_OFF_LD + KV_NS * 2 * SUB * 4;
constexpr size_t KV_SMEM = KV_OFF_BAR + 512 + 1024;          // barriers, then alignment slack
// dK/dV TMEM columns: S^T[2] 0..127, dP^T[2] 128..255, dV 256..319, dK
// 320..383, P^T[2] 384..447, dS^T[2] 448..511 (bf16 pairs, 32 columns each)
constexpr uint32_t KV_TM_ST = 0, KV_TM_DPT = 128, KV_TM_DV = 256, KV_TM_DK = 320, KV_TM_PT = 384,
                   KV_TM_DST = 448;

// dQ kernel: Q, dO and O of the item double buffered (by item), K and V in a
// ring of 64-key sub-blocks
constexpr int DQ_NS = 6;
constexpr int DQ_OFF_Q = 0;                                  // [2] 16 KB
constexpr int DQ_OFF_DO = DQ_OFF_Q + 2 * AT_TILE;            // [2]
constexpr int DQ_OFF_O = DQ_OFF_DO + 2 * AT_TILE;            // [2] forward output tile (for D)
constexpr int DQ_OFF_K = DQ_OFF_O + 2 * AT_TILE;             // [NS] 8 KB
constexpr int DQ_OFF_V = DQ_OFF_K + DQ_NS * SUB_TILE;        // [NS]
constexpr int DQ_OFF_OUT = DQ_OFF_V + DQ_NS * SUB_TILE;      // [8 warps] dQ slabs
constexpr int DQ_OFF_BAR = DQ_OFF_OUT + 8 * OUT32;
constexpr size_t DQ_SMEM = DQ_OFF_BAR + 512 + 1024;
// dQ TMEM columns: S[2] 0..127, dP[2] 128..255, dQ[2] 256..383 (by item),
// dS[2] 384..447 (bf16 pairs)
constexpr uint32_t DQ_TM_S = 0, DQ_TM_DP = 128, DQ_TM_DQ = 256, DQ_TM_DS = 384;
// dQ kernel registers: the launch gives each of the 640 threads DQ_REGS; the
// producer and issuer warpgroup (warps 16..19) drops to DQ_REGS_LOW and the
// four elementwise warpgroups rise to DQ_REGS_HIGH (setmaxnreg). The shares
// must add up to no more than the launch's total, or the increase would wait
// forever; the host checks that the kernel was compiled with DQ_REGS.
constexpr int DQ_REGS = 96, DQ_REGS_LOW = 56, DQ_REGS_HIGH = 104;
static_assert(4 * DQ_REGS_LOW + 16 * DQ_REGS_HIGH <= 20 * DQ_REGS, "register split exceeds the launch");
static_assert(DQ_THREADS == 640 && BW_PRODUCER == 16, "warpgroup layout of the dQ kernel");
constexpr uint32_t BW_TMEM_COLS = 512;

// Four K=16 products of a 64-row step into one accumulator: D (+)= A B over
// the step's head dimension or rows. a0/b0 are the step's first descriptors,
// advanced by a_step/b_step bytes per product (a_tmem: A is a TMEM address
// advanced by 8 columns).
__device__ __forceinline__ void mma4_ss(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc, bool acc_first) {
#pragma unroll
    for (int kk = 0; kk < 4; kk++)
        mma_bf16(d, desc_adv(a0, 32 * kk), desc_adv(b0, 32 * kk), idesc, (acc_first || kk > 0) ? 1u : 0u);
}
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a_tmem, uint64_t b0, uint32_t idesc, bool acc_first) {
#pragma unroll
    for (int kk = 0; kk < 4; kk++)
        mma_bf16_ta(d, a_tmem + 8 * kk, desc_adv(b0, 2048 * kk), idesc, (acc_first || kk > 0) ? 1u : 0u);
}

}  // namespace

// Work items (key block kb, b, h), most sub-blocks first (kb = w / (B*H)); an
// item walks the 64-query sub-blocks from the diagonal to T. G counts
// sub-blocks over all items (ring slots, TMEM buffers), `it` counts items.
__global__ void __launch_bounds__(KV_THREADS, 1)
fa_tc_bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_out,
                     const float* __restrict__ lse, const float* __restrict__ Dg, int T, int H, int BH,
                     DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sK = smem + KV_OFF_K;
    uint8_t* sV = smem + KV_OFF_V;
    uint8_t* sQ = smem + KV_OFF_Q;
    uint8_t* sDO = smem + KV_OFF_DO;
    uint8_t* sOut = smem + KV_OFF_OUT;
    float* sLD = (float*)(smem + KV_OFF_LD);
    uint64_t* bars = (uint64_t*)(smem + KV_OFF_BAR);
    uint64_t* kv_full = bars;                          // [2]
    uint64_t* kv_empty = bars + 2;                     // [2] S^T and dP^T issuers
    uint64_t* qd_full = bars + 4;                      // [NS]
    uint64_t* qd_empty = bars + 4 + KV_NS;             // [NS] dV and dK issuers
    uint64_t* ld_full = bars + 4 + 2 * KV_NS;          // [NS]
    uint64_t* st_full = bars + 4 + 3 * KV_NS;          // [2] S^T and dP^T issuers
    uint64_t* st_free = st_full + 2;                   // [2] elementwise warps
    uint64_t* ps_full = st_full + 4;                   // [2] elementwise warps
    uint64_t* ps_free = st_full + 6;                   // [2] dV and dK issuers
    uint64_t* acc_full = st_full + 8;                  // dV and dK issuers
    uint64_t* acc_free = st_full + 9;                  // elementwise warps
    uint64_t* drain = st_full + 10;                    // [4] one per issuer
    uint32_t* tmem_slot = (uint32_t*)(st_full + 14);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nb = (T + AT_BK - 1) / AT_BK;
    const int items = nb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 2);
            mbar_init(&st_full[i], 2);
            mbar_init(&st_free[i], NEW);
            mbar_init(&ps_full[i], NEW);
            mbar_init(&ps_free[i], 2);
        }
        for (int s = 0; s < KV_NS; s++) {
            mbar_init(&qd_full[s], 1);
            mbar_init(&qd_empty[s], 2);
            mbar_init(&ld_full[s], 1);
        }
        mbar_init(acc_full, 2);
        mbar_init(acc_free, NEW);
        for (int i = 0; i < 4; i++) mbar_init(&drain[i], 1);
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == BW_ISSUE0) tmem_alloc(tmem_slot, BW_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();                              // the previous kernel's outputs are visible

    if (warp == BW_PRODUCER) {
        // ---------------- producer warp: lane 0 issues the TMA copies; all lanes
        // stage the lse (log2 units) and D values of each query sub-block
        int g = 0, it = 0, nkvl = 0, nql = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int kb = w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int n = (T - kb * AT_BK + SUB - 1) / SUB;
            const int ks = it & 1;
            if (lane == 0) {
                ok = mbar_wait(&kv_empty[ks], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag);
                if (ok) {
                    mbar_arrive_expect_tx(&kv_full[ks], 2 * AT_TILE);
                    tma_load_3d(sK + ks * AT_TILE, &tm_kv, &kv_full[ks], C + h * AT_HS, kb * AT_BK, b);
                    tma_load_3d(sV + ks * AT_TILE, &tm_kv, &kv_full[ks], 2 * C + h * AT_HS, kb * AT_BK, b);
                    nkvl++;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
            for (int i = 0; i < n; i++) {
                const int G = g + i, qs = G % KV_NS;
                const int q0 = kb * AT_BK + i * SUB;
                ok = mbar_wait(&qd_empty[qs], (uint32_t)(((G / KV_NS) & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&qd_full[qs], 2 * SUB_TILE);
                    tma_load_3d(sQ + qs * SUB_TILE, &tm_q, &qd_full[qs], h * AT_HS, q0, b);
                    tma_load_3d(sDO + qs * SUB_TILE, &tm_do, &qd_full[qs], h * AT_HS, q0, b);
                    nql++;
                }
                float* ldst = sLD + qs * 2 * SUB;
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int qq = u * 32 + lane, q = q0 + qq;
                    ldst[qq] = q < T ? lse[(int64_t)bh * T + q] * LOG2E_F : INFINITY;
                    ldst[SUB + qq] = q < T ? Dg[(int64_t)bh * T + q] : 0.f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ld_full[qs]);
            }
            g += n;
        }
        if (lane == 0) pdl_trigger();        // every copy of this CTA is issued
        if (lane == 0 && (!ok || *abort_flag)) {
            for (int i = (nkvl > 2 ? nkvl - 2 : 0); i < nkvl; i++) wait_bounded(&kv_full[i & 1], (uint32_t)((i >> 1) & 1));
            for (int i = (nql > KV_NS ? nql - KV_NS : 0); i < nql; i++)
                wait_bounded(&qd_full[i % KV_NS], (uint32_t)((i / KV_NS) & 1));
        }
    } else if (warp > BW_PRODUCER) {
        if (lane == 0) {
            // ---------------- issuers: 0 S^T = K Q^T, 1 dP^T = V dO^T (M = 128 keys,
            // N = 64 queries, K = head dim); 2 dV += P^T dO, 3 dK += dS^T Q (A from
            // TMEM, dO / Q read MN-major: the reduction runs over the 64 query rows)
            const int role = warp - BW_ISSUE0;
            const bool score = role < 2;
            constexpr uint32_t id_s = make_idesc(AT_BK, SUB, false, false);
            constexpr uint32_t id_a = make_idesc(AT_BK, AT_HS, false, true);
            const uint64_t dkv0 = smem_desc(smem_u32(role == 0 ? sK : sV), 16, 1024);
            const uint64_t dop0 = smem_desc(smem_u32((role == 0 || role == 3) ? sQ : sDO), 16, 1024);
            const uint64_t dopm0 = smem_desc(smem_u32(role == 3 ? sQ : sDO), 8192, 1024);
            const uint32_t d_score = tmem_base + (role == 0 ? KV_TM_ST : KV_TM_DPT);
            const uint32_t d_acc = tmem_base + (role == 2 ? KV_TM_DV : KV_TM_DK);
            const uint32_t a_acc = tmem_base + (role == 2 ? KV_TM_PT : KV_TM_DST);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int kb = w / BH;
                const int n = (T - kb * AT_BK + SUB - 1) / SUB;
                const int ks = it & 1;
                if (score) {
                    if (!mbar_wait(&kv_full[ks], (uint32_t)((it >> 1) & 1), abort_flag)) { ok = false; break; }
                } else {
                    if (!mbar_wait(acc_free, (uint32_t)((it & 1) ^ 1), abort_flag)) { ok = false; break; }
                }
                const uint64_t dkv = desc_adv(dkv0, ks * AT_TILE);
                for (int i = 0; i < n; i++) {
                    const int G = g + i, qs = G % KV_NS, sb = G & 1;
                    if (score) {
                        if (!mbar_wait(&qd_full[qs], (uint32_t)((G / KV_NS) & 1), abort_flag)) { ok = false; break; }
                        if (!mbar_wait(&st_free[sb], (uint32_t)(((G >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        mma4_ss(d_score + sb * SUB, dkv, desc_adv(dop0, qs * SUB_TILE), id_s, false);
                        mma_commit(&st_full[sb]);
                        if (i == n - 1) mma_commit(&kv_empty[ks]);
                    } else {
                        if (!mbar_wait(&ps_full[sb], (uint32_t)((G >> 1) & 1), abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        mma4_ts(d_acc, a_acc + sb * (SUB / 2), desc_adv(dopm0, qs * SUB_TILE), id_a, i > 0);
                        mma_commit(&ps_free[sb]);
                        mma_commit(&qd_empty[qs]);
                        if (i == n - 1) mma_commit(acc_full);
                    }
                    any = true;
                }
                g += n;
            }
            if (any) {
                mma_commit(&drain[role]);
                wait_bounded(&drain[role], 0);
            }
        }
    } else {
        // ---------------- warps 0..15: warp w reads TMEM lane quarter q4 = w % 4
        // (thread row r = key r of the item) and query columns 16 cg .. +15 of
        // each 64-query sub-block, cg = w / 4
        const int q4 = warp & 3, cg = warp >> 2;
        const int r = q4 * 32 + lane;
        const float sl2 = LOG2E_F * 0.125f;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q4 * 32) << 16);
        uint8_t* slab = sOut + warp * OUT32;
        bool ok = true;
        int g = 0, it = 0;
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int kb = w / BH, bh = w % BH, h = bh % H, b = bh / H;
            const int n = (T - kb * AT_BK + SUB - 1) / SUB;
            const int key = kb * AT_BK + r;
            for (int i = 0; i < n; i++) {
                const int G = g + i, qs = G % KV_NS, sb = G & 1;
                ok = mbar_wait(&ld_full[qs], (uint32_t)((G / KV_NS) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ok = mbar_wait(&st_full[sb], (uint32_t)((G >> 1) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                // P^T / dS^T buffer sb is free once the products of two steps ago read it
                ok = mbar_wait(&ps_free[sb], (uint32_t)(((G >> 1) & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[16], dr[16];
                tmem_ld16_nowait(lane_base + KV_TM_ST + sb * SUB + 16 * cg, sr);
                tmem_ld16_nowait(lane_base + KV_TM_DPT + sb * SUB + 16 * cg, dr);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st_free[sb]);
                const float* L = sLD + qs * 2 * SUB + 16 * cg;
                const float* Dq = L + SUB;
                const int qc0 = kb * AT_BK + i * SUB + 16 * cg;     // query of column 0 of this group
                uint32_t pp[8], pd[8];
                float p[16];
#pragma unroll
                for (int t4 = 0; t4 < 4; t4++) {
                    const float4 l4 = *(const float4*)&L[4 * t4];       // broadcast reads
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        p[4 * t4 + u] = ex2f(fmaf(__uint_as_float(sr[4 * t4 + u]), sl2, -lv[u]));
                }
                if (qc0 < key) {                                   // some query before this key: mask
#pragma unroll
                    for (int c = 0; c < 16; c++)
                        if (qc0 + c < key) p[c] = 0.f;
                }
#pragma unroll
                for (int t4 = 0; t4 < 4; t4++) {
                    const float4 d4 = *(const float4*)&Dq[4 * t4];
                    const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                    float d[4];
#pragma unroll
                    for (int u = 0; u < 4; u++) d[u] = p[4 * t4 + u] * (__uint_as_float(dr[4 * t4 + u]) - dv4[u]);
                    pp[2 * t4] = pack2_bf16(p[4 * t4], p[4 * t4 + 1]);
                    pp[2 * t4 + 1] = pack2_bf16(p[4 * t4 + 2], p[4 * t4 + 3]);
                    pd[2 * t4] = pack2_bf16(d[0], d[1]);
                    pd[2 * t4 + 1] = pack2_bf16(d[2], d[3]);
                }
                tmem_st8(lane_base + KV_TM_PT + sb * (SUB / 2) + 8 * cg, pp);
                tmem_st8(lane_base + KV_TM_DST + sb * (SUB / 2) + 8 * cg, pd);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ps_full[sb]);
            }
            if (!ok) break;
            // the item's dK, dV rows: warp groups 0, 1 take dK columns 0..31,
            // 32..63, groups 2, 3 dV; one 32 x 32 TMA store per warp
            ok = mbar_wait(acc_full, (uint32_t)(it & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t acc[32];
            const int half = cg & 1;
            tmem_ld32_nowait(lane_base + (cg < 2 ? KV_TM_DK : KV_TM_DV) + 32 * half, acc);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            if (lane == 0) tma_wait_read<0>();               // the previous item's store has read the slab
            __syncwarp();
            stage_out_slab32(slab, lane, acc, cg < 2 ? 0.125f : 1.f);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int row0 = kb * AT_BK + q4 * 32;
                if (row0 < T) tma_store_3d(&tm_out, slab, (cg < 2 ? C : 2 * C) + h * AT_HS + 32 * half, row0, b);
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
    if (warp == BW_ISSUE0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, BW_TMEM_COLS);
    }
}

// Work items (query block qb, b, h), most sub-blocks first; an item walks the
// 64-key sub-blocks from 0 to the diagonal. Kernel 1 of the backward: also
// computes D = rowsum(dO * O) per query row for the dK/dV kernel.
__global__ void __launch_bounds__(DQ_THREADS, 1)
fa_tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ lse,
                    float* __restrict__ Dg, int T, int H, int BH, DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + DQ_OFF_Q;
    uint8_t* sDO = smem + DQ_OFF_DO;
    uint8_t* sO = smem + DQ_OFF_O;
    uint8_t* sK = smem + DQ_OFF_K;
    uint8_t* sV = smem + DQ_OFF_V;
    uint8_t* sOut = smem + DQ_OFF_OUT;
    uint64_t* bars = (uint64_t*)(smem + DQ_OFF_BAR);
    uint64_t* qd_full = bars;                          // [2]
    uint64_t* qd_empty = bars + 2;                     // [2] S and dP issuers + elementwise warps
    uint64_t* kv_full = bars + 4;                      // [NS]
    uint64_t* kv_empty = bars + 4 + DQ_NS;             // [NS] dQ issuer
    uint64_t* st_full = bars + 4 + 2 * DQ_NS;          // [2] S and dP issuers
    uint64_t* st_free = st_full + 2;                   // [2] elementwise warps
    uint64_t* ds_full = st_full + 4;                   // [2] elementwise warps
    uint64_t* ds_free = st_full + 6;                   // [2] dQ issuer
    uint64_t* acc_full = st_full + 8;                  // [2] dQ issuer
    uint64_t* acc_free = st_full + 10;                 // [2] elementwise warps
    uint64_t* drain = st_full + 12;                    // [3] one per issuer
    uint32_t* tmem_slot = (uint32_t*)(st_full + 15);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nqb = (T + AT_BQ - 1) / AT_BQ;
    const int nsb = (T + SUB - 1) / SUB;               // key sub-blocks of a sequence
    const int items = nqb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&qd_full[i], 1);
            // released by the item's last S and dP products and by the
            // elementwise warps once they have read their dO and O rows (for D)
            mbar_init(&qd_empty[i], 2 + NEW);
            mbar_init(&st_full[i], 2);
            mbar_init(&st_free[i], NEW);
            mbar_init(&ds_full[i], NEW);
            mbar_init(&ds_free[i], 1);
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], NEW);
        }
        for (int s = 0; s < DQ_NS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 3; i++) mbar_init(&drain[i], 1);
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == BW_ISSUE0) tmem_alloc(tmem_slot, BW_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();                              // the previous kernel's outputs are visible
    // sub-blocks of the item whose query block is qb: keys 0 .. min(T, 128 qb + 128)
    auto nsub = [&](int qb) { return min(nsb, 2 * qb + 2); };

    if (warp >= BW_PRODUCER) {
    // one register-split instruction per warpgroup (all four warps run it)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(DQ_REGS_LOW));
    if (warp == BW_PRODUCER) {
        if (lane == 0) {
            // ---------------- TMA producer
            int g = 0, it = 0, nql = 0, nkvl = 0;
            bool ok = true;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH, bh = w % BH, h = bh % H, b = bh / H;
                const int n = nsub(qb);
                const int qs = it & 1;
                if (!mbar_wait(&qd_empty[qs], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&qd_full[qs], 3 * AT_TILE);
                tma_load_3d(sQ + qs * AT_TILE, &tm_q, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                tma_load_3d(sDO + qs * AT_TILE, &tm_do, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                tma_load_3d(sO + qs * AT_TILE, &tm_o, &qd_full[qs], h * AT_HS, qb * AT_BQ, b);
                nql++;
                for (int j = 0; j < n; j++) {
                    const int G = g + j, s = G % DQ_NS;
                    if (!mbar_wait(&kv_empty[s], (uint32_t)(((G / DQ_NS) & 1) ^ 1), abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(&kv_full[s], 2 * SUB_TILE);
                    tma_load_3d(sK + s * SUB_TILE, &tm_kv, &kv_full[s], C + h * AT_HS, j * SUB, b);
                    tma_load_3d(sV + s * SUB_TILE, &tm_kv, &kv_full[s], 2 * C + h * AT_HS, j * SUB, b);
                    nkvl++;
                }
                g += n;
            }
            pdl_trigger();                   // every copy of this CTA is issued
            if (!ok || *abort_flag) {
                for (int i = (nql > 2 ? nql - 2 : 0); i < nql; i++) wait_bounded(&qd_full[i & 1], (uint32_t)((i >> 1) & 1));
                for (int i = (nkvl > DQ_NS ? nkvl - DQ_NS : 0); i < nkvl; i++)
                    wait_bounded(&kv_full[i % DQ_NS], (uint32_t)((i / DQ_NS) & 1));
            }
        }
    } else if (warp > BW_PRODUCER) {
        if (lane == 0) {
            // ---------------- issuers: 0 S = Q K^T, 1 dP = dO V^T (M = 128 queries,
            // N = 64 keys, K = head dim); 2 dQ += dS K (A = dS from TMEM, K read
            // MN-major: the reduction runs over the sub-block's 64 key rows)
            const int role = warp - BW_ISSUE0;
            constexpr uint32_t id_s = make_idesc(AT_BQ, SUB, false, false);
            constexpr uint32_t id_a = make_idesc(AT_BQ, AT_HS, false, true);
            const uint64_t da0 = smem_desc(smem_u32(role == 0 ? sQ : sDO), 16, 1024);
            const uint64_t db0 = smem_desc(smem_u32(role == 0 ? sK : sV), 16, 1024);
            const uint64_t dkm0 = smem_desc(smem_u32(sK), 8192, 1024);
            const uint32_t d_score = tmem_base + (role == 0 ? DQ_TM_S : DQ_TM_DP);
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH;
                const int n = nsub(qb);
                const int qs = it & 1, ab = it & 1;
                if (role < 2) {
                    if (!mbar_wait(&qd_full[qs], (uint32_t)((it >> 1) & 1), abort_flag)) { ok = false; break; }
                } else {
                    if (!mbar_wait(&acc_free[ab], (uint32_t)(((it >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                }
                const uint64_t da = desc_adv(da0, qs * AT_TILE);
                for (int j = 0; j < n; j++) {
                    const int G = g + j, s = G % DQ_NS, sb = G & 1;
                    if (role < 2) {
                        if (!mbar_wait(&kv_full[s], (uint32_t)((G / DQ_NS) & 1), abort_flag)) { ok = false; break; }
                        if (!mbar_wait(&st_free[sb], (uint32_t)(((G >> 1) & 1) ^ 1), abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        mma4_ss(d_score + sb * SUB, da, desc_adv(db0, s * SUB_TILE), id_s, false);
                        mma_commit(&st_full[sb]);
                        if (j == n - 1) mma_commit(&qd_empty[qs]);
                    } else {
                        if (!mbar_wait(&ds_full[sb], (uint32_t)((G >> 1) & 1), abort_flag)) { ok = false; break; }
                        tc_fence_after();
                        mma4_ts(tmem_base + DQ_TM_DQ + ab * AT_HS, tmem_base + DQ_TM_DS + sb * (SUB / 2),
                                desc_adv(dkm0, s * SUB_TILE), id_a, j > 0);
                        mma_commit(&ds_free[sb]);
                        mma_commit(&kv_empty[s]);
                        if (j == n - 1) mma_commit(&acc_full[ab]);
                    }
                    any = true;
                }
                g += n;
            }
            if (any) {
                mma_commit(&drain[role]);
                wait_bounded(&drain[role], 0);
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(DQ_REGS_HIGH));
        // ---------------- warps 0..15: warp w reads TMEM lane quarter q4 = w % 4
        // (thread row r = query r of the item) and key columns 16 cg .. +15 of
        // each 64-key sub-block, cg = w / 4
        const int q4 = warp & 3, cg = warp >> 2;
        const int r = q4 * 32 + lane;
        const float sl2 = LOG2E_F * 0.125f;
        const uint32_t lane_base = tmem_base + ((uint32_t)(q4 * 32) << 16);
        uint8_t* slab = sOut + (cg * 4 + q4) * OUT32;   // used by groups 0 and 1
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
            const int n = nsub(qb);
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
            if (cg == 0 && q < T) Dg[(int64_t)bh * T + q] = Dq;
            for (int j = 0; j < n; j++) {
                const int G = g + j, sb = G & 1;
                ok = mbar_wait(&st_full[sb], (uint32_t)((G >> 1) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                // dS buffer sb is free once the product of two steps ago read it
                ok = mbar_wait(&ds_free[sb], (uint32_t)(((G >> 1) & 1) ^ 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[16], dr[16];
                tmem_ld16_nowait(lane_base + DQ_TM_S + sb * SUB + 16 * cg, sr);
                tmem_ld16_nowait(lane_base + DQ_TM_DP + sb * SUB + 16 * cg, dr);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st_free[sb]);
                const int k0 = j * SUB + 16 * cg;                   // key of column 0 of this group
                float p[16];
#pragma unroll
                for (int c = 0; c < 16; c++) p[c] = ex2f(fmaf(__uint_as_float(sr[c]), sl2, -lse2));
                if (k0 + 15 > q || k0 + 16 > T) {                   // a key after this query or past T
#pragma unroll
                    for (int c = 0; c < 16; c++)
                        if (k0 + c > q || k0 + c >= T) p[c] = 0.f;
                }
                uint32_t pd[8];
#pragma unroll
                for (int t = 0; t < 8; t++)
                    pd[t] = pack2_bf16(p[2 * t] * (__uint_as_float(dr[2 * t]) - Dq),
                                       p[2 * t + 1] * (__uint_as_float(dr[2 * t + 1]) - Dq));
                tmem_st8(lane_base + DQ_TM_DS + sb * (SUB / 2) + 8 * cg, pd);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ds_full[sb]);
            }
            if (!ok) break;
            ok = mbar_wait(&acc_full[ab], (uint32_t)((it >> 1) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            // groups 0 and 1 write the dQ rows, columns 0..31 and 32..63
            uint32_t dq[32];
            if (cg < 2) {
                tmem_ld32_nowait(lane_base + DQ_TM_DQ + ab * AT_HS + 32 * cg, dq);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[ab]);
            if (cg < 2) {
                if (lane == 0) tma_wait_read<0>();
                __syncwarp();
                stage_out_slab32(slab, lane, dq, 0.125f);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int row0 = qb * AT_BQ + q4 * 32;
                    if (row0 < T) tma_store_3d(&tm_out, slab, h * AT_HS + 32 * cg, row0, b);
                    tma_commit();
                }
            }
            g += n;
        }
        if (lane == 0) tma_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 5;
    }
    if (warp == BW_ISSUE0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, BW_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
cudaError_t attention_bwd_tc(const bf16* qkv, const bf16* out, const bf16* dout, const float* lse,
                             float* D, bf16* dqkv, int B, int T, int H, int hs, DevState* st,
                             cudaStream_t s) {
    if (hs != AT_HS || T < 1 || B < 1 || H < 1 || !st) return cudaErrorInvalidValue;
    if (((uintptr_t)qkv & 15) || ((uintptr_t)dout & 15) || ((uintptr_t)dqkv & 15) || ((uintptr_t)out & 15))
        return cudaErrorInvalidValue;
    const int C = H * hs;
    // 128-row tiles of the item, 64-row sub-blocks of the streamed operand
    CUtensorMap q128, q64, do128, do64, o128, dqkv_out;
    if (!make_rows_map(&q128, qkv, B, T, 3 * C, AT_BQ, true) || !make_rows_map(&q64, qkv, B, T, 3 * C, SUB, true) ||
        !make_rows_map(&do128, dout, B, T, C, AT_BQ, true) || !make_rows_map(&do64, dout, B, T, C, SUB, true) ||
        !make_rows_map(&o128, out, B, T, C, AT_BQ, true) ||
        !make_rows_map(&dqkv_out, dqkv, B, T, 3 * C, 32, false, 32))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        // the dQ kernel's register split assumes the launch's DQ_REGS per thread
        cudaFuncAttributes fa;
        CUDA_OK(cudaFuncGetAttributes(&fa, fa_tc_bwd_dq_kernel));
        if (fa.numRegs != DQ_REGS) return cudaErrorInvalidConfiguration;
        CUDA_OK(cudaFuncSetAttribute(fa_tc_bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)KV_SMEM));
        CUDA_OK(cudaFuncSetAttribute(fa_tc_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)DQ_SMEM));
        attr_done.fetch_or(dbit);
    }
    const int items = ((T + AT_BQ - 1) / AT_BQ) * B * H;
    const int grid = items < num_sms() ? items : num_sms();
    // the dQ kernel also computes D = rowsum(dO * O), which the dK/dV kernel reads
    (void)pdl_launch(fa_tc_bwd_dq_kernel, grid, DQ_THREADS, DQ_SMEM, s, q128, q64, do128, o128, dqkv_out, lse, D, T, H,
                                                          B * H, st);
    CUDA_OK(cudaGetLastError());
    (void)pdl_launch(fa_tc_bwd_dkv_kernel, grid, KV_THREADS, KV_SMEM, s, q128, q64, do64, dqkv_out, lse, D, T, H, B * H, st);
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
