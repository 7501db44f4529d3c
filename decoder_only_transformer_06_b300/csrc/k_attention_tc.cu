// Causal flash attention forward on the 5th-generation tensor cores (tcgen05,
// sm_103a): bf16 q, k, v, fp32 scores and output accumulation in tensor memory.
//
// Semantics: the manual attention of nanoGPT's CausalSelfAttention (nanoGPT
// guide Deep dive 1): S = q k^T / sqrt(hs), keys j > i masked to -inf before
// the softmax, o = softmax(S) v; the T x T scores never leave the chip (online
// softmax over key blocks: "Let's reproduce GPT-2" 02:00:18, Flash Attention).
// Also writes lse = log sum_j exp(S_ij) per query for the backward.
//
// Work item = (128-query block, b, h); persistent CTAs, 384 threads:
//   warps 0..7  softmax, two warps per query row: warp w reads TMEM lane
//               quarter w % 4 (its 32 rows) and the key half hf = w / 4
//               (columns 64 hf .. +63) of each 128-key block. Each half keeps
//               its own running max m and row sum l and its own output
//               accumulator O_hf (the online softmax of its keys), so the two
//               warps of a row never wait for each other inside an item; at
//               the item's end the halves combine exactly:
//                 O = (O_0 2^(m_0 - M) + O_1 2^(m_1 - M)) / (l_0 2^(m_0 - M) + l_1 2^(m_1 - M)),
//               M = max(m_0, m_1) (log2 units). P = exp(S - m) is written in
//               bf16 over the warp's own, already read S columns in TMEM, where
//               the P V product reads it as its A operand; a half rescales its
//               O_hf when its max grew by more than 2^8 (otherwise P may exceed
//               1 by up to 2^8, which the final division absorbs exactly).
//   warp 8      TMA producer: Q once per item, then K and V of each block of
//               128 keys into one slot of a five-slot ring.
//   warp 9      allocates 512 TMEM columns (S triple buffer, the two halves'
//               O); lane 0 issues S_j = Q K_j^T (M=128, N=128, K=64) into
//               S[j%3] once the P V products that read the P written over it
//               are done.
//   warps 10,11 lane 0 of warp 10 + hf issues O_hf += P_hf V_hf as soon as that
//               half's P is in TMEM (M=128, N=64, K=64; A = P from TMEM): one
//               issuing thread sustains about one tcgen05.mma per hundred
//               cycles, so each half has its own. The tensor core computes
//               S_{j+1}, S_{j+2} and P_j V_j while the softmax works on S_{j+1}.
// An item's output is written after the next item's first key block (by then
// its last P V products have landed): each softmax warp combines the halves
// for its 32 rows and 32 of the 64 columns and sends them through a 2 KB
// shared-memory slab and one TMA store. Warps 8..11 give up registers to the
// softmax warpgroups (setmaxnreg). Every mbarrier wait is bounded; on expiry
// the CTA records ERR_TIMEOUT, drains its copies and MMAs (bounded), frees TMEM
// and returns.
#include "attn_tc.cuh"

namespace k {

using namespace tc;
using namespace attn;

namespace {

constexpr int AT_SLOTS = 5;                    // K and V ring depth (32 KB a slot)
constexpr int FW_THREADS = 384;                // forward: 8 softmax warps, producer, three MMA issuers
constexpr int FW_PRODUCER = 8, FW_ISSUE_S = 9, FW_ISSUE_PV = 10;   // P V issuers: warps 10, 11
constexpr int FW_SBUF = 3;                     // S buffers in TMEM
// Registers: the launch gives each of the 384 threads FW_REGS; the producer
// and issuer warpgroup (warps 8..11) then drops to FW_REGS_LOW and the two
// softmax warpgroups rise to FW_REGS_HIGH (setmaxnreg). The shares must add up
// to no more than the launch's total, or the increase would wait forever; the
// host checks that the kernel was compiled with FW_REGS registers.
constexpr int FW_REGS = 168, FW_REGS_LOW = 56, FW_REGS_HIGH = 224;
static_assert(4 * FW_REGS_LOW + 8 * FW_REGS_HIGH <= 12 * FW_REGS, "register split exceeds the launch");
constexpr int OFF_Q = 0;                       // Q double buffer
constexpr int OFF_K = OFF_Q + 2 * AT_TILE;
constexpr int OFF_V = OFF_K + AT_SLOTS * AT_TILE;
constexpr int OFF_OUT = OFF_V + AT_SLOTS * AT_TILE;   // [4 row quarters][2 column halves] 2 KB O slabs
constexpr int OFF_ML = OFF_OUT + 4 * OUT_SLAB;        // [2 item buffers][2 halves][128 rows] (m, l)
constexpr int OFF_BAR = OFF_ML + 2 * 2 * 128 * 8;
constexpr size_t AT_SMEM = OFF_BAR + 512 + 1024;
// forward TMEM columns: S[i] 128 i .. 128 i + 127 for i < 3 (P of half hf in
// bf16 pairs over columns 64 hf .. 64 hf + 31 of its S buffer), O_0 384..447,
// O_1 448..511 (one item at a time)
constexpr uint32_t TM_O = 384;
constexpr uint32_t AT_TMEM_COLS = 512;

}  // namespace

// Persistent: one CTA per SM walks work items w = blockIdx.x, +gridDim.x, ...
// ordered heaviest first (query block qb = nqb-1 - w / (B*H)). Barrier phases
// run on counters that every role advances identically: g counts key blocks
// over all items (K/V ring slots, S buffers), `it` counts items (Q double
// buffer, the O accumulators, the (m, l) hand-off).
__global__ void __launch_bounds__(FW_THREADS, 1)
fa_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_out,
                 float* __restrict__ lse, int T, int H, int BH, DevState* st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sQ = smem + OFF_Q;
    uint8_t* sK = smem + OFF_K;
    uint8_t* sV = smem + OFF_V;
    float2* sML = (float2*)(smem + OFF_ML);
    uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
    uint64_t* q_full = bars;           // [2]
    uint64_t* q_empty = bars + 2;      // [2]
    uint64_t* kv_full = bars + 4;                  // [AT_SLOTS] K and V block j
    uint64_t* kv_empty = kv_full + AT_SLOTS;       // [AT_SLOTS]
    uint64_t* s_full = kv_empty + AT_SLOTS;        // [FW_SBUF]
    uint64_t* p_full = s_full + FW_SBUF;           // [FW_SBUF buffers][2 halves]
    uint64_t* pv_done = p_full + 2 * FW_SBUF;      // [FW_SBUF] both halves' P V products of the block
    uint64_t* o_free = pv_done + FW_SBUF;          // the O accumulators have been read
    uint64_t* ml_full = o_free + 1;                // [2] both halves' (m, l) of an item are in smem
    uint64_t* drain = ml_full + 2;                 // [3] one per issuing thread
    uint32_t* tmem_slot = (uint32_t*)(drain + 3);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int nqb = (T + AT_BQ - 1) / AT_BQ;
    const int items = nqb * BH;
    const int C = H * AT_HS;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
            mbar_init(&ml_full[i], 8);
        }
        for (int i = 0; i < FW_SBUF; i++) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[2 * i], 4);
            mbar_init(&p_full[2 * i + 1], 4);
            mbar_init(&pv_done[i], 2);
            mbar_init(&drain[i], 1);
        }
        mbar_init(o_free, 8);
        for (int s = 0; s < AT_SLOTS; s++) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 2);      // both P V issuers
        }
        abort_flag[0] = 0;
        abort_flag[1] = (int)wait_limit_of(st);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == FW_ISSUE_S) tmem_alloc(tmem_slot, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();                              // the previous kernel's outputs are visible

    if (warp >= FW_PRODUCER) {
    // one register-split instruction per warpgroup (all four warps run it)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(FW_REGS_LOW));
    if (warp == FW_PRODUCER) {
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
            pdl_trigger();                   // every copy of this CTA is issued
            if (!ok || *abort_flag) {
                // wait (bounded) for every copy still in flight before the CTA exits
                for (int i = (nq > 2 ? nq - 2 : 0); i < nq; i++) wait_bounded(&q_full[i & 1], (uint32_t)((i >> 1) & 1));
                for (int i = (nkv_l > AT_SLOTS ? nkv_l - AT_SLOTS : 0); i < nkv_l; i++)
                    wait_bounded(&kv_full[i % AT_SLOTS], (uint32_t)((i / AT_SLOTS) & 1));
            }
        }
    } else if (warp == FW_ISSUE_S) {
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
                    const int G = g + j, s = G % AT_SLOTS, sb = G % FW_SBUF;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / AT_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    // S[sb] is free once the P V products of three blocks ago (which read
                    // the P written over it) are done
                    if (!mbar_wait(&pv_done[sb], (uint32_t)(((G / FW_SBUF) & 1) ^ 1), abort_flag)) { ok = false; break; }
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
    } else {
        if (lane == 0) {
            // ---------------- O_hf += P_hf V_hf issuer, hf = warp - 10 (P from TMEM,
            // V rows 64 hf .. +63 read MN-major)
            const int hf = warp - FW_ISSUE_PV;
            constexpr uint32_t id_o = make_idesc(AT_BQ, AT_HS, false, true);
            const uint64_t dv0 = smem_desc(smem_u32(sV), 8192, 1024);
            const uint32_t to = tmem_base + TM_O + 64 * hf;
            bool ok = true, any = false;
            int g = 0, it = 0;
            for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
                const int qb = nqb - 1 - w / BH;
                const int nkv = qb + 1;
                if (!mbar_wait(o_free, (uint32_t)((it & 1) ^ 1), abort_flag)) { ok = false; break; }
                for (int j = 0; j < nkv; j++) {
                    const int G = g + j, s = G % AT_SLOTS, pb = G % FW_SBUF;
                    if (!mbar_wait(&kv_full[s], (uint32_t)((G / AT_SLOTS) & 1), abort_flag)) { ok = false; break; }
                    if (!mbar_wait(&p_full[2 * pb + hf], (uint32_t)((G / FW_SBUF) & 1), abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dv = desc_adv(dv0, s * AT_TILE + hf * 8192);
                    const uint32_t tp = tmem_base + pb * AT_BK + 64 * hf;
#pragma unroll
                    for (int kk = 0; kk < 4; kk++)
                        mma_bf16_ta(to, tp + kk * 8, desc_adv(dv, kk * 2048), id_o, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&pv_done[pb]);
                    mma_commit(&kv_empty[s]);
                    any = true;
                }
                g += nkv;
            }
            if (any) {
                mma_commit(&drain[1 + hf]);
                wait_bounded(&drain[1 + hf], 0);
            }
        }
    }
    } else {
        // ---------------- softmax warps 0..7: warp w owns rows r = 32 (w % 4) + lane
        // (TMEM lane r) and the key half hf = w / 4 of every block
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(FW_REGS_HIGH));
        const int q4 = warp & 3, hf = warp >> 2;
        const int r = q4 * 32 + lane;
        const float sl2 = LOG2E_F * 0.125f;   // log2(e) / sqrt(64)
        const uint32_t lane_base = tmem_base + ((uint32_t)(q4 * 32) << 16);
        uint8_t* slab = smem + OFF_OUT + q4 * OUT_SLAB + hf * (OUT_SLAB / 2);
        bool ok = true;
        int g = 0, it = 0;
        // The output of an item is written after the first key block of the
        // next one (its last P V products have landed by then, so nothing waits
        // for them). The pending item is the previous one of this CTA: work
        // item p_w, item count p_it, its last key block p_GL.
        auto item_output = [&](int p_w, int p_it, int p_GL) -> bool {
            const int p_qb = nqb - 1 - p_w / BH, p_bh = p_w % BH;
            const int p_h = p_bh % H, p_b = p_bh / H, pq = p_qb * AT_BQ + r, pob = p_it & 1;
            bool okk = mbar_wait(&pv_done[p_GL % FW_SBUF], (uint32_t)((p_GL / FW_SBUF) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, okk)) return false;
            okk = mbar_wait(&ml_full[pob], (uint32_t)((p_it >> 1) & 1), abort_flag);
            if (!__all_sync(0xffffffffu, okk)) return false;
            // each half writes output columns 32 hf .. 32 hf + 31 of its rows
            // from both O halves
            const float2 ml0 = sML[(pob * 2) * 128 + r], ml1 = sML[(pob * 2 + 1) * 128 + r];
            const float M = fmaxf(ml0.x, ml1.x);
            const float w0 = ml0.x == -INFINITY ? 0.f : ex2f(ml0.x - M);
            const float w1 = ml1.x == -INFINITY ? 0.f : ex2f(ml1.x - M);
            const float l_row = ml0.y * w0 + ml1.y * w1;
            const float a0 = w0 / l_row, a1 = w1 / l_row;
            tc_fence_after();
            if (lane == 0) tma_wait_read<0>();           // the previous output store has read the slab
            __syncwarp();
#pragma unroll 1
            for (int k2 = 0; k2 < 2; k2++) {
                uint32_t o0[16], o1[16];
                tmem_ld16_nowait(lane_base + TM_O + 32 * hf + 16 * k2, o0);
                tmem_ld16_nowait(lane_base + TM_O + 64 + 32 * hf + 16 * k2, o1);
                tmem_wait_ld();
#pragma unroll
                for (int pc = 0; pc < 2; pc++) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; e++)
                        v[e] = __uint_as_float(o0[8 * pc + e]) * a0 + __uint_as_float(o1[8 * pc + e]) * a1;
                    const int piece = 2 * k2 + pc;
                    *(uint4*)(slab + lane * 64 + ((piece ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]), pack2_bf16(v[4], v[5]),
                                   pack2_bf16(v[6], v[7]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&tm_out, slab, p_h * AT_HS + 32 * hf, p_qb * AT_BQ + q4 * 32, p_b);
                tma_commit();
            }
            if (hf == 0 && pq < T) lse[(int64_t)p_bh * T + pq] = (M + log2f(l_row)) * LN2;
            return true;
        };
        for (int w = blockIdx.x; w < items && ok; w += gridDim.x, it++) {
            const int qb = nqb - 1 - w / BH;
            const int nkv = qb + 1;
            const int q = qb * AT_BQ + r;
            const int ob = it & 1;                 // the (m, l) hand-off buffer
            const uint32_t o_half = lane_base + TM_O + 64 * hf;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; j < nkv; j++) {
                const int G = g + j, sb = G % FW_SBUF;
                ok = mbar_wait(&s_full[sb], (uint32_t)((G / FW_SBUF) & 1), abort_flag);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[64];
                const uint32_t s_addr = lane_base + (uint32_t)(sb * AT_BK + 64 * hf);
                tmem_ld32_nowait(s_addr, sr);
                tmem_ld32_nowait(s_addr + 32, sr + 32);
                tmem_wait_ld();
                // mask (raw scores; the scale is applied in the exponent), this half's max
                const int key0 = j * AT_BK + 64 * hf;
                if ((j == qb) || (key0 + 64 > T)) {
#pragma unroll
                    for (int i = 0; i < 64; i++)
                        if (key0 + i > q || key0 + i >= T) sr[i] = __float_as_uint(-INFINITY);
                }
                float pm[8];
#pragma unroll
                for (int t = 0; t < 8; t++) pm[t] = __uint_as_float(sr[t]);
#pragma unroll
                for (int i = 8; i < 56; i += 16)
#pragma unroll
                    for (int t = 0; t < 8; t++)
                        pm[t] = fmax3f(pm[t], __uint_as_float(sr[i + t]), __uint_as_float(sr[i + 8 + t]));
#pragma unroll
                for (int t = 0; t < 8; t++) pm[t] = fmaxf(pm[t], __uint_as_float(sr[56 + t]));
                const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                       fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * sl2;
                const float m_new = fmaxf(m_run, mx);
                // a half whose keys were all masked so far keeps m = -inf, l = 0, O = 0
                const bool resc = (j > 0) && (m_new > m_run + 8.f);
                if (__any_sync(0xffffffffu, resc)) {
                    // rescale O_hf once the previous block's P V products have landed
                    ok = mbar_wait(&pv_done[(G - 1) % FW_SBUF], (uint32_t)(((G - 1) / FW_SBUF) & 1), abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    const float f = resc ? ex2f(m_run - m_new) : 1.f;
                    uint32_t o[32];
#pragma unroll
                    for (int c2 = 0; c2 < 2; c2++) {
                        tmem_ld32(o_half + 32 * c2, o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                        tmem_st32(o_half + 32 * c2, o);
                    }
                    if (resc) {
                        l_run *= f;
                        m_run = m_new;
                    }
                }
                if (j == 0) m_run = m_new;
                const float msub = m_run == -INFINITY ? 0.f : m_run;   // all masked: exps of -inf are 0
                // exponents and partial sums two columns at a time on the packed
                // fp32 pipe; ps[t] sums columns 2c, 2c+1 for c = t mod 4
                uint64_t ps[4] = {0ull, 0ull, 0ull, 0ull};
                uint32_t pk[32];                    // 64 probabilities as bf16 pairs
                const uint64_t sl2x2 = f2(sl2, sl2), nmx2 = f2(-msub, -msub);
#pragma unroll
                for (int c = 0; c < 32; c++) {
                    float a0, a1;
                    f2_split(f2_fma(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sl2x2, nmx2),
                             a0, a1);
                    const float e0 = ex2f(a0), e1 = ex2f(a1);
                    const uint64_t e = f2(e0, e1);
                    ps[c & 3] = f2_add(ps[c & 3], e);
                    pk[c] = pack2_bf16(e0, e1);
                }
                // over this warp's own S columns, already in registers
                tmem_st32(s_addr, pk);
                float psum[8];
#pragma unroll
                for (int t = 0; t < 4; t++) f2_split(ps[t], psum[2 * t], psum[2 * t + 1]);
                l_run += ((psum[0] + psum[1]) + (psum[2] + psum[3])) + ((psum[4] + psum[5]) + (psum[6] + psum[7]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[2 * sb + hf]);
                if (j == 0 && it > 0) {
                    ok = item_output(w - (int)gridDim.x, it - 1, g - 1);
                    if (!ok) break;
                }
            }
            if (!ok) break;
            // hand this half's (m, l) to the item's output, written after the
            // next item's first key block
            sML[(ob * 2 + hf) * 128 + r] = make_float2(m_run, l_run);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ml_full[ob]);
            g += nkv;
        }
        if (ok && it > 0) ok = item_output(blockIdx.x + (it - 1) * (int)gridDim.x, it - 1, g - 1);
        if (lane == 0) tma_wait_all();
    }
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 3;
    }
    if (warp == FW_ISSUE_S) {
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
    // qkv [B, T, 3C] read in 128-row boxes; out written by per-warp 32 x 32 stores
    if (!make_rows_map(&map, qkv, B, T, 3 * H * hs, AT_BQ, true) ||
        !make_rows_map(&omap, out, B, T, H * hs, 32, false, 32))
        return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};   // per device
    const unsigned long long dbit = device_bit();
    if (!(attr_done.load() & dbit)) {
        // the register split assumes the launch's FW_REGS per thread
        cudaFuncAttributes fa;
        CUDA_OK(cudaFuncGetAttributes(&fa, fa_tc_fwd_kernel));
        if (fa.numRegs != FW_REGS) return cudaErrorInvalidConfiguration;
        CUDA_OK(cudaFuncSetAttribute(fa_tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AT_SMEM));
        attr_done.fetch_or(dbit);
    }
    const int items = ((T + AT_BQ - 1) / AT_BQ) * B * H;
    const int grid = items < num_sms() ? items : num_sms();
    (void)pdl_launch(fa_tc_fwd_kernel, grid, FW_THREADS, AT_SMEM, s, map, omap, lse, T, H, B * H, st);
    return cudaGetLastError();
}

}  // namespace k
