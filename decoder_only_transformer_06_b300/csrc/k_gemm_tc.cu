// bf16 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   D[m,n] = sum_k A(m,k) B(n,k), fp32 accumulation in tensor memory (TMEM),
//   followed by a fused epilogue (bias, tanh-GELU, GELU backward, fp32
//   gradient accumulation).
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
//   warps 2..9  epilogue, two per TMEM lane quarter (32 rows of the tile, half
//               the columns each): tcgen05.ld 32 columns at a time (one row
//               per lane), fused math in registers, the result written to a
//               swizzled shared-memory tile and sent out by one TMA store (or
//               TMA reduce-add for the fp32 gradient). A second operand of the
//               epilogue (the GELU derivative saved by the forward) arrives by
//               TMA load, prefetched one chunk ahead.
// Moving epilogue traffic through the TMA engine keeps the SM's load/store
// and shared-memory pipes free for the operand stream of the main loop; with
// per-lane global stores the epilogue, not the tensor pipe, set the pace.
// Two TMEM accumulators (2*BN columns) let the epilogue of one tile overlap
// the main loop of the next. Every mbarrier wait is bounded: on expiry the
// CTA records ERR_TIMEOUT in the device status word, drains its in-flight
// copies and MMAs (again bounded), frees TMEM and returns.
#include "common.cuh"
#include "tc.cuh"
#include <cuda.h>
#include <cstring>

namespace k {

using namespace tc;

static constexpr int TC_BM = 128, TC_BK = 64;
static constexpr int EPI_WARPS = 8;
static constexpr int TC_THREADS = 32 * (2 + EPI_WARPS);

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

// ------------------------------------------------------------------ epilogue math
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
// gelu(x) = 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), and
// gelu'(x) = 0.5 (1 + t) + 0.5 x (1 - t^2) du/dx from one tanh, for two
// values at a time on the packed fp32 pipe (the epilogue of the fc Linear is
// bound by these instructions):
//   x2 = x*x, u = x (k0 + k1 x2), t = tanh(u), hx = x/2, g = hx t + hx,
//   gelu' = (hx (t*t - 1)) (-(k0 + 3 k1 x2)) + (t/2 + 1/2).
__device__ __forceinline__ void gelu_and_grad_x2(float& xa, float& xb, float& ga, float& gb) {
    const float k0 = 0.7978845608028654f;              // sqrt(2/pi)
    const float k1 = 0.7978845608028654f * 0.044715f;
    const uint64_t x = f2(xa, xb);
    const uint64_t x2 = f2_mul(x, x);
    float ua, ub;
    f2_split(f2_mul(x, f2_fma(f2(k1, k1), x2, f2(k0, k0))), ua, ub);
    const uint64_t t = f2(tanh_hw(ua), tanh_hw(ub));
    const uint64_t half = f2(0.5f, 0.5f);
    const uint64_t hx = f2_mul(half, x);
    f2_split(f2_fma(hx, t, hx), ga, gb);
    const uint64_t q = f2_mul(hx, f2_fma(t, t, f2(-1.0f, -1.0f)));
    const uint64_t nd = f2_fma(f2(-3.0f * k1, -3.0f * k1), x2, f2(-k0, -k0));
    f2_split(f2_fma(q, nd, f2_fma(half, t, half)), xa, xb);
}

// Staging tiles are laid out as the TMA expects them with swizzling, which
// also makes the per-row writes (one row per lane) bank-conflict free:
//   bf16 32x32 tile, 64 B rows, 64B swizzle: 16-byte piece q of row r sits at
//     r*64 + ((q ^ ((r >> 1) & 3)) << 4)
//   fp32 32x32 tile, 128 B rows, 128B swizzle: piece q of row r at
//     r*128 + ((q ^ (r & 7)) << 4)
__device__ __forceinline__ uint32_t sw64(int r, int q) { return r * 64 + ((q ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ uint32_t sw128(int r, int q) { return r * 128 + ((q ^ (r & 7)) << 4); }

// Row `lane` of a bf16 32x32 staging tile from 32 fp32 values.
__device__ __forceinline__ void stage_bf16(uint8_t* tile, int lane, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        *(uint4*)(tile + sw64(lane, q)) = w;
    }
}
__device__ __forceinline__ void stage_f32(uint8_t* tile, int lane, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 8; q++)
        *(float4*)(tile + sw128(lane, q)) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
__device__ __forceinline__ void unstage_bf16(const uint8_t* tile, int lane, float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint4 w = *(const uint4*)(tile + sw64(lane, q));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 f = __bfloat1622float2(*(const __nv_bfloat162*)&u[j]);
            v[8 * q + 2 * j] = f.x;
            v[8 * q + 2 * j + 1] = f.y;
        }
    }
}

// ------------------------------------------------------------------ kernel
// PAIR: the tile is 256 x BN and is shared by a cluster of two CTAs (one
// tcgen05.mma with cta_group::2 covers both): each CTA stages its own 128 rows
// of A and half (BN/2 rows) of B, and holds its own 128 x BN accumulator.
// The GELU epilogue (two outputs) gets 8 KB of staging per warp instead of 4 KB,
// paid for by one operand stage: its GEMM has K = d_model, where five stages
// still cover the copy latency. (The GELU-backward epilogue measured slower
// with the same trade and a deeper prefetch of its extra operand, so it keeps
// six stages and prefetches that operand one chunk ahead.)
template <int BN, bool PAIR, int KIND>
struct TcCfg {
    static constexpr bool WIDE_EPI = (KIND == EPI_GELU);
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = B_ROWS * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = STAGE_BYTES == 32768 ? (WIDE_EPI ? 5 : 6) : (WIDE_EPI ? 3 : 4);
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_WARP_BYTES = WIDE_EPI ? 8192 : 4096;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
    static constexpr int AUX_RING = 1;            // GELU-derivative chunks in flight per warp
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + EPI_BYTES + 1024 + 512;
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Tensor maps of the epilogue: o1 (bf16 out / fp32 out / fp32 reduce target /
// GELU derivative), o2 (GELU post-activation), aux (GELU derivative to read).
struct EpiMaps {
    CUtensorMap o1, o2, aux;
};

template <int BN, bool A_MN, bool B_MN, int KIND, bool PAIR>
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ EpiMaps maps, int M, int N, int K, int splits,
               const float* __restrict__ bias, float* __restrict__ colsum, DevState* st) {
    using Cfg = TcCfg<BN, PAIR, KIND>;
    constexpr int STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* sEpi = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* full = (uint64_t*)(sEpi + Cfg::EPI_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* auxbar = tempty + 2;              // [EPI_WARPS][AUX_RING]
    uint64_t* drain = auxbar + EPI_WARPS * Cfg::AUX_RING;
    uint32_t* tmem_slot = (uint32_t*)(drain + 1);
    volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // pair: rank 0 issues the MMAs; its full[] barriers count both CTAs'
    // operand bytes and its tempty[] barriers both CTAs' epilogue warps
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
        }
        for (int i = 0; i < EPI_WARPS * Cfg::AUX_RING; i++) mbar_init(&auxbar[i], 1);
        mbar_init(drain, 1);
        abort_flag[0] = 0;
        // a pair keeps the full limit (see wait_limit_of)
        abort_flag[1] = (int)(PAIR ? (unsigned int)WAIT_LIMIT_CYCLES : wait_limit_of(st));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        if constexpr (PAIR) tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        else tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync();      // the peer's barriers exist before any remote arrive
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();                              // the previous kernel's outputs are visible
    // work is dealt per pair: both CTAs of a cluster walk the same tile list
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr int TILE_M = PAIR ? 2 * TC_BM : TC_BM;

    const int num_m = (M + TILE_M - 1) / TILE_M;
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
            // the barrier that counts this CTA's bytes: its own, or the leader's
            const uint32_t full0 = PAIR ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
            for (int w = unit; w < total && ok; w += units) {
                int split = w / tiles, mt, nt;
                tile_coords(w - split * tiles, num_m, num_n, mt, nt);
                const int m_row = mt * TILE_M + (int)rank * TC_BM;
                const int n_row = nt * BN + (int)rank * Cfg::B_ROWS;
                int kb0 = split * kpb, kb1 = min(kb0 + kpb, kblocks);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) { ok = false; break; }
                    if (leader) mbar_arrive_expect_tx(&full[stage], (PAIR ? 2 : 1) * Cfg::STAGE_BYTES);
                    uint8_t* a = sA + stage * Cfg::A_BYTES;
                    uint8_t* b = sB + stage * Cfg::B_BYTES;
                    const int k0 = kb * TC_BK;
                    if constexpr (PAIR) {
                        const uint32_t fb = full0 + (uint32_t)stage * 8u;
                        if (!A_MN) {
                            tma_load_2d_pair(a, &tmA, fb, k0, m_row);
                        } else {
                            tma_load_2d_pair(a, &tmA, fb, m_row, k0);
                            tma_load_2d_pair(a + 8192, &tmA, fb, m_row + 64, k0);
                        }
                        if (!B_MN) {
                            tma_load_2d_pair(b, &tmB, fb, k0, n_row);
                        } else {
#pragma unroll
                            for (int j = 0; j < Cfg::B_ROWS / 64; j++)
                                tma_load_2d_pair(b + j * 8192, &tmB, fb, n_row + 64 * j, k0);
                        }
                    } else {
                        if (!A_MN) {
                            tma_load_2d(a, &tmA, &full[stage], k0, m_row);
                        } else {
                            tma_load_2d(a, &tmA, &full[stage], m_row, k0);
                            tma_load_2d(a + 8192, &tmA, &full[stage], m_row + 64, k0);
                        }
                        if (!B_MN) {
                            tma_load_2d(b, &tmB, &full[stage], k0, n_row);
                        } else {
#pragma unroll
                            for (int j = 0; j < BN / 64; j++)
                                tma_load_2d(b + j * 8192, &tmB, &full[stage], n_row + 64 * j, k0);
                        }
                    }
                    issued++;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            pdl_trigger();                   // every copy of this CTA is issued
            // the peer's copies complete on the leader's barriers, which the
            // leader's MMA issuer waits for; only the leader drains here
            if (leader && (!ok || *abort_flag)) {
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
        if (lane == 0 && leader) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = make_idesc(TILE_M, BN, A_MN, B_MN);
            constexpr uint32_t A_LBO = A_MN ? 8192 : 16, B_LBO = B_MN ? 8192 : 16;
            constexpr uint32_t KSTEP_A = A_MN ? 2048 : 32, KSTEP_B = B_MN ? 2048 : 32;
            const uint64_t dA0 = smem_desc(smem_u32(sA), A_LBO, 1024);
            const uint64_t dB0 = smem_desc(smem_u32(sB), B_LBO, 1024);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int w = unit; w < total && ok; w += units) {
                int split = w / tiles;
                int kb0 = split * kpb, kb1 = min(kb0 + kpb, kblocks);
                if (!(PAIR ? mbar_wait_cluster(&tempty[acc], acc_phase ^ 1, abort_flag)
                           : mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag))) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!mbar_wait(&full[stage], phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = desc_adv(dA0, stage * Cfg::A_BYTES);
                    const uint64_t bd = desc_adv(dB0, stage * Cfg::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / 16; kk++) {
                        if constexpr (PAIR)
                            mma_bf16_pair(d_tmem, desc_adv(ad, kk * KSTEP_A), desc_adv(bd, kk * KSTEP_B),
                                          idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                        else
                            mma_bf16(d_tmem, desc_adv(ad, kk * KSTEP_A), desc_adv(bd, kk * KSTEP_B), idesc,
                                     (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    if constexpr (PAIR) mma_commit_pair(&empty[stage], 3);
                    else mma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if constexpr (PAIR) mma_commit_pair(&tfull[acc], 3);
                else mma_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
            if constexpr (PAIR) {
                // every MMA of the pair completes (in both CTAs' TMEM and
                // shared memory) before either CTA releases them
                mma_commit_pair(drain, 3);
            } else if (any) {
                // all MMAs of this CTA complete before TMEM is released
                mma_commit(drain);
                const long long t0 = wait_clock();
                while (!mbar_try_wait(drain, 0) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
            }
        }
        if (PAIR && lane == 0) {
            const long long t0 = wait_clock();
            while (!mbar_try_wait_cluster(drain, 0) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
        }
    } else {
        // ---------------- epilogue warps 2..9: TMEM lane quarter q4 = warp % 4
        // (the hardware's access rule), i.e. rows q4*32..q4*32+31 of the tile;
        // the two warps of a quarter take the left and right half of the columns.
        // Each warp stages through its own 4 KB (8 KB for GELU):
        //   STORE_ACT  bf16 result in alternating 2 KB halves, so that one TMA
        //              store can still be reading while the next chunk is written
        //   GELU       gelu'(pre) and gelu(pre), 2 KB each, in alternating 4 KB sets
        //   GELU_BWD   the bf16 result in 2 KB, then AUX_RING 2 KB slots of the
        //              GELU derivative operand, loaded by TMA AUX_RING chunks
        //              ahead (across tile boundaries)
        //   fp32 kinds one 32x32 fp32 tile in all 4 KB
        const int ew = warp - 2;
        const int q4 = warp & 3;
        const int half = ew >> 2;
        constexpr int NCH = BN / 64;                 // 32-column chunks per warp per tile
        constexpr int NA = Cfg::AUX_RING;
        constexpr bool ALT = (KIND == EPI_STORE_ACT || KIND == EPI_GELU);
        constexpr uint32_t ALT_BYTES = KIND == EPI_GELU ? 4096u : 2048u;
        uint8_t* wbuf = sEpi + ew * Cfg::EPI_WARP_BYTES;
        uint8_t* aring = wbuf + 2048;
        uint64_t* abar = auxbar + ew * NA;
        // The GELU derivative chunks of this warp, in the order the epilogue uses
        // them (tile by tile, NCH chunks each), go into ring slot q % NA. The
        // next chunk to load is chunk a_c of tile a_w, whose corner is (a_x, a_y).
        long a_issued = 0, a_used = 0;
        int a_w = unit, a_c = 0, a_x = 0, a_y = 0;
        auto aux_tile = [&]() {
            if (a_w >= total) return;
            const int split = a_w / tiles;
            int mt, nt;
            tile_coords(a_w - split * tiles, num_m, num_n, mt, nt);
            a_x = nt * BN + half * (BN / 2);
            a_y = mt * TILE_M + (int)rank * TC_BM + q4 * 32;
        };
        auto issue_aux = [&]() {
            if (a_w >= total) return;
            const int slot = (int)(a_issued % NA);
            mbar_arrive_expect_tx(&abar[slot], 2048);
            tma_load_2d(aring + slot * 2048, &maps.aux, &abar[slot], a_x + 32 * a_c, a_y);
            a_issued++;
            if (++a_c == NCH) {
                a_c = 0;
                a_w += units;
                aux_tile();
            }
        };
        if (KIND == EPI_GELU_BWD && lane == 0) {
            aux_tile();
            for (int q = 0; q < NA; q++) issue_aux();
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        uint32_t seq = 0;
        bool ok = true;
        // the MMA issuer's tempty[] barriers (the leader's, in a pair)
        const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);
        for (int w = unit; w < total && ok; w += units) {
            int split = w / tiles, mt, nt;
            tile_coords(w - split * tiles, num_m, num_n, mt, nt);
            const int m_base = mt * TILE_M + (int)rank * TC_BM + q4 * 32;
            const int n_half = nt * BN + half * (BN / 2);
            // this warp's bias values, column n_half + 32 c + lane in breg[c], loaded
            // before the accumulator is waited for (their latency overlaps the wait)
            float breg[NCH];
#pragma unroll
            for (int c = 0; c < NCH; c++) {
                const int n = n_half + 32 * c + lane;
                breg[c] = (bias != nullptr && n < N) ? __ldg(bias + n) : 0.f;
            }
            ok = mbar_wait(&tfull[acc], acc_phase, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN + half * (BN / 2));
            // the TMEM loads run one chunk ahead of the math
            uint32_t rb[2][32];
            tmem_ld32_nowait(t_row, rb[0]);
#pragma unroll
            for (int c = 0; c < NCH; c++, seq++) {
                const int n0 = n_half + 32 * c;
                uint8_t* sbuf = wbuf + (ALT ? (seq & 1) * ALT_BYTES : 0);
                tmem_wait_ld();
                if (c + 1 < NCH) tmem_ld32_nowait(t_row + 32 * (c + 1), rb[(c + 1) & 1]);
                if (c == NCH - 1) {
                    // the accumulator is free for the MMA once its last chunk is in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR) mbar_arrive_cluster(tempty0 + (uint32_t)acc * 8u);
                        else mbar_arrive(&tempty[acc]);
                    }
                }
                const uint32_t(&rc)[32] = rb[c & 1];
                float v[32];
                if (bias != nullptr) {
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        f2_split(f2_add(f2(__uint_as_float(rc[j]), __uint_as_float(rc[j + 1])),
                                        f2(__shfl_sync(0xffffffffu, breg[c], j),
                                           __shfl_sync(0xffffffffu, breg[c], j + 1))),
                                 v[j], v[j + 1]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j++) v[j] = __uint_as_float(rc[j]);
                }
                if (KIND == EPI_GELU_BWD) {
                    const long q = a_used;
                    const int slot = (int)(q % NA);
                    ok = mbar_wait(&abar[slot], (uint32_t)((q / NA) & 1), abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    a_used = q + 1;
                    float dg[32];
                    unstage_bf16(aring + slot * 2048, lane, dg);
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        f2_split(f2_mul(f2(v[j], v[j + 1]), f2(dg[j], dg[j + 1])), v[j], v[j + 1]);
                    __syncwarp();                        // every lane has read the slot
                    if (lane == 0) issue_aux();          // refill it NA chunks ahead
                }
                // the TMA store that last read this staging area is done
                if (lane == 0) {
                    if (ALT) tma_wait_read<1>();
                    else tma_wait_read<0>();
                }
                __syncwarp();
                if (KIND == EPI_STORE_F32 || KIND == EPI_ACCUM_F32) {
                    stage_f32(sbuf, lane, v);
                } else if (KIND == EPI_GELU) {
                    // o1 = gelu'(pre) (saved for the backward), o2 = gelu(pre)
                    float g[32];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) gelu_and_grad_x2(v[j], v[j + 1], g[j], g[j + 1]);
                    stage_bf16(sbuf, lane, v);
                    stage_bf16(sbuf + 2048, lane, g);
                } else {
                    stage_bf16(sbuf, lane, v);
                }
                if (KIND == EPI_GELU_BWD && colsum != nullptr) {
                    // lane j sums column n0 + j of this warp's 32 rows of the
                    // staged bf16 result, rows in order; one partial per
                    // (32-row group, column), reduced in group order later
                    __syncwarp();
                    float csum = 0.f;
                    const int cq = lane >> 3, ce = lane & 7;
#pragma unroll
                    for (int rr = 0; rr < 32; rr++)
                        csum += __bfloat162float(*(const bf16*)(sbuf + sw64(rr, cq) + 2 * ce));
                    if (n0 + lane < N && m_base < M) colsum[(int64_t)(m_base / 32) * N + n0 + lane] = csum;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0 && n0 < N && m_base < M) {
                    if (KIND == EPI_STORE_F32) {
                        tma_store_3d(&maps.o1, sbuf, n0, m_base, split);
                    } else if (KIND == EPI_ACCUM_F32) {
                        tma_reduce_add_2d(&maps.o1, sbuf, n0, m_base);
                    } else {
                        tma_store_2d(&maps.o1, sbuf, n0, m_base);
                        if (KIND == EPI_GELU) tma_store_2d(&maps.o2, sbuf + 2048, n0, m_base);
                    }
                }
                if (lane == 0) tma_commit();
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        tmem_wait_ld();                              // no TMEM load left in flight after an abort
        if (lane == 0) {
            tma_wait_all();
            // after an abort, prefetches of the GELU derivative may still be in
            // flight: wait for them (bounded) before the CTA exits
            if (KIND == EPI_GELU_BWD) {
                for (long q = a_used; q < a_issued; q++) {
                    const long long t0 = wait_clock();
                    while (!mbar_try_wait(&abar[q % NA], (uint32_t)((q / NA) & 1)) &&
                           wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
                }
            }
        }
    }
    // pair: no remote arrive or copy may still target a CTA that has exited
    tc_fence_before();
    if constexpr (PAIR) cluster_sync();
    else __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        atomicOr(&st->err, ERR_TIMEOUT);
        st->timeout_site = 1;
    }
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
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

// Tensor map of a row-major matrix of `outer` lines of `inner` elements, `ld`
// elements between lines. rank 3 adds a third dimension of `splits` such
// matrices stored back to back (the map's rank must match the dimensionality
// of the TMA instructions that use it). Boxes of box_inner x box_outer (x 1).
static bool make_map(CUtensorMap* map, const void* ptr, CUtensorMapDataType dt, int esize,
                     uint64_t inner, uint64_t outer, int64_t ld, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle sw, int rank = 2, int splits = 1) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, outer, (cuuint64_t)splits};
    cuuint64_t strides[2] = {(cuuint64_t)ld * esize, (cuuint64_t)ld * esize * outer};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (rank != 2 && rank != 3) return false;
    CUresult r = enc(map, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
static bool make_operand_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer) {
    return make_map(map, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, ld, box_inner,
                    box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

bool gemm_bf16_tc_supported(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi) {
    if (M <= 0 || N <= 0 || K <= 0) return false;
    if ((A.ld % 8) || (B.ld % 8)) return false;
    if (!aligned16(A.ptr) || !aligned16(B.ptr)) return false;
    if (!epi.out || !aligned16(epi.out)) return false;
    switch (epi.kind) {
        case EPI_STORE_ACT:
            if (epi.ldo % 8) return false;
            break;
        case EPI_GELU:
            if (epi.ldo % 8 || !epi.out2 || !aligned16(epi.out2) || epi.ldo2 % 8) return false;
            break;
        case EPI_GELU_BWD:
            if (epi.ldo % 8 || !epi.aux || !aligned16(epi.aux) || epi.ld_aux % 8 || epi.bias) return false;
            break;
        case EPI_STORE_F32:
            if (epi.ldo % 4) return false;
            break;
        case EPI_ACCUM_F32:
            if (epi.ldo % 4 || epi.bias) return false;
            break;
        default:
            return false;   // the residual add is fused into the LayerNorm, not done here
    }
    if (!get_encode()) return false;
    return true;
}

// Clusters of two 1-CTA-per-SM GEMM CTAs that can be resident at once.
template <typename Kern>
static int max_pairs(Kern kern, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int BN, bool A_MN, bool B_MN, int KIND, bool PAIR>
static cudaError_t launch_tc(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                             int splits, DevState* st, cudaStream_t s) {
    using Cfg = TcCfg<BN, PAIR, KIND>;
    CUtensorMap ta, tb;
    bool ok = A_MN ? make_operand_map(&ta, A.ptr, (uint64_t)M, (uint64_t)K, A.ld, 64, 64)
                   : make_operand_map(&ta, A.ptr, (uint64_t)K, (uint64_t)M, A.ld, 64, TC_BM);
    ok = ok && (B_MN ? make_operand_map(&tb, B.ptr, (uint64_t)N, (uint64_t)K, B.ld, 64, 64)
                     : make_operand_map(&tb, B.ptr, (uint64_t)K, (uint64_t)N, B.ld, 64, Cfg::B_ROWS));
    EpiMaps maps;
    memset(&maps, 0, sizeof maps);
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (KIND == EPI_STORE_F32)          // 3-D store: {n, m, split}
        ok = ok && make_map(&maps.o1, epi.out, F32, 4, N, M, epi.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                            3, splits);
    else if (KIND == EPI_ACCUM_F32)     // 2-D reduce-add
        ok = ok && make_map(&maps.o1, epi.out, F32, 4, N, M, epi.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    else
        ok = ok && make_map(&maps.o1, epi.out, BF, 2, N, M, epi.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (KIND == EPI_GELU)
        ok = ok && make_map(&maps.o2, epi.out2, BF, 2, N, M, epi.ldo2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (KIND == EPI_GELU_BWD)
        ok = ok && make_map(&maps.aux, epi.aux, BF, 2, N, M, epi.ld_aux, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return cudaErrorInvalidValue;
    // GELU_BWD with out2 set: per-32-row column sums of the result (the
    // bias gradient of the Linear whose input gradient it is)
    float* colsum = KIND == EPI_GELU_BWD ? (float*)epi.out2 : nullptr;
    auto kern = gemm_tc_kernel<BN, A_MN, B_MN, KIND, PAIR>;
    static bool attr_set = false;
    static int pairs = 0;
    if (!attr_set) {
        CUDA_OK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM));
        if (PAIR) {
            pairs = max_pairs(kern, Cfg::SMEM);
            if (pairs < 1) return cudaErrorInvalidConfiguration;
        }
        attr_set = true;
    }
    constexpr int TILE_M = PAIR ? 2 * TC_BM : TC_BM;
    const int tiles = ((M + TILE_M - 1) / TILE_M) * ((N + BN - 1) / BN);
    const int total = tiles * splits;
    if (!PAIR) {
        const int grid = total < num_sms() ? total : num_sms();
        (void)pdl_launch(kern, grid, TC_THREADS, Cfg::SMEM, s, ta, tb, maps, M, N, K, splits, epi.bias, colsum, st);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * (total < pairs ? total : pairs), 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_on() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, maps, M, N, K, splits, epi.bias, colsum, st);
}

// BN = 256 tiles run as CTA pairs (cta_group::2); BN = 128 as single CTAs.
template <int BN, bool A_MN, bool B_MN>
static cudaError_t launch_kind(int M, int N, int K, GemmOperand A, GemmOperand B, const GemmEpi& epi,
                               int splits, DevState* st, cudaStream_t s) {
    constexpr bool P = (BN == 256);
    switch (epi.kind) {
        case EPI_STORE_ACT: return launch_tc<BN, A_MN, B_MN, EPI_STORE_ACT, P>(M, N, K, A, B, epi, splits, st, s);
        case EPI_GELU: return launch_tc<BN, A_MN, B_MN, EPI_GELU, P>(M, N, K, A, B, epi, splits, st, s);
        case EPI_GELU_BWD: return launch_tc<BN, A_MN, B_MN, EPI_GELU_BWD, P>(M, N, K, A, B, epi, splits, st, s);
        case EPI_STORE_F32: return launch_tc<BN, A_MN, B_MN, EPI_STORE_F32, P>(M, N, K, A, B, epi, splits, st, s);
        case EPI_ACCUM_F32: return launch_tc<BN, A_MN, B_MN, EPI_ACCUM_F32, P>(M, N, K, A, B, epi, splits, st, s);
        default: return cudaErrorInvalidValue;
    }
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
        return launch_kind<BNV, AM, BM_>(M, N, K, A, B, epi, splits, st, s);
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
