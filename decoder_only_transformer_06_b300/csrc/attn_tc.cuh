// Shared pieces of the tcgen05 causal-attention kernels (forward in
// k_attention_tc.cu, backward in k_attention_bwd_tc.cu): tile constants,
// small device helpers and the tensor maps over the fused qkv buffer.
#pragma once

#include "common.cuh"
#include "tc.cuh"
#include <cuda.h>
#include <cstring>

namespace k {
namespace attn {

constexpr int AT_BQ = 128;                     // query rows of a 128-row tile
constexpr int AT_BK = 128;                     // key rows of a 128-row tile
constexpr int AT_HS = 64;                      // head size
constexpr int AT_TILE = AT_BQ * AT_HS * 2;     // 16 KB: 128 rows x 128 B
constexpr int OUT_SLAB = 32 * AT_HS * 2;       // one warp's 32 output rows, 4 KB
constexpr float LN2 = 0.6931471805599453f;
constexpr float LOG2E_F = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *(uint32_t*)&h;
}
// Drain wait after an abort: always the full limit (the copy or product it
// waits for is in flight and must land before the CTA exits).
__device__ __forceinline__ void wait_bounded(uint64_t* bar, uint32_t parity) {
    const long long t0 = wait_clock();
    while (!tc::mbar_try_wait(bar, parity) && wait_clock() - t0 < WAIT_LIMIT_CYCLES) {}
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

// A warp's 32 rows x 32 columns (fp32 values times `scale`) as bf16 into a
// 64B-swizzled 2 KB slab: lane = row, 16-byte piece q of row r at
// r*64 + ((q ^ ((r >> 1) & 3)) << 4), the layout the TMA store of a 32 x 32
// box with 64B swizzle expects.
__device__ __forceinline__ void stage_out_slab32(uint8_t* slab, int lane, const uint32_t (&a)[32], float scale) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float* f = (const float*)&a[8 * q];
        *(uint4*)(slab + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(pack2_bf16(f[0] * scale, f[1] * scale), pack2_bf16(f[2] * scale, f[3] * scale),
                       pack2_bf16(f[4] * scale, f[5] * scale), pack2_bf16(f[6] * scale, f[7] * scale));
    }
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFnA)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFnA encode_fn() {
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

// A [B, T, width] bf16 tensor as a 3-D map {width, T, B} with boxes of
// 64 columns x box_rows rows x 1 and 128B swizzle. Loads: rows beyond T of a
// sequence read as zeros (never the next sequence's rows); stores: rows beyond
// T are clipped. 64 x box_rows boxes with 128B swizzle are the K-major (and
// MN-major) operand layout of the tcgen05 descriptors.
// With box_cols = 32 the swizzle is 64B (32 bf16 = 64-byte rows), the layout
// of stage_out_slab32.
inline bool make_rows_map(CUtensorMap* map, const bf16* ptr, int B, int T, int width, int box_rows,
                          bool l2_promote, int box_cols = 64) {
    EncodeTiledFnA enc = encode_fn();
    if (!enc) return false;
    memset(map, 0, sizeof *map);
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * T};
    cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               l2_promote ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace attn
}  // namespace k
