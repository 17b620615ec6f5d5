// Per-token E4M3 quantisation of the activations of the FP8 up projection
// (MOE_BF16_FP8UP).  The pages name FP8 for the expert GEMMs ("技术日报
// 2026-04-14" §7.4, FP8 against BF16); on the 5th-generation tensor cores both
// operands of an FP8 MMA are FP8, so the rows that enter the up projection are
// quantised too: one fp32 scale per row, s = amax / 448, and the codes
// E4M3(x / s), rounded to nearest even and saturated to +-448 (an all-zero row
// gets s = 0 and zero codes).  The same rule as the per-channel weight scales,
// applied along a row: the scale of a row factors out of every dot product of
// that row, so the GEMM epilogue multiplies the accumulator by s_row * s_column.
//
// One warp per row: a first pass over the row's 16-byte vectors for its maximum,
// a second pass (the row is in L1 / L2) converting pairs with cvt.rn.satfinite.
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3 codes of (a, b) as two bytes, a in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    unsigned short pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(b), "f"(a));
    return pair;
}

// Eight bf16 (one 16-byte vector) divided by s -> eight codes (8 bytes).
__device__ __forceinline__ uint2 quantize8(const uint4 &v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = e4m3x2(bf16_lo(w[i]) / s, bf16_hi(w[i]) / s);
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__global__ void __launch_bounds__(256)
    quantize_rows_kernel(const uint4 *__restrict__ x, int64_t rows, int vecs, uint2 *__restrict__ q,
                         float *__restrict__ scale) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const uint4 *src = x + (size_t)r * vecs;
        float amax = 0.f;
        for (int v = lane; v < vecs; v += 32 * 4) {
            uint4 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < vecs) t[u] = src[v + 32 * u];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (v + 32 * u < vecs) {
                    const uint32_t w[4] = {t[u].x, t[u].y, t[u].z, t[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax / 448.f;
        uint2 *dst = q + (size_t)r * vecs;
        for (int v = lane; v < vecs; v += 32 * 4) {
            uint4 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < vecs) t[u] = src[v + 32 * u];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v + 32 * u < vecs) dst[v + 32 * u] = (s == 0.f) ? make_uint2(0, 0) : quantize8(t[u], s);
        }
        if (lane == 0) scale[r] = s;
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const void *x, int64_t rows, int d, uint8_t *q, float *s, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int vecs = d / 8;   // 16-byte vectors of bf16
    int64_t blocks = (rows + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    return launch_dependent(quantize_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, false,
                            static_cast<const uint4 *>(x), rows, vecs, reinterpret_cast<uint2 *>(q), s);
}

}  // namespace moe
