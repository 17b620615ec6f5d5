// Gate-weighted combine back to token order ("技术日报 2026-04-14" §3.1:
// y = sum_i G(x)_i E_i(x); §3.4 / §9.1: shared experts added unweighted;
// "MoE稀疏架构" §4 step 5).
//
// One warp per (token, span of the row).  The warp first lists the token's
// (row, weight) pairs in order -- slots j = 0..k-1 for token choice, experts e
// ascending for Expert Choice -- then every lane accumulates 16-byte vectors of
// those Y rows in fp32 -- four of its vectors of two rows in flight at once, so a
// token with few experts still has eight loads outstanding per lane -- and writes
// its part of the token's output row once.  A span is the whole row unless there are fewer tokens than
// eight warps per SM; then the rows are split so that the work spreads.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

template <typename T>
struct Vec;   // 16 bytes of T
template <>
struct Vec<float> {
    static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
};

template <typename T>
__device__ __forceinline__ void accumulate(float (&acc)[Vec<T>::N], const uint4 &v, float w) {
    if constexpr (sizeof(T) == 4) {
        acc[0] = fmaf(w, __uint_as_float(v.x), acc[0]);
        acc[1] = fmaf(w, __uint_as_float(v.y), acc[1]);
        acc[2] = fmaf(w, __uint_as_float(v.z), acc[2]);
        acc[3] = fmaf(w, __uint_as_float(v.w), acc[3]);
    } else {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
        }
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack(const float (&acc)[Vec<T>::N]) {
    uint4 v;
    if constexpr (sizeof(T) == 4) {
        v.x = __float_as_uint(acc[0]);
        v.y = __float_as_uint(acc[1]);
        v.z = __float_as_uint(acc[2]);
        v.w = __float_as_uint(acc[3]);
    } else {
        __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    }
    return v;
}

struct CombineArgs {
    const uint4 *Y;
    const int32_t *slot_of;
    const float *w;
    uint4 *y;
    int T, E, k, mode, vecs;
    int span;              // 16-byte vectors of a row per work item, a multiple of kStepVecs
    int64_t shared_row0;   // first shared row of Y, -1 without shared experts
};

constexpr int kStepVecs = 32;   // vectors one warp step covers: one per lane
constexpr int kCols = 4;        // vectors per lane handled together (4 x 32 x 16 bytes of a row per warp)
constexpr int kRows = 2;        // rows loaded together

template <typename T>
__global__ void __launch_bounds__(32 * kWarps) combine_kernel(CombineArgs a) {
    __shared__ int s_row[kWarps][kMaxE];
    __shared__ float s_w[kWarps][kMaxE];
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_tok = (a.mode == MOE_EXPERT_CHOICE) ? a.E : a.k;
    const int nch = (a.vecs + a.span - 1) / a.span;
    const int64_t items = (int64_t)a.T * nch;
    for (int64_t item = (int64_t)blockIdx.x * kWarps + warp; item < items; item += (int64_t)gridDim.x * kWarps) {
        const int t = (int)(item / nch), c = (int)(item % nch);
        int n = 0;
        for (int j0 = 0; j0 < per_tok; j0 += 32) {
            const int j = j0 + lane;
            int row = -1;
            float w = 0.f;
            if (j < per_tok) {
                row = a.slot_of[(size_t)t * per_tok + j];
                if (row >= 0) w = (a.mode == MOE_EXPERT_CHOICE) ? a.w[row] : a.w[(size_t)t * per_tok + j];
            }
            const unsigned b = __ballot_sync(0xffffffffu, row >= 0);
            if (row >= 0) {
                const int p = n + __popc(b & ((1u << lane) - 1u));
                s_row[warp][p] = row;
                s_w[warp][p] = w;
            }
            n += __popc(b);
        }
        __syncwarp();
        const uint4 *ys = a.shared_row0 >= 0 ? a.Y + (size_t)(a.shared_row0 + t) * a.vecs : nullptr;
        const int vend = min(a.vecs, (c + 1) * a.span);
        // kCols vectors of the lane (32 apart) at a time; rows kRows at a time, all
        // kRows x kCols loads in flight before they are accumulated.  Every output
        // element still adds its rows in slot order, then the shared row.
        for (int v0 = c * a.span + lane; v0 < vend; v0 += kStepVecs * kCols) {
            float acc[kCols][Vec<T>::N];
#pragma unroll
            for (int u = 0; u < kCols; ++u)
#pragma unroll
                for (int q = 0; q < Vec<T>::N; ++q) acc[u][q] = 0.f;
            for (int i = 0; i < n; i += kRows) {
                uint4 r[kRows][kCols];
#pragma unroll
                for (int q = 0; q < kRows; ++q)
#pragma unroll
                    for (int u = 0; u < kCols; ++u)
                        if (i + q < n && v0 + kStepVecs * u < vend)
                            r[q][u] = a.Y[(size_t)s_row[warp][i + q] * a.vecs + v0 + kStepVecs * u];
#pragma unroll
                for (int q = 0; q < kRows; ++q)
                    if (i + q < n) {
                        const float w = s_w[warp][i + q];
#pragma unroll
                        for (int u = 0; u < kCols; ++u)
                            if (v0 + kStepVecs * u < vend) accumulate<T>(acc[u], r[q][u], w);
                    }
            }
            if (ys) {
                uint4 r[kCols];
#pragma unroll
                for (int u = 0; u < kCols; ++u)
                    if (v0 + kStepVecs * u < vend) r[u] = ys[v0 + kStepVecs * u];
#pragma unroll
                for (int u = 0; u < kCols; ++u)
                    if (v0 + kStepVecs * u < vend) accumulate<T>(acc[u], r[u], 1.f);
            }
#pragma unroll
            for (int u = 0; u < kCols; ++u)
                if (v0 + kStepVecs * u < vend) a.y[(size_t)t * a.vecs + v0 + kStepVecs * u] = pack<T>(acc[u]);
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_combine(const moe_config &c, const Sizes &z, const void *Y, const int32_t *slot_of,
                           const float *w, void *y, cudaStream_t s) {
    CombineArgs a;
    a.Y = static_cast<const uint4 *>(Y);
    a.slot_of = slot_of;
    a.w = w;
    a.y = static_cast<uint4 *>(y);
    a.T = c.T;
    a.E = c.E;
    a.k = c.k;
    a.mode = c.mode;
    a.vecs = c.d * z.elt / 16;
    a.shared_row0 = (c.n_shared > 0) ? z.rows_routed : -1;
    // one warp per token; with fewer tokens than eight warps per SM the rows are
    // split into spans so that the work still spreads over the GPU
    const int64_t target = (int64_t)num_sms() * 8;
    const int max_ch = (a.vecs + kStepVecs - 1) / kStepVecs;
    int64_t nch = (target + c.T - 1) / (c.T > 0 ? c.T : 1);
    nch = nch < 1 ? 1 : (nch > max_ch ? max_ch : nch);
    a.span = (int)(((a.vecs + nch - 1) / nch + kStepVecs - 1) / kStepVecs * kStepVecs);
    const int64_t items = (int64_t)c.T * ((a.vecs + a.span - 1) / a.span);
    int64_t blocks = (items + kWarps - 1) / kWarps;
    auto kern = c.dtype == MOE_F32 ? combine_kernel<float> : combine_kernel<__nv_bfloat16>;
    // no more blocks than are resident at once (the warps loop over the items): a
    // second wave of blocks would start only as the first one drains
    static int resident[2] = {0, 0};
    int &per_sm = resident[c.dtype == MOE_F32 ? 1 : 0];
    if (per_sm == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kWarps, 0) != cudaSuccess) {
        (void)cudaGetLastError();
        per_sm = 0;
    }
    const int64_t cap = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 8);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_dependent(kern, dim3((unsigned)blocks), dim3(32 * kWarps), 0, s, false, a);
}

}  // namespace moe
