// Grouped SwiGLU experts on CUDA cores (the fp32 path; no TF32 anywhere).
//
// Expert FFN with W1, W3 up and W2 down ("lnwmold.com GPT-4 MoE article" §2.2),
// read as SwiGLU: H = SiLU(X W1) * (X W3), Y = H W2, fp32 accumulation.
//
// Both GEMMs walk the ragged expert segments of the expert-ordered rows with a
// persistent tile loop; the tile table is rebuilt on the device from off[], so
// no host synchronisation is needed between dispatch and the experts.
//   up   : tile 64 rows x 64 hidden columns (one packed group = 64 W1 + 64 W3 rows)
//   down : tile 64 rows x 64 output columns
// Each of the 256 threads owns a 4x4 block of the tile (x2 for gate/up).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kKC = 16;
constexpr int kThreads = 256;

struct SimtArgs {
    GroupedShape g;
    const void *A0;   // routed rows (x_perm or H)
    const void *A1;   // shared rows (x or Hs)
    const void *B0;   // routed packed weights
    const void *B1;   // shared packed weights
    void *C0;         // routed output
    void *C1;         // shared output
    int K0, K1;       // reduction width routed / shared
    int ldc0, ldc1;   // output row pitch (elements)
    int b_rows0;      // packed rows per routed expert (2f for up, d for down)
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

template <typename T, bool kUp>
__global__ void __launch_bounds__(kThreads) ffn_simt_kernel(SimtArgs a) {
    __shared__ int tile_start[kMaxE + 2], seg_row0[kMaxE + 1], seg_rows[kMaxE + 1];
    constexpr int kBCols = kUp ? 2 * kBN : kBN;
    __shared__ float As[kKC][kBM + 4];
    __shared__ float Bs[kKC][kBCols + 4];
    const int S = build_tile_table<kBM>(a.g, tile_start, seg_row0, seg_rows);
    const int total = tile_start[S];
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;

    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int s, mb, nb;
        decode_tile<kBM>(a.g, tile_start, seg_rows, S, tile, s, mb, nb);
        const bool routed = s < a.g.E;
        const T *A = static_cast<const T *>(routed ? a.A0 : a.A1);
        const T *B = static_cast<const T *>(routed ? a.B0 : a.B1);
        T *C = static_cast<T *>(routed ? a.C0 : a.C1);
        const int K = routed ? a.K0 : a.K1;
        const int ldc = routed ? a.ldc0 : a.ldc1;
        const int row0 = seg_row0[s] + mb * kBM;          // first row in A / C
        const int rows = min(kBM, seg_rows[s] - mb * kBM);
        const size_t b_row0 = (routed ? (size_t)s * a.b_rows0 : 0) + (size_t)nb * kBCols;

        float acc[kUp ? 2 : 1][4][4];
#pragma unroll
        for (int h = 0; h < (kUp ? 2 : 1); ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[h][i][j] = 0.f;

        for (int k0 = 0; k0 < K; k0 += kKC) {
            for (int i = tid; i < kBM * kKC; i += kThreads) {
                const int m = i / kKC, kk = i % kKC;
                As[kk][m] = (m < rows && k0 + kk < K) ? to_f32(A[(size_t)(row0 + m) * K + k0 + kk]) : 0.f;
            }
            for (int i = tid; i < kBCols * kKC; i += kThreads) {
                const int n = i / kKC, kk = i % kKC;
                Bs[kk][n] = (k0 + kk < K) ? to_f32(B[(b_row0 + n) * K + k0 + kk]) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < kKC; ++kk) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[0][i][j] = fmaf(av[i], bv[j], acc[0][i][j]);
                if constexpr (kUp) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][kBN + tx * 4 + j];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[1][i][j] = fmaf(av[i], bv[j], acc[1][i][j]);
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = ty * 4 + i;
            if (m >= rows) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = nb * kBN + tx * 4 + j;
                float v = acc[0][i][j];
                if constexpr (kUp) v = silu(v) * acc[1][i][j];
                C[(size_t)(row0 + m) * ldc + n] = from_f32<T>(v);
            }
        }
    }
}

template <typename T>
cudaError_t run_up(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off, const void *packed,
                   const void *x, void *H, void *Hs, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const int shared_rows = c.n_shared > 0 ? c.T : 0;
    const int64_t max_tiles_m = (z.rows_routed + kBM - 1) / kBM + c.E + (shared_rows + kBM - 1) / kBM;
    SimtArgs up{};
    up.g = GroupedShape{off, c.E, shared_rows, c.f / kBN, z.fs_tot / kBN};
    up.A0 = x_perm;
    up.A1 = x;
    up.B0 = pk + L.w13;
    up.B1 = pk + L.w13s;
    up.C0 = H;
    up.C1 = Hs;
    up.K0 = c.d;
    up.K1 = c.d;
    up.ldc0 = c.f;
    up.ldc1 = z.fs_tot;
    up.b_rows0 = 2 * c.f;
    const int nb = std::max(c.f, z.fs_tot) / kBN;
    const int g1 = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms() * 4, max_tiles_m * nb));
    ffn_simt_kernel<T, true><<<g1, kThreads, 0, s>>>(up);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_down(const moe_config &c, const Sizes &z, const void *H, const void *Hs, const int32_t *off,
                     const void *packed, void *Y, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const int shared_rows = c.n_shared > 0 ? c.T : 0;
    const int64_t max_tiles_m = (z.rows_routed + kBM - 1) / kBM + c.E + (shared_rows + kBM - 1) / kBM;
    SimtArgs dn{};
    dn.g = GroupedShape{off, c.E, shared_rows, c.d / kBN, c.d / kBN};
    dn.A0 = H;
    dn.A1 = Hs;
    dn.B0 = pk + L.w2;
    dn.B1 = pk + L.w2s;
    dn.C0 = Y;
    dn.C1 = static_cast<char *>(Y) + (size_t)z.rows_routed * c.d * sizeof(T);
    dn.K0 = c.f;
    dn.K1 = z.fs_tot;
    dn.ldc0 = c.d;
    dn.ldc1 = c.d;
    dn.b_rows0 = c.d;
    const int g2 = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms() * 4, max_tiles_m * (c.d / kBN)));
    ffn_simt_kernel<T, false><<<g2, kThreads, 0, s>>>(dn);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_up_simt(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                               const void *packed, const void *x, void *H, void *Hs, cudaStream_t s) {
    // fp32 only: bf16 weights are packed as tensor-core tile images for the tcgen05 path
    if (c.dtype != MOE_F32) return cudaErrorNotSupported;
    return run_up<float>(c, z, x_perm, off, packed, x, H, Hs, s);
}

cudaError_t launch_ffn_down_simt(const moe_config &c, const Sizes &z, const void *H, const void *Hs,
                                 const int32_t *off, const void *packed, void *Y, cudaStream_t s) {
    if (c.dtype != MOE_F32) return cudaErrorNotSupported;
    return run_down<float>(c, z, H, Hs, off, packed, Y, s);
}

}  // namespace moe
