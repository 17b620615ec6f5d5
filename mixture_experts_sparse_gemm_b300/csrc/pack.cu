// One-time re-layout of the expert weights into the operand layout of the grouped
// GEMMs (the weights of "lnwmold.com GPT-4 MoE article" §2.2: W1, W3 up, W2 down).
//
//   up   : W1[e][d][f], W3[e][d][f]  ->  w13[e][2f][d]  (K-major rows; rows come in
//          groups of 2*kGroup: kGroup rows of W1 columns, then the same W3 columns)
//   down : W2[e][f][d]               ->  w2[e][d][f]    (K-major rows)
// Shared experts are merged along the hidden dimension (sum_s FFN_s(x) is one FFN
// whose hidden width is n_shared * f_shared) and packed the same way.
//
// Both are tiled 32x32 transposes through shared memory.  For bf16 the
// destination is the tensor-core tile image (tiled_offset: BN x 64 tiles with the
// 128-byte swizzle already applied), so the GEMMs stream each weight tile as one
// contiguous bulk copy; fp32 (CUDA-core path) keeps plain K-major rows.
#include "moe_internal.cuh"

namespace moe {
namespace {

// source element (e, i, h) with h split into nsub sub-experts of width fsub
// Destination of (row p, column i) of one expert's [N][K] operand: plain K-major
// rows (tile_n == 0), or the tensor-core tile images of tiled_offset.
__device__ __forceinline__ size_t dst_offset(int p, int i, int K, int tile_n) {
    return tile_n ? tiled_offset(p, i, tile_n, K) : (size_t)p * K + i;
}

template <typename T>
__global__ void pack_up_kernel(const T *__restrict__ W1, const T *__restrict__ W3, T *__restrict__ out, int d,
                               int nsub, int fsub, int tile_n) {
    __shared__ T tile[32][33];
    const int ftot = nsub * fsub;
    const int e = blockIdx.z >> 1, m = blockIdx.z & 1;
    const T *W = m ? W3 : W1;
    const int h0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    for (int ii = threadIdx.y; ii < 32; ii += blockDim.y) {
        const int i = i0 + ii, h = h0 + threadIdx.x;
        if (i < d && h < ftot) {
            const size_t src = ((size_t)(e * nsub + h / fsub) * d + i) * fsub + (h % fsub);
            tile[ii][threadIdx.x] = W[src];
        }
    }
    __syncthreads();
    for (int hh = threadIdx.y; hh < 32; hh += blockDim.y) {
        const int h = h0 + hh, i = i0 + threadIdx.x;
        if (i < d && h < ftot) {
            const int r = (h / kGroup) * (2 * kGroup) + m * kGroup + (h % kGroup);
            out[(size_t)e * 2 * ftot * d + dst_offset(r, i, d, tile_n)] = tile[threadIdx.x][hh];
        }
    }
}

template <typename T>
__global__ void pack_down_kernel(const T *__restrict__ W2, T *__restrict__ out, int d, int nsub, int fsub,
                                 int tile_n) {
    __shared__ T tile[32][33];
    const int ftot = nsub * fsub;
    const int e = blockIdx.z;
    const int n0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
    for (int hh = threadIdx.y; hh < 32; hh += blockDim.y) {
        const int h = h0 + hh, n = n0 + threadIdx.x;
        if (h < ftot && n < d) {
            const size_t src = ((size_t)(e * nsub + h / fsub) * fsub + (h % fsub)) * d + n;
            tile[hh][threadIdx.x] = W2[src];
        }
    }
    __syncthreads();
    for (int nn = threadIdx.y; nn < 32; nn += blockDim.y) {
        const int n = n0 + nn, h = h0 + threadIdx.x;
        if (h < ftot && n < d) out[(size_t)e * d * ftot + dst_offset(n, h, ftot, tile_n)] = tile[threadIdx.x][nn];
    }
}

template <typename T>
cudaError_t pack_typed(const moe_config &c, const void *W1, const void *W3, const void *W2, const void *W1s,
                       const void *W3s, const void *W2s, void *packed, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    char *base = static_cast<char *>(packed);
    const dim3 blk(32, 8);
    // bf16 weights feed the tensor-core GEMMs as tile images; fp32 stays K-major rows
    const int tn_up = (c.dtype == MOE_BF16) ? up_tile_n(c) : 0;
    const int tn_dn = (c.dtype == MOE_BF16) ? down_tile_n(c) : 0;
    {
        const dim3 g((c.f + 31) / 32, (c.d + 31) / 32, c.E * 2);
        pack_up_kernel<T><<<g, blk, 0, s>>>(static_cast<const T *>(W1), static_cast<const T *>(W3),
                                            reinterpret_cast<T *>(base + L.w13), c.d, 1, c.f, tn_up);
        const dim3 g2((c.d + 31) / 32, (c.f + 31) / 32, c.E);
        pack_down_kernel<T><<<g2, blk, 0, s>>>(static_cast<const T *>(W2), reinterpret_cast<T *>(base + L.w2), c.d, 1,
                                               c.f, tn_dn);
    }
    if (c.n_shared > 0) {
        const int fs = c.n_shared * c.f_shared;
        const dim3 g((fs + 31) / 32, (c.d + 31) / 32, 2);
        pack_up_kernel<T><<<g, blk, 0, s>>>(static_cast<const T *>(W1s), static_cast<const T *>(W3s),
                                            reinterpret_cast<T *>(base + L.w13s), c.d, c.n_shared, c.f_shared, tn_up);
        const dim3 g2((c.d + 31) / 32, (fs + 31) / 32, 1);
        pack_down_kernel<T><<<g2, blk, 0, s>>>(static_cast<const T *>(W2s), reinterpret_cast<T *>(base + L.w2s), c.d,
                                               c.n_shared, c.f_shared, tn_dn);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const moe_config &c, const void *W1, const void *W3, const void *W2, const void *W1s,
                        const void *W3s, const void *W2s, void *packed, cudaStream_t s) {
    if (c.dtype == MOE_F32) return pack_typed<float>(c, W1, W3, W2, W1s, W3s, W2s, packed, s);
    return pack_typed<unsigned short>(c, W1, W3, W2, W1s, W3s, W2s, packed, s);   // bf16 bits
}

}  // namespace moe
