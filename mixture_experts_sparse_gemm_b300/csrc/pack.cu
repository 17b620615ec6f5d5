// One-time re-layout of the expert weights into the operand layout of the grouped
// GEMMs (the weights of "lnwmold.com GPT-4 MoE article" §2.2: W1, W3 up, W2 down).
//
//   up   : W1[e][d][f], W3[e][d][f]  ->  w13[e][2f][d]  (K-major rows; rows come in
//          groups of 2*kGroup: kGroup rows of W1 columns, then the same W3 columns)
//   down : W2[e][f][d]               ->  w2[e][d][f]    (K-major rows)
// Shared experts are merged along the hidden dimension (sum_s FFN_s(x) is one FFN
// whose hidden width is n_shared * f_shared) and packed the same way.
//
// Both are tiled 32x32 transposes through shared memory.  MOE_BF16_FP8W first
// takes one scale per output channel, then writes E4M3 codes as FP8 tile images
// (tiled_offset8) and the scales after the matrices.  For bf16 the
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

// ----------------------------------------------------------------------------- FP8 weights
// E4M3 quantisation with one scale per output channel: s = amax / 448 over the
// channel's K inputs (fp32), code = E4M3(w / s) rounded to nearest even and
// saturated to +-448 (cvt.rn.satfinite); s = 0 and codes 0 for an all-zero channel.
__device__ __forceinline__ float bf16_bits_to_f32(unsigned short b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint8_t e4m3_code(float w, float s) {
    if (s == 0.f) return 0;
    const float v = w / s;
    unsigned short pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(v));   // both halves the same value
    return (uint8_t)(pair & 0xFF);
}

// Up projection: scale of packed row r(h, m) (W1 when m = 0, W3 when m = 1) =
// amax over i of |W[e][i][h]| / 448.  One thread per (expert, m, h), looping over i
// (neighbouring threads read neighbouring h: coalesced).
__global__ void amax_up_kernel(const unsigned short *__restrict__ W1, const unsigned short *__restrict__ W3, float *sc,
                               int d, int nsub, int fsub, int nmat_e) {
    const int ftot = nsub * fsub;
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    const int e = blockIdx.y >> 1, m = blockIdx.y & 1;
    if (h >= ftot) return;
    const unsigned short *W = m ? W3 : W1;
    const size_t base = (size_t)(e * nsub + h / fsub) * d * fsub + (h % fsub);
    float amax = 0.f;
    for (int i = 0; i < d; ++i) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(W[base + (size_t)i * fsub])));
    const int r = (h / kGroup) * (2 * kGroup) + m * kGroup + (h % kGroup);
    sc[(size_t)e * nmat_e + r] = amax / 448.f;
}

// Down projection: scale of output column n = amax over h of |W2[e][h][n]| / 448.
__global__ void amax_down_kernel(const unsigned short *__restrict__ W2, float *sc, int d, int nsub, int fsub) {
    const int ftot = nsub * fsub;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int e = blockIdx.y;
    if (n >= d) return;
    float amax = 0.f;
    for (int h = 0; h < ftot; ++h) {
        const size_t src = ((size_t)(e * nsub + h / fsub) * fsub + (h % fsub)) * d + n;
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(W2[src])));
    }
    sc[(size_t)e * d + n] = amax / 448.f;
}

// Codes of the up projection, transposed through shared memory into FP8 tile images:
// 64-byte rows for the converter warps (mma_ready == 0), or the 128-byte swizzled
// rows that kind::f8f6f4 reads directly (mma_ready == 1, tiled_offset_f8).
__global__ void quant_up_kernel(const unsigned short *__restrict__ W1, const unsigned short *__restrict__ W3,
                                const float *__restrict__ sc, uint8_t *__restrict__ out, int d, int nsub, int fsub,
                                int tile_n, int mma_ready) {
    __shared__ float tile[32][33];
    const int ftot = nsub * fsub;
    const int e = blockIdx.z >> 1, m = blockIdx.z & 1;
    const unsigned short *W = m ? W3 : W1;
    const int h0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    for (int ii = threadIdx.y; ii < 32; ii += blockDim.y) {
        const int i = i0 + ii, h = h0 + threadIdx.x;
        if (i < d && h < ftot) {
            const size_t src = ((size_t)(e * nsub + h / fsub) * d + i) * fsub + (h % fsub);
            tile[ii][threadIdx.x] = bf16_bits_to_f32(W[src]);
        }
    }
    __syncthreads();
    for (int hh = threadIdx.y; hh < 32; hh += blockDim.y) {
        const int h = h0 + hh, i = i0 + threadIdx.x;
        if (i < d && h < ftot) {
            const int r = (h / kGroup) * (2 * kGroup) + m * kGroup + (h % kGroup);
            const float s = sc[(size_t)e * 2 * ftot + r];
            const size_t o = mma_ready ? tiled_offset_f8(r, i, tile_n, d) : tiled_offset8(r, i, tile_n, d);
            out[(size_t)e * 2 * ftot * d + o] = e4m3_code(tile[threadIdx.x][hh], s);
        }
    }
}

// Codes of the down projection: W2[e][h][n] -> tile images of [d][ftot].
__global__ void quant_down_kernel(const unsigned short *__restrict__ W2, const float *__restrict__ sc,
                                  uint8_t *__restrict__ out, int d, int nsub, int fsub, int tile_n) {
    __shared__ float tile[32][33];
    const int ftot = nsub * fsub;
    const int e = blockIdx.z;
    const int n0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
    for (int hh = threadIdx.y; hh < 32; hh += blockDim.y) {
        const int h = h0 + hh, n = n0 + threadIdx.x;
        if (h < ftot && n < d) {
            const size_t src = ((size_t)(e * nsub + h / fsub) * fsub + (h % fsub)) * d + n;
            tile[hh][threadIdx.x] = bf16_bits_to_f32(W2[src]);
        }
    }
    __syncthreads();
    for (int nn = threadIdx.y; nn < 32; nn += blockDim.y) {
        const int n = n0 + nn, h = h0 + threadIdx.x;
        if (h < ftot && n < d) {
            const float s = sc[(size_t)e * d + n];
            out[(size_t)e * d * ftot + tiled_offset8(n, h, tile_n, ftot)] = e4m3_code(tile[threadIdx.x][nn], s);
        }
    }
}

cudaError_t pack_fp8(const moe_config &c, const void *W1, const void *W3, const void *W2, const void *W1s,
                     const void *W3s, const void *W2s, void *packed, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    char *base = static_cast<char *>(packed);
    const dim3 blk(32, 8);
    const int tn_up = up_tile_n(c), tn_dn = down_tile_n(c);
    using U = unsigned short;
    auto f = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    auto q = [&](size_t off) { return reinterpret_cast<uint8_t *>(base + off); };
    amax_up_kernel<<<dim3((c.f + 255) / 256, c.E * 2), 256, 0, s>>>(static_cast<const U *>(W1),
                                                                   static_cast<const U *>(W3), f(L.sc13), c.d, 1,
                                                                   c.f, 2 * c.f);
    amax_down_kernel<<<dim3((c.d + 255) / 256, c.E), 256, 0, s>>>(static_cast<const U *>(W2), f(L.sc2), c.d, 1,
                                                                  c.f);
    quant_up_kernel<<<dim3((c.f + 31) / 32, (c.d + 31) / 32, c.E * 2), blk, 0, s>>>(
        static_cast<const U *>(W1), static_cast<const U *>(W3), f(L.sc13), q(L.w13), c.d, 1, c.f, tn_up, 0);
    quant_down_kernel<<<dim3((c.d + 31) / 32, (c.f + 31) / 32, c.E), blk, 0, s>>>(
        static_cast<const U *>(W2), f(L.sc2), q(L.w2), c.d, 1, c.f, tn_dn);
    if (c.n_shared > 0) {
        const int fs = c.n_shared * c.f_shared;
        amax_up_kernel<<<dim3((fs + 255) / 256, 2), 256, 0, s>>>(static_cast<const U *>(W1s),
                                                                  static_cast<const U *>(W3s), f(L.sc13s), c.d,
                                                                  c.n_shared, c.f_shared, 2 * fs);
        amax_down_kernel<<<dim3((c.d + 255) / 256, 1), 256, 0, s>>>(static_cast<const U *>(W2s), f(L.sc2s), c.d,
                                                                     c.n_shared, c.f_shared);
        quant_up_kernel<<<dim3((fs + 31) / 32, (c.d + 31) / 32, 2), blk, 0, s>>>(
            static_cast<const U *>(W1s), static_cast<const U *>(W3s), f(L.sc13s), q(L.w13s), c.d, c.n_shared,
            c.f_shared, tn_up, 0);
        quant_down_kernel<<<dim3((c.d + 31) / 32, (fs + 31) / 32, 1), blk, 0, s>>>(
            static_cast<const U *>(W2s), f(L.sc2s), q(L.w2s), c.d, c.n_shared, c.f_shared, tn_dn);
    }
    return cudaGetLastError();
}

// FP8 up projection: W1 / W3 as E4M3 codes in the tile images kind::f8f6f4 reads
// (one scale per output channel), W2 as bf16 tile images.
cudaError_t pack_fp8_up(const moe_config &c, const void *W1, const void *W3, const void *W2, const void *W1s,
                        const void *W3s, const void *W2s, void *packed, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    char *base = static_cast<char *>(packed);
    const dim3 blk(32, 8);
    const int tn_up = up_tile_n(c), tn_dn = down_tile_n(c);
    using U = unsigned short;
    auto f = [&](size_t off) { return reinterpret_cast<float *>(base + off); };
    auto q = [&](size_t off) { return reinterpret_cast<uint8_t *>(base + off); };
    amax_up_kernel<<<dim3((c.f + 255) / 256, c.E * 2), 256, 0, s>>>(static_cast<const U *>(W1),
                                                                   static_cast<const U *>(W3), f(L.sc13), c.d, 1,
                                                                   c.f, 2 * c.f);
    quant_up_kernel<<<dim3((c.f + 31) / 32, (c.d + 31) / 32, c.E * 2), blk, 0, s>>>(
        static_cast<const U *>(W1), static_cast<const U *>(W3), f(L.sc13), q(L.w13), c.d, 1, c.f, tn_up, 1);
    pack_down_kernel<U><<<dim3((c.d + 31) / 32, (c.f + 31) / 32, c.E), blk, 0, s>>>(
        static_cast<const U *>(W2), reinterpret_cast<U *>(base + L.w2), c.d, 1, c.f, tn_dn);
    if (c.n_shared > 0) {
        const int fs = c.n_shared * c.f_shared;
        amax_up_kernel<<<dim3((fs + 255) / 256, 2), 256, 0, s>>>(static_cast<const U *>(W1s),
                                                                  static_cast<const U *>(W3s), f(L.sc13s), c.d,
                                                                  c.n_shared, c.f_shared, 2 * fs);
        quant_up_kernel<<<dim3((fs + 31) / 32, (c.d + 31) / 32, 2), blk, 0, s>>>(
            static_cast<const U *>(W1s), static_cast<const U *>(W3s), f(L.sc13s), q(L.w13s), c.d, c.n_shared,
            c.f_shared, tn_up, 1);
        pack_down_kernel<U><<<dim3((c.d + 31) / 32, (fs + 31) / 32, 1), blk, 0, s>>>(
            static_cast<const U *>(W2s), reinterpret_cast<U *>(base + L.w2s), c.d, c.n_shared, c.f_shared, tn_dn);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const moe_config &c, const void *W1, const void *W3, const void *W2, const void *W1s,
                        const void *W3s, const void *W2s, void *packed, cudaStream_t s) {
    if (c.dtype == MOE_F32) return pack_typed<float>(c, W1, W3, W2, W1s, W3s, W2s, packed, s);
    if (fp8_weights(c)) return pack_fp8(c, W1, W3, W2, W1s, W3s, W2s, packed, s);
    if (fp8_up(c)) return pack_fp8_up(c, W1, W3, W2, W1s, W3s, W2s, packed, s);
    return pack_typed<unsigned short>(c, W1, W3, W2, W1s, W3s, W2s, packed, s);   // bf16 bits
}

}  // namespace moe
