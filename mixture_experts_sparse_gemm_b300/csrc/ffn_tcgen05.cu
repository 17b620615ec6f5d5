// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (bf16 in, fp32
// accumulate in TMEM).
//
// Expert FFN with W1, W3 up and W2 down ("lnwmold.com GPT-4 MoE article" §2.2),
// read as SwiGLU:  H_e = SiLU(X_e W1_e) * (X_e W3_e),  Y_e = H_e W2_e.
//
// One persistent kernel per GEMM, one CTA per SM, 6 warps:
//   warp 0      TMA producer: 128x64 A tile + BNx64 B tile per stage, 128-byte
//               swizzle, into a STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1      TMEM allocator and MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16)
//               per stage into one of two TMEM accumulators (2 x BN columns)
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (one row per
//               thread), SwiGLU or bf16 conversion, masked row stores; overlaps
//               the next tile's main loop through the second accumulator
// Tiles never straddle experts: the tile table is built on the device from off[]
// (segment s < E = routed expert s, segment E = merged shared experts), and a
// segment's last M tile reads rows past its end (the next expert's rows, or zero
// fill beyond the tensor) whose results are never stored.
//
// Up projection: the packed B rows of a 256-wide tile are [64 W1 cols | the same
// 64 W3 cols | next 64 W1 | same W3], so a thread holds gate and up values of the
// same hidden columns and writes SiLU(gate) * up straight to H.
#include <algorithm>

#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr int kEpiSwiGLU = 0;
constexpr int kEpiStore = 1;

template <int BN>
struct TcCfg {
    static constexpr int kStages = (BN == 256) ? 4 : 6;
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kBarBytes = (2 * kStages + 5) * 8;
    static constexpr int kMiscBytes = 64 + sizeof(int) * (3 * (kMaxE + 2));
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes + kMiscBytes;
};

struct TcArgs {
    GroupedShape g;
    int K0, K1;        // reduction width, routed / shared
    int b_rows0;       // packed B rows per routed expert
    void *C0;          // routed output rows (bf16)
    void *C1;          // shared output rows (bf16)
    int ldc0, ldc1;    // output row pitch in elements
    unsigned *err;
};

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                           const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                           TcArgs a) {
    using C = TcCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(tiles + (size_t)C::kStages * C::kStageBytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::kStages;
    uint64_t *tfull = bars + 2 * C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *tile_start = reinterpret_cast<int *>(tmem_holder + 16);
    int *seg_row0 = tile_start + (kMaxE + 2);
    int *seg_rows = seg_row0 + (kMaxE + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull[i]), 1);
            mbar_init(smem_u32(&tempty[i]), 4);
        }
        mbar_init(smem_u32(drain), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tmap(&tmA0);
        prefetch_tmap(&tmA1);
        prefetch_tmap(&tmB0);
        prefetch_tmap(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
        fence_before();
    }
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int S = build_tile_table<kBM>(a.g, tile_start, seg_row0, seg_rows);
    const int total = tile_start[S];

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int s, mb, nb;
                decode_tile<kBM>(a.g, tile_start, seg_rows, S, tile, s, mb, nb);
                const bool routed = s < a.g.E;
                const CUtensorMap *mA = routed ? &tmA0 : &tmA1;
                const CUtensorMap *mB = routed ? &tmB0 : &tmB1;
                const int arow = seg_row0[s] + mb * kBM;
                const int brow = (routed ? s * a.b_rows0 : 0) + nb * BN;
                const int nk = (routed ? a.K0 : a.K1) / kBK;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    uint8_t *st = tiles + (size_t)stage * C::kStageBytes;
                    mbar_arrive_expect_tx(fb, C::kStageBytes);
                    tma_load_2d(smem_u32(st), mA, kb * kBK, arow, fb);
                    tma_load_2d(smem_u32(st + C::kABytes), mB, kb * kBK, brow, fb);
                    ++issued;
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // leave no copy in flight: wait (bounded) for the last stages issued
                const int n = issued < C::kStages ? issued : C::kStages;
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < n; ++i) {
                    if (--st < 0) {
                        st = C::kStages - 1;
                        ph ^= 1u;
                    }
                    const uint32_t fb = smem_u32(&full[st]);
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(fb, ph) && globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
                int s, mb, nb;
                decode_tile<kBM>(a.g, tile_start, seg_rows, S, tile, s, mb, nb);
                const int nk = ((s < a.g.E) ? a.K0 : a.K1) / kBK;
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, a.err)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(smem_u32(&full[stage]), phase, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint32_t sa = smem_u32(tiles + (size_t)stage * C::kStageBytes);
                    const uint64_t adesc = sdesc_k128(sa);
                    const uint64_t bdesc = sdesc_k128(sa + C::kABytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // advance 16 bf16 = 32 bytes inside the swizzle atom (encoded >> 4)
                        mma_bf16(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), kIdesc,
                                 (kb | kk) != 0);
                    }
                    mma_commit(smem_u32(&empty[stage]));
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull[acc]));
            }
            // every MMA issued has finished before TMEM is released
            mma_commit(smem_u32(drain));
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(smem_u32(drain), 0) && globaltimer() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;   // TMEM lanes [32*quarter, 32*quarter + 32)
        const int row = quarter * 32 + lane;
        int it = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
            int s, mb, nb;
            decode_tile<kBM>(a.g, tile_start, seg_rows, S, tile, s, mb, nb);
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            int ok = 1;
            if (lane == 0) ok = wait_bounded(smem_u32(&tfull[acc]), acc_phase, abort_flag, a.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            fence_after();
            const bool routed = s < a.g.E;
            const int rows = min(kBM, seg_rows[s] - mb * kBM);
            const int grow = seg_row0[s] + mb * kBM + row;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            __nv_bfloat16 *Cp = static_cast<__nv_bfloat16 *>(routed ? a.C0 : a.C1);
            const int ldc = routed ? a.ldc0 : a.ldc1;
            if constexpr (EPI == kEpiSwiGLU) {
#pragma unroll 1
                for (int grp = 0; grp < BN / 128; ++grp) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t g[16], u[16];
                        tmem_ld16(taddr + grp * 128 + c * 16, g);
                        tmem_ld16(taddr + grp * 128 + 64 + c * 16, u);
                        tmem_ld_wait();
                        uint32_t o[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                            const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                            o[i] = pack_bf16x2(h0, h1);
                        }
                        if (row < rows) {
                            uint4 *dst = reinterpret_cast<uint4 *>(Cp + (size_t)grow * ldc + nb * (BN / 2) +
                                                                   grp * 64 + c * 16);
                            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c * 16, v);
                    tmem_ld_wait();
                    uint32_t o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    if (row < rows) {
                        uint4 *dst = reinterpret_cast<uint4 *>(Cp + (size_t)grow * ldc + nb * BN + c * 16);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int BN, int EPI>
cudaError_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0, const CUtensorMap &b1,
                        const TcArgs &args, int64_t max_tiles, cudaStream_t s) {
    auto kern = tc_grouped_gemm_kernel<BN, EPI>;
    const size_t smem = TcCfg<BN>::kSmem;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)std::max<int64_t>(1, max_tiles);
    kern<<<grid, kThreads, smem, s>>>(a0, a1, b0, b1, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                               const void *packed, const void *x, void *H, void *Hs, void *Y, unsigned *err,
                               cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const bool shared = c.n_shared > 0;
    const int shared_rows = shared ? c.T : 0;
    const int fs = z.fs_tot;
    const uint64_t rr = (uint64_t)z.rows_routed;
    const int64_t mtiles = (z.rows_routed + kBM - 1) / kBM + c.E;
    const int64_t mtiles_s = (shared_rows + kBM - 1) / kBM;

    // ---- up projection + SwiGLU: H = SiLU(X W1) * (X W3)
    const bool wide1 = (c.f % 128 == 0) && (!shared || fs % 128 == 0);
    const int bn1 = wide1 ? 256 : 128;
    CUtensorMap a0, a1, b0, b1;
    bool ok = make_tmap_bf16(&a0, x_perm, rr, c.d, kBM);
    ok = ok && make_tmap_bf16(&a1, shared ? x : x_perm, shared ? (uint64_t)c.T : rr, c.d, kBM);
    ok = ok && make_tmap_bf16(&b0, pk + L.w13, (uint64_t)c.E * 2 * c.f, c.d, bn1);
    ok = ok && make_tmap_bf16(&b1, shared ? pk + L.w13s : pk + L.w13, shared ? (uint64_t)2 * fs : (uint64_t)c.E * 2 * c.f,
                              c.d, bn1);
    if (!ok) return cudaErrorInvalidValue;
    TcArgs g1{};
    g1.g = GroupedShape{off, c.E, shared_rows, 2 * c.f / bn1, shared ? 2 * fs / bn1 : 0};
    g1.K0 = c.d;
    g1.K1 = c.d;
    g1.b_rows0 = 2 * c.f;
    g1.C0 = H;
    g1.C1 = Hs;
    g1.ldc0 = c.f;
    g1.ldc1 = fs;
    g1.err = err;
    const int64_t tiles1 = mtiles * g1.g.nblk_routed + mtiles_s * g1.g.nblk_shared;
    cudaError_t e = wide1 ? launch_gemm<256, kEpiSwiGLU>(a0, a1, b0, b1, g1, tiles1, s)
                          : launch_gemm<128, kEpiSwiGLU>(a0, a1, b0, b1, g1, tiles1, s);
    if (e != cudaSuccess) return e;

    // ---- down projection: Y = H W2
    const int bn2 = (c.d % 256 == 0) ? 256 : 128;
    ok = make_tmap_bf16(&a0, H, rr, c.f, kBM);
    ok = ok && make_tmap_bf16(&a1, shared ? Hs : H, shared ? (uint64_t)c.T : rr, shared ? fs : c.f, kBM);
    ok = ok && make_tmap_bf16(&b0, pk + L.w2, (uint64_t)c.E * c.d, c.f, bn2);
    ok = ok && make_tmap_bf16(&b1, shared ? pk + L.w2s : pk + L.w2, shared ? (uint64_t)c.d : (uint64_t)c.E * c.d,
                              shared ? fs : c.f, bn2);
    if (!ok) return cudaErrorInvalidValue;
    TcArgs g2{};
    g2.g = GroupedShape{off, c.E, shared_rows, c.d / bn2, c.d / bn2};
    g2.K0 = c.f;
    g2.K1 = shared ? fs : c.f;
    g2.b_rows0 = c.d;
    g2.C0 = Y;
    g2.C1 = static_cast<__nv_bfloat16 *>(Y) + (size_t)z.rows_routed * c.d;
    g2.ldc0 = c.d;
    g2.ldc1 = c.d;
    g2.err = err;
    const int64_t tiles2 = (mtiles + mtiles_s) * (c.d / bn2);
    return bn2 == 256 ? launch_gemm<256, kEpiStore>(a0, a1, b0, b1, g2, tiles2, s)
                      : launch_gemm<128, kEpiStore>(a0, a1, b0, b1, g2, tiles2, s);
}

}  // namespace moe
