// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (bf16 in, fp32
// accumulate in TMEM): host launchers of the persistent kernel in tc_gemm.cuh.
//
// Expert FFN with W1, W3 up and W2 down ("lnwmold.com GPT-4 MoE article" §2.2),
// read as SwiGLU:  H_e = SiLU(X_e W1_e) * (X_e W3_e),  Y_e = H_e W2_e.
// Up: A = x_perm rows (shared experts: x), B = packed [W1|W3] groups, K = d,
//     256-wide tiles (128 hidden columns) when f % 128 == 0, else 128-wide.
// Down: A = H rows, B = packed W2, K = f, 256-wide tiles when d % 256 == 0.
#include <algorithm>

#include "tc_gemm.cuh"

namespace moe {

cudaError_t launch_ffn_up_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                                  const void *packed, const void *x, void *H, void *Hs, unsigned *err,
                                  cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const bool shared = c.n_shared > 0;
    const int shared_rows = shared ? c.T : 0;
    const int fs = z.fs_tot;
    const uint64_t rr = (uint64_t)z.rows_routed;
    const int64_t mtiles = (z.rows_routed + kBM - 1) / kBM + c.E;
    const int64_t mtiles_s = (shared_rows + kBM - 1) / kBM;

    // H = SiLU(X W1) * (X W3); B = packed [W1|W3] tile images, one bulk copy per stage
    const int bn1 = up_tile_n(c);
    const bool wide1 = bn1 == 256;
    CUtensorMap a0, a1;
    bool ok = make_tmap_bf16(&a0, x_perm, rr, c.d, kBM);
    ok = ok && make_tmap_bf16(&a1, shared ? x : x_perm, shared ? (uint64_t)c.T : rr, c.d, kBM);
    if (!ok) return cudaErrorInvalidValue;
    const CUtensorMap &b0 = a0, &b1 = a1;   // unused: B is not loaded through tensor maps
    TcArgs g1{};
    g1.g = GroupedShape{off, c.E, shared_rows, 2 * c.f / bn1, shared ? 2 * fs / bn1 : 0};
    g1.K0 = c.d;
    g1.K1 = c.d;
    g1.b_rows0 = 2 * c.f;
    g1.Bt0 = reinterpret_cast<const uint8_t *>(pk + L.w13);
    g1.Bt1 = reinterpret_cast<const uint8_t *>(pk + L.w13s);
    g1.bt_seg0 = (size_t)2 * c.f * c.d * 2;
    g1.C0 = H;
    g1.C1 = Hs;
    g1.ldc0 = c.f;
    g1.ldc1 = fs;
    g1.err = err;
    const int64_t tiles1 = mtiles * g1.g.nblk_routed + mtiles_s * g1.g.nblk_shared;
    return wide1 ? launch_gemm<256, kEpiSwiGLU>(a0, a1, b0, b1, g1, tiles1, s)
                 : launch_gemm<128, kEpiSwiGLU>(a0, a1, b0, b1, g1, tiles1, s);
}

cudaError_t launch_ffn_down_tcgen05(const moe_config &c, const Sizes &z, const void *H, const void *Hs,
                                    const int32_t *off, const void *packed, void *Y, unsigned *err, cudaStream_t s) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const bool shared = c.n_shared > 0;
    const int shared_rows = shared ? c.T : 0;
    const int fs = z.fs_tot;
    const uint64_t rr = (uint64_t)z.rows_routed;
    const int64_t mtiles = (z.rows_routed + kBM - 1) / kBM + c.E;
    const int64_t mtiles_s = (shared_rows + kBM - 1) / kBM;

    // Y = H W2; B = packed W2 tile images, one bulk copy per stage
    const int bn2 = down_tile_n(c);
    CUtensorMap a0, a1;
    bool ok = make_tmap_bf16(&a0, H, rr, c.f, kBM);
    ok = ok && make_tmap_bf16(&a1, shared ? Hs : H, shared ? (uint64_t)c.T : rr, shared ? fs : c.f, kBM);
    if (!ok) return cudaErrorInvalidValue;
    const CUtensorMap &b0 = a0, &b1 = a1;   // unused: B is not loaded through tensor maps
    TcArgs g2{};
    g2.g = GroupedShape{off, c.E, shared_rows, c.d / bn2, c.d / bn2};
    g2.K0 = c.f;
    g2.K1 = shared ? fs : c.f;
    g2.b_rows0 = c.d;
    g2.Bt0 = reinterpret_cast<const uint8_t *>(pk + L.w2);
    g2.Bt1 = reinterpret_cast<const uint8_t *>(pk + L.w2s);
    g2.bt_seg0 = (size_t)c.d * c.f * 2;
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
