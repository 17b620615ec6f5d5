// Grouped SwiGLU expert GEMMs on the 5th-generation tensor cores (bf16 in, fp32
// accumulate in TMEM): host launchers of the persistent kernel in tc_gemm.cuh.
//
// Expert FFN with W1, W3 up and W2 down ("lnwmold.com GPT-4 MoE article" §2.2),
// read as SwiGLU:  H_e = SiLU(X_e W1_e) * (X_e W3_e),  Y_e = H_e W2_e.
// Up: A = x_perm rows (shared experts: x), B = packed [W1|W3] tile images, K = d,
//     256-wide tiles (128 hidden columns) when f % 128 == 0, else 128-wide.
// Down: A = H rows, B = packed W2 tile images, K = f, 256-wide tiles when d % 256 == 0.
// Fused: both GEMMs in one persistent launch, down tiles after up tiles, each
//     down tile waiting (on the device) for the up tiles that produce its H rows.
// FP8 weights (MOE_BF16_FP8W): the same launches with the W8 kernel, which streams
//     E4M3 tile images, expands them to bf16 in shared memory and applies the
//     per-column scales in the epilogue.
// FP8 up projection (MOE_BF16_FP8UP): the fused launch with the F8A kernel; the up
//     tiles multiply E4M3 activation rows by E4M3 W1|W3 images on kind::f8f6f4 and
//     scale by row and column, the down tiles stay bf16.
#include <algorithm>

#include "tc_gemm.cuh"

namespace moe {
namespace {

struct FfnMaps {
    CUtensorMap a0, a1;
};

// M tiles per group of the tile order (tc_gemm.cuh): as many 128-row blocks of A as
// fit `share` bytes, which stay in L2 while the group's N blocks stream the weights.
// By default x_perm rows of the up projection take 40 MiB and H rows of the down
// projection 64 MiB: the L2 (126 MB) spans two dies, and rows that CTAs on both dies
// read are held on both, so a group fills at most about half of it.
int tile_group(uint64_t share, int K) {
    return (int)std::min<uint64_t>(1u << 20, std::max<uint64_t>(1, share / ((uint64_t)kBM * K * 2)));
}

// Up projection: A = x_perm (routed) / x (shared), B = [W1|W3] images, C = H / Hs.
// FP8 up projection (f8 != nullptr): x_perm and x hold E4M3 codes, with the row
// scales of f8.
bool up_gemm(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off, const void *packed,
             const void *x, void *H, void *Hs, TcGemm &G, FfnMaps &m, const F8Rows *f8 = nullptr) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const bool shared = c.n_shared > 0;
    const int fs = z.fs_tot;
    const int bn = up_tile_n(c);
    const uint64_t rr = (uint64_t)z.rows_routed;
    auto tmap = f8 ? make_tmap_u8 : make_tmap_bf16;
    bool ok = tmap(&m.a0, x_perm, rr, c.d, kBM);
    ok = ok && tmap(&m.a1, shared ? x : x_perm, shared ? (uint64_t)c.T : rr, c.d, kBM);
    G = TcGemm{};
    G.g = GroupedShape{off, c.E, shared ? c.T : 0, 2 * c.f / bn, shared ? 2 * fs / bn : 0};
    G.K0 = c.d;
    G.K1 = c.d;
    G.b_rows0 = 2 * c.f;
    const size_t wb = (fp8_weights(c) || fp8_up(c)) ? 1 : 2;   // bytes per stored weight
    G.Bt0 = reinterpret_cast<const uint8_t *>(pk + L.w13);
    G.Bt1 = reinterpret_cast<const uint8_t *>(pk + L.w13s);
    G.bt_seg0 = (size_t)2 * c.f * c.d * wb;
    if (fp8_weights(c) || fp8_up(c)) {
        G.sc0 = reinterpret_cast<const float *>(pk + L.sc13);
        G.sc1 = reinterpret_cast<const float *>(pk + L.sc13s);
    }
    if (f8) {
        G.a_f8 = 1;
        G.rs0 = f8->rs0;
        G.rtok0 = f8->rtok0;
        G.rs1 = f8->rs1;
    }
    G.img_rows = bn;
    G.group_m = tile_group(tile_group_bytes(0), c.d);
    G.C0 = H;
    G.C1 = Hs;
    G.ldc0 = c.f;
    G.ldc1 = fs;
    return ok;
}

// Down projection: A = H (routed) / Hs (shared), B = W2 images, C = Y rows.
bool down_gemm(const moe_config &c, const Sizes &z, const void *H, const void *Hs, const int32_t *off,
               const void *packed, void *Y, TcGemm &G, FfnMaps &m) {
    const PackedLayout L = packed_layout(c);
    const char *pk = static_cast<const char *>(packed);
    const bool shared = c.n_shared > 0;
    const int fs = z.fs_tot;
    const int bn = down_tile_n(c);
    const uint64_t rr = (uint64_t)z.rows_routed;
    bool ok = make_tmap_bf16(&m.a0, H, rr, c.f, kBM);
    ok = ok && make_tmap_bf16(&m.a1, shared ? Hs : H, shared ? (uint64_t)c.T : rr, shared ? fs : c.f, kBM);
    G = TcGemm{};
    G.g = GroupedShape{off, c.E, shared ? c.T : 0, c.d / bn, c.d / bn};
    G.K0 = c.f;
    G.K1 = shared ? fs : c.f;
    G.b_rows0 = c.d;
    const size_t wb = fp8_weights(c) ? 1 : 2;
    G.Bt0 = reinterpret_cast<const uint8_t *>(pk + L.w2);
    G.Bt1 = reinterpret_cast<const uint8_t *>(pk + L.w2s);
    G.bt_seg0 = (size_t)c.d * c.f * wb;
    if (fp8_weights(c)) {
        G.sc0 = reinterpret_cast<const float *>(pk + L.sc2);
        G.sc1 = reinterpret_cast<const float *>(pk + L.sc2s);
    }
    G.img_rows = bn;
    G.group_m = tile_group(tile_group_bytes(1), c.f);
    G.C0 = Y;
    G.C1 = static_cast<__nv_bfloat16 *>(Y) + (size_t)z.rows_routed * c.d;
    G.ldc0 = c.d;
    G.ldc1 = c.d;
    return ok;
}

// Upper bound on the M tiles of a launch (real count is known on the device only).
int64_t max_mtiles(const moe_config &c, const Sizes &z) {
    return (z.rows_routed + kBM - 1) / kBM + c.E + (c.n_shared > 0 ? (c.T + kBM - 1) / kBM : 0);
}

}  // namespace

size_t ffn_dep_counters(const moe_config &c) { return (size_t)max_mtiles(c, sizes_of(c)) + 1; }

bool ffn_fused_supported(const moe_config &c) { return up_tile_n(c) == 256 && down_tile_n(c) == 256; }

cudaError_t launch_ffn_up_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                                  const void *packed, const void *x, void *H, void *Hs, unsigned *err,
                                  cudaStream_t s) {
    TcArgs g{};
    FfnMaps m;
    if (!up_gemm(c, z, x_perm, off, packed, x, H, Hs, g.p[0], m)) return cudaErrorInvalidValue;
    g.err = err;
    const int64_t tiles = max_mtiles(c, z) * std::max(g.p[0].g.nblk_routed, g.p[0].g.nblk_shared);
    if (fp8_weights(c)) return launch_gemm<256, kEpiSwiGLU, true>(m.a0, m.a1, m.a0, m.a1, g, tiles, s);
    return g.p[0].img_rows == 256 ? launch_gemm<256, kEpiSwiGLU>(m.a0, m.a1, m.a0, m.a1, g, tiles, s)
                                  : launch_gemm<128, kEpiSwiGLU>(m.a0, m.a1, m.a0, m.a1, g, tiles, s);
}

cudaError_t launch_ffn_down_tcgen05(const moe_config &c, const Sizes &z, const void *H, const void *Hs,
                                    const int32_t *off, const void *packed, void *Y, unsigned *err, cudaStream_t s,
                                    const int32_t *row_token, const float *row_gate) {
    TcArgs g{};
    FfnMaps m;
    if (!down_gemm(c, z, H, Hs, off, packed, Y, g.p[0], m)) return cudaErrorInvalidValue;
    g.err = err;
    g.gated = row_token != nullptr;
    g.row_token = row_token;
    g.row_gate = row_gate;
    const int64_t tiles = max_mtiles(c, z) * g.p[0].g.nblk_routed;
    if (fp8_weights(c)) return launch_gemm<256, kEpiStore, true>(m.a0, m.a1, m.a0, m.a1, g, tiles, s);
    return g.p[0].img_rows == 256 ? launch_gemm<256, kEpiStore>(m.a0, m.a1, m.a0, m.a1, g, tiles, s)
                                  : launch_gemm<128, kEpiStore>(m.a0, m.a1, m.a0, m.a1, g, tiles, s);
}

cudaError_t launch_ffn_fused_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                                     const void *packed, const void *x, void *H, void *Hs, void *Y, int *dep,
                                     unsigned *err, cudaStream_t s, const int32_t *row_token, const float *row_gate,
                                     bool dep_zeroed, const F8Rows *f8) {
    TcArgs g{};
    FfnMaps mu, md;
    if (!up_gemm(c, z, x_perm, off, packed, x, H, Hs, g.p[0], mu, f8)) return cudaErrorInvalidValue;
    if (!down_gemm(c, z, H, Hs, off, packed, Y, g.p[1], md)) return cudaErrorInvalidValue;
    g.dep = dep;
    g.err = err;
    g.gated = row_token != nullptr;
    g.row_token = row_token;
    g.row_gate = row_gate;
    if (!dep_zeroed) {
        const cudaError_t e = cudaMemsetAsync(dep, 0, sizeof(int) * ffn_dep_counters(c), s);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = max_mtiles(c, z) * (g.p[0].g.nblk_routed + g.p[1].g.nblk_routed);
    if (fp8_weights(c)) return launch_gemm<256, kEpiFfn, true>(mu.a0, mu.a1, mu.a0, mu.a1, md.a0, md.a1, g, tiles, s);
    if (f8) return launch_gemm<256, kEpiFfn, false, true>(mu.a0, mu.a1, mu.a0, mu.a1, md.a0, md.a1, g, tiles, s);
    return launch_gemm<256, kEpiFfn>(mu.a0, mu.a1, mu.a0, mu.a1, md.a0, md.a1, g, tiles, s);
}

}  // namespace moe
