// Router on the tensor cores (bf16): the logits u = x W_r are one dense GEMM
// [T, d] x [d, E], so they run on tcgen05 through the persistent GEMM of
// tc_gemm.cuh (M = 128 tokens per tile, N = E rounded up to 16..256, K = d), and
// the whole scoring step lives in its TMEM epilogue: one thread per token reads
// its row of E logits, applies the logit offset, scores them (softmax or
// sigmoid, "技术日报 2026-04-14" §3.2 / §3.5), selects the top k on
// score + selection bias (§3.1, §4.3) and writes indices and (renormalised,
// §9.1) weights; for Expert Choice (§3.3) it writes the softmax scores
// expert-major for the column selection.  The logits never reach HBM.
//
// W_r arrives as [d][E] (the pages' x W_r).  When its rows are whole 16-byte units
// (E a multiple of 8) the MMA reads it in place as an MN-major B operand: TMA boxes
// of [64 d rows][64 experts], columns past E zero-filled, N = E rounded up to 64..256.
// Otherwise a small transpose writes W_r^T [Npad][d] (zero rows E..Npad-1) into the
// workspace for the K-major path.  The token rows are the tile table's one
// unrouted segment [0, T), so no segment table is needed in device memory.
#include "tc_gemm.cuh"

namespace moe {
namespace {

int padded_n(int E) {
    int n = 16;
    while (n < E) n *= 2;
    return n;   // 16, 32, 64, 128 or 256
}

// K splits of the router GEMM: with few 128-token tiles (T small, d large) the
// d-reduction is spread over up to 8 CTAs per tile so that ~all 148 SMs of a B300
// stream x; the CTAs of one tile form a cluster that sums their partial logits
// through distributed shared memory and selects in the same launch.  Fixed SM
// count: workspace sizes are computed without a device query.
constexpr int kRouteSms = 148;
int route_splits(const moe_config &c) {
    const int mtiles = (c.T + kBM - 1) / kBM;
    // the fused scoring epilogue wins when the tiles already cover half the SMs, or
    // when each tile is short (d < 2048) and its top-k cheap (E * k-slots < 256)
    const int kslots = (c.mode == MOE_EXPERT_CHOICE || c.k <= 1) ? 1 : (c.k <= 2 ? 2 : (c.k <= 4 ? 4 : 8));
    if (mtiles >= kRouteSms / 2) return 1;
    if (c.d / kBK < 32 && c.E * kslots < 256) return 1;
    int s = kRouteSms / (mtiles > 0 ? mtiles : 1);
    s = s < kMaxRouteSplits ? s : kMaxRouteSplits;
    const int quarter_k = (c.d / kBK) / 4;
    s = s < quarter_k ? s : quarter_k;
    return s >= 2 ? s : 1;
}

// W_r read in place (MN-major B): its rows of E bf16 are 16-byte multiples
bool wr_in_place(const moe_config &c) { return c.E % 8 == 0; }
// N of the router GEMM: the MN-major boxes are 64 experts wide
int route_n(const moe_config &c) {
    const int n = padded_n(c.E);
    return wr_in_place(c) && n < 64 ? 64 : n;
}
size_t wr_t_bytes(const moe_config &c) {
    return wr_in_place(c) ? 0 : align_up((size_t)route_n(c) * c.d * 2, 256);
}

// wr_t[e][i] = W_r[i][e] for e < E, 0 for E <= e < npad
__global__ void transpose_router_kernel(const __nv_bfloat16 *__restrict__ Wr, __nv_bfloat16 *__restrict__ wr_t,
                                        int d, int E, int npad) {
    __shared__ __nv_bfloat16 tile[32][34];
    pdl_trigger();   // the router GEMM may start its setup; it waits for this grid before reading
    const int e0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    for (int ii = threadIdx.y; ii < 32; ii += blockDim.y) {
        const int i = i0 + ii, e = e0 + threadIdx.x;
        tile[ii][threadIdx.x] = (i < d && e < E) ? Wr[(size_t)i * E + e] : __float2bfloat16_rn(0.f);
    }
    __syncthreads();
    for (int ee = threadIdx.y; ee < 32; ee += blockDim.y) {
        const int e = e0 + ee, i = i0 + threadIdx.x;
        if (e < npad && i < d) wr_t[(size_t)e * d + i] = tile[threadIdx.x][ee];
    }
}

template <int EPI>
cudaError_t launch_route_n(int npad, const CUtensorMap &a0, const CUtensorMap &b0, const TcArgs &g, int64_t tiles,
                           cudaStream_t s) {
    switch (npad) {
        case 16: return launch_gemm<16, EPI>(a0, a0, b0, b0, g, tiles, s);
        case 32: return launch_gemm<32, EPI>(a0, a0, b0, b0, g, tiles, s);
        case 64: return launch_gemm<64, EPI>(a0, a0, b0, b0, g, tiles, s);
        case 128: return launch_gemm<128, EPI>(a0, a0, b0, b0, g, tiles, s);
        default: return launch_gemm<256, EPI>(a0, a0, b0, b0, g, tiles, s);
    }
}

// split-K router in clusters of `splits` CTAs; the selecting warps hold
// max(1, npad / 32) experts per lane
cudaError_t launch_split_n(int npad, const CUtensorMap &a0, const CUtensorMap &b0, const TcArgs &g, int tiles,
                           int splits, cudaStream_t s) {
    switch (npad) {
        case 16: return launch_gemm_split_route<16, kEpiSplitRoute + 1>(a0, b0, g, tiles, splits, s);
        case 32: return launch_gemm_split_route<32, kEpiSplitRoute + 1>(a0, b0, g, tiles, splits, s);
        case 64: return launch_gemm_split_route<64, kEpiSplitRoute + 2>(a0, b0, g, tiles, splits, s);
        case 128: return launch_gemm_split_route<128, kEpiSplitRoute + 4>(a0, b0, g, tiles, splits, s);
        default: return launch_gemm_split_route<256, kEpiSplitRoute + 8>(a0, b0, g, tiles, splits, s);
    }
}

}  // namespace

bool route_tcgen05_supported(const moe_config &c) { return bf16_acts(c) && c.E <= kMaxE && c.d % 64 == 0; }

size_t route_tcgen05_scratch_bytes(const moe_config &c) { return wr_t_bytes(c); }

int route_tcgen05_launches(const moe_config &c) { return (wr_in_place(c) ? 0 : 1) + 1; }

cudaError_t launch_route_tcgen05(const moe_config &c, const void *x, const void *W_r, const float *logit_offset,
                                 const float *sel_bias, int32_t *topk_idx, float *topk_w, float *scores_t,
                                 float *psum_rows, void *wr_t, unsigned *err, cudaStream_t s) {
    const int npad = route_n(c);
    char *scratch = static_cast<char *>(wr_t);
    const int splits = route_splits(c);
    CUtensorMap a0, b0;
    bool ok = make_tmap_bf16(&a0, x, (uint64_t)c.T, c.d, kBM);
    TcArgs g{};
    if (wr_in_place(c)) {
        // [d][E] row-major, boxes of 64 d rows x 64 experts (past E: zero fill)
        ok = ok && make_tmap_bf16(&b0, W_r, (uint64_t)c.d, c.E, 64);
        g.p[0].b_mn = 1;
    } else {
        __nv_bfloat16 *wt = reinterpret_cast<__nv_bfloat16 *>(scratch);
        const dim3 tg((npad + 31) / 32, (c.d + 31) / 32);
        transpose_router_kernel<<<tg, dim3(32, 8), 0, s>>>(static_cast<const __nv_bfloat16 *>(W_r), wt, c.d, c.E,
                                                           npad);
        ok = ok && make_tmap_bf16(&b0, wt, (uint64_t)npad, c.d, npad);
    }
    if (!ok) return cudaErrorInvalidValue;
    g.p[0].g = GroupedShape{nullptr, 0, c.T, 1, 1};   // one unrouted segment: the T token rows
    g.p[0].K0 = c.d;
    g.p[0].K1 = c.d;
    g.p[0].b_rows0 = npad;
    g.route = RouteEpi{logit_offset, sel_bias, topk_idx, topk_w, scores_t, psum_rows, c.T, c.E, c.k, c.gate, c.mode,
                       c.renormalize};
    g.err = err;
    const int64_t tiles = (c.T + kBM - 1) / kBM;
    if (splits > 1) {
        // split-K partial logits, reduced and selected inside each token tile's cluster
        g.p[0].g.nblk_shared = splits;
        g.p[0].ksplit = splits;
        return launch_split_n(npad, a0, b0, g, (int)tiles, splits, s);
    }
    const int kmax = (c.mode == MOE_EXPERT_CHOICE || c.k <= 1) ? 1 : (c.k <= 2 ? 2 : (c.k <= 4 ? 4 : 8));
    switch (kmax) {
        case 1: return launch_route_n<kEpiRoute + 1>(npad, a0, b0, g, tiles, s);
        case 2: return launch_route_n<kEpiRoute + 2>(npad, a0, b0, g, tiles, s);
        case 4: return launch_route_n<kEpiRoute + 4>(npad, a0, b0, g, tiles, s);
        default: return launch_route_n<kEpiRoute + 8>(npad, a0, b0, g, tiles, s);
    }
}

}  // namespace moe
