// Internal declarations shared by the CUDA translation units of the MoE library.
// Nothing here is part of the C ABI (that is include/moe_b300.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_b300.h"

namespace moe {

constexpr int kMaxE = 256;     // routed experts
constexpr int kMaxK = 8;       // experts per token (token choice)
constexpr int kPsumRows = 64;   // rows of per-CTA router score sums (CTA index mod 64)
constexpr int kMaxRouteSplits = 8;   // split-K ways of the tensor-core router at most
constexpr int kGroup = 64;     // W1/W3 interleave width of the packed up-projection

// bits of the device error word
constexpr unsigned kErrWaitTimeout = 1u;
constexpr unsigned kErrBadIndex = 2u;     // an expert or token id outside its range was skipped

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// bf16 activations (MOE_BF16, MOE_BF16_FP8W, MOE_BF16_FP8UP): the tensor-core paths
inline bool bf16_acts(const moe_config &c) {
    return c.dtype == MOE_BF16 || c.dtype == MOE_BF16_FP8W || c.dtype == MOE_BF16_FP8UP;
}
// expert weights stored as E4M3 codes + per-output-channel fp32 scales
inline bool fp8_weights(const moe_config &c) { return c.dtype == MOE_BF16_FP8W; }
// the up projection on E4M3 operands (kind::f8f6f4): activations per token, W1/W3
// per output channel; H, W2 and Y in bf16
inline bool fp8_up(const moe_config &c) { return c.dtype == MOE_BF16_FP8UP; }

// ----------------------------------------------------------------------------- sizes
struct Sizes {
    int64_t rows_routed;   // T*k (token choice) or E*cap (expert choice)
    int64_t rows_total;    // + T when shared experts exist
    int32_t cap;           // per-expert capacity, -1 unlimited
    int32_t fs_tot;        // n_shared * f_shared
    int32_t elt;           // bytes per element of cfg->dtype
};
Sizes sizes_of(const moe_config &c);

// N width of the tensor-core tiles of the two expert GEMMs (bf16).  The packed
// bf16 weights are tiled with the same widths, so pack and GEMM must agree.
inline int up_tile_n(const moe_config &c) {
    const int fs = c.n_shared > 0 ? c.n_shared * c.f_shared : 0;
    return (c.f % 128 == 0 && fs % 128 == 0) ? 256 : 128;
}
inline int down_tile_n(const moe_config &c) { return (c.d % 256 == 0) ? 256 : 128; }

// Element offset of (row p, column i) of a [N][K] bf16 operand stored as the
// tensor-core tile images: tiles of BN rows x 64 columns, N-tile major then
// K-tile, each tile BN rows of 128 bytes with the 16-byte chunks of row r
// permuted by chunk ^ (r % 8) -- the 128-byte swizzle a TMA load would apply.
// One tile is then a single contiguous copy that lands in shared memory
// exactly as the MMA descriptor expects.
__host__ __device__ inline size_t tiled_offset(int p, int i, int BN, int K) {
    const int nb = p / BN, r = p % BN, kb = i / 64, ch = (i % 64) / 8, w = i % 8;
    return (((size_t)nb * (K / 64) + kb) * BN + r) * 64 + (size_t)((ch ^ (r & 7)) * 8 + w);
}

// Byte offset of (row p, column i) of a [N][K] FP8 operand stored as tile images:
// BN rows x 64 one-byte columns per tile, N-tile major then K-tile, rows plain
// (the converter warps of the grouped GEMM expand a tile to the swizzled bf16 layout).
__host__ __device__ inline size_t tiled_offset8(int p, int i, int BN, int K) {
    const int nb = p / BN, r = p % BN, kb = i / 64;
    return (((size_t)nb * (K / 64) + kb) * BN + r) * 64 + (size_t)(i % 64);
}

// Byte offset of (row p, column i) of a [N][K] E4M3 operand stored as the
// tensor-core tile images of kind::f8f6f4: tiles of BN rows x 128 one-byte
// columns (one k block of 128), N-tile major then K-tile, each row 128 bytes with
// its 16-byte chunks permuted by chunk ^ (r % 8), the 128-byte swizzle.
__host__ __device__ inline size_t tiled_offset_f8(int p, int i, int BN, int K) {
    const int nb = p / BN, r = p % BN, kb = i / 128, ch = (i % 128) / 16, w = i % 16;
    return (((size_t)nb * (K / 128) + kb) * BN + r) * 128 + (size_t)((ch ^ (r & 7)) * 16 + w);
}

// Byte offsets inside the packed weight buffer.
//   w13 : [E][2f][d]      up-projection, K-major, W1/W3 interleaved in groups of kGroup rows
//   w2  : [E][d][f]       down-projection, K-major
//   w13s: [2*fs_tot][d]   shared experts merged along the hidden dimension
//   w2s : [d][fs_tot]
//   FP8 weights: the same matrices as E4M3 codes (one byte each), then fp32 scales
//   sc13: [E][2f] and sc2: [E][d] per output row of w13 / w2, sc13s: [2*fs_tot], sc2s: [d]
//   FP8 up projection: w13 / w13s as E4M3 codes (tiled_offset_f8), w2 / w2s bf16
//   tile images, scales sc13 and sc13s only
struct PackedLayout {
    size_t w13, w2, w13s, w2s, sc13, sc2, sc13s, sc2s, total;
};
PackedLayout packed_layout(const moe_config &c);

// ----------------------------------------------------------------------------- grouped segments
// Segment s < E is routed expert s (rows off[s]..off[s+1] of the expert-ordered
// buffer); segment E, when present, is the merged shared expert over all T tokens.
struct GroupedShape {
    const int32_t *off;   // device [E+1]
    int E;
    int shared_rows;      // T when shared experts exist, else 0
    int nblk_routed;      // N tiles per routed segment
    int nblk_shared;      // N tiles of the shared segment
};

// ----------------------------------------------------------------------------- launchers
cudaError_t launch_route_simt(const moe_config &c, const void *x, const void *W_r,
                              const float *logit_offset, const float *sel_bias, int32_t *topk_idx,
                              float *topk_w, float *scores_t, float *psum_rows, unsigned *err, cudaStream_t s);
cudaError_t launch_ec_select(const moe_config &c, const float *scores_t, int32_t *ec_tok, float *ec_w,
                             cudaStream_t s);
// per column e of scores_t[E][T]: the min(col_cnt[e], cap) largest (ties to the lower
// token), ascending token ids -> tok[e][0..), their scores -> w[e][0..)
cudaError_t launch_column_select(const moe_config &c, const float *scores_t, int cap, const int32_t *col_cnt,
                                 int32_t *tok, float *w, cudaStream_t s);
// Extra work of the dispatch gather in the forward of a layer whose down GEMM
// writes each kept token's output row itself (one expert per token, no shared
// experts): zero the output rows of the dropped tokens (slot_of[t] < 0) and the
// fused expert launch's dependency counters.  slot_of == nullptr: nothing extra.
struct GatherZero {
    const int32_t *slot_of = nullptr;   // [T] (k = 1)
    int64_t T = 0;
    uint4 *y = nullptr;                 // [T][d] in the activation type
    int y_vecs = 0;                     // 16-byte vectors of a row of y
    int *dep = nullptr;
    int ndep = 0;
};
// row_bytes: bytes of a row of x / x_perm (0: d times the activation size; the FP8
// up projection gathers one-byte E4M3 rows)
cudaError_t launch_dispatch_tc(const moe_config &c, int32_t cap, const int32_t *topk_idx, const void *x,
                               int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm,
                               int32_t *chunk_cnt, int32_t *row_token, unsigned *err, cudaStream_t s,
                               const GatherZero &zero = GatherZero{}, int row_bytes = 0);
size_t dispatch_tc_scratch_ints(int64_t assignments, int E);
// affinity-ordered capacity drop (token choice): scratch S[E][T] fp32, kept[E][cap]
// tokens and weights; launches a scatter, the column select, the row placement
// and the gather (slot_of and cnt_raw zeroed / set here)
cudaError_t launch_dispatch_affinity(const moe_config &c, int32_t cap, const int32_t *topk_idx, const float *topk_w,
                                     const void *x, int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm,
                                     float *S, int32_t *kept, float *kept_w, int32_t *row_token, unsigned *err,
                                     cudaStream_t s, const GatherZero &zero = GatherZero{}, int row_bytes = 0);
int dispatch_tc_launches(int64_t assignments);
cudaError_t launch_dispatch_ec(const moe_config &c, const int32_t *ec_tok, const void *x, int32_t *off,
                               int32_t *cnt_raw, int32_t *slot_of, void *x_perm, unsigned *err, cudaStream_t s,
                               int row_bytes = 0);
cudaError_t launch_combine(const moe_config &c, const Sizes &z, const void *Y, const int32_t *slot_of,
                           const float *w, void *y, cudaStream_t s);
cudaError_t launch_pack(const moe_config &c, const void *W1, const void *W3, const void *W2,
                        const void *W1s, const void *W3s, const void *W2s, void *packed, cudaStream_t s);
cudaError_t launch_ffn_up_simt(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                               const void *packed, const void *x, void *H, void *Hs, cudaStream_t s);
cudaError_t launch_ffn_down_simt(const moe_config &c, const Sizes &z, const void *H, const void *Hs,
                                 const int32_t *off, const void *packed, void *Y, cudaStream_t s);
// tcgen05 path (bf16)
cudaError_t launch_ffn_up_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                                  const void *packed, const void *x, void *H, void *Hs, unsigned *err,
                                  cudaStream_t s);
// With row_token/row_gate (token choice, k == 1, no shared experts) the combine is
// folded into the epilogue: Y is the layer output y[T][d] and row r is written to
// y[row_token[r]] scaled by row_gate[row_token[r]]; rows of dropped tokens are
// not written (the caller zeroes them: moe_forward's dispatch gather does).
cudaError_t launch_ffn_down_tcgen05(const moe_config &c, const Sizes &z, const void *H, const void *Hs,
                                    const int32_t *off, const void *packed, void *Y, unsigned *err, cudaStream_t s,
                                    const int32_t *row_token = nullptr, const float *row_gate = nullptr);
// Row scales of E4M3 activations (the FP8 up projection): routed row r has scale
// rs0[rtok0 ? rtok0[r] : r], shared-expert row t has rs1[t].
struct F8Rows {
    const float *rs0 = nullptr;
    const int32_t *rtok0 = nullptr;
    const float *rs1 = nullptr;
};
// Both expert GEMMs in one persistent (cooperative) launch: up tiles, then down tiles,
// each waiting for the up tiles of its rows through `dep` (ffn_dep_counters ints,
// zeroed here).  Needs 256-wide tiles for both (ffn_fused_supported).
cudaError_t launch_ffn_fused_tcgen05(const moe_config &c, const Sizes &z, const void *x_perm, const int32_t *off,
                                     const void *packed, const void *x, void *H, void *Hs, void *Y, int *dep,
                                     unsigned *err, cudaStream_t s, const int32_t *row_token = nullptr,
                                     const float *row_gate = nullptr, bool dep_zeroed = false,
                                     const F8Rows *f8 = nullptr);
size_t ffn_dep_counters(const moe_config &c);
bool ffn_fused_supported(const moe_config &c);
// psum_rows (nullable, [kPsumRows][E], zeroed by the caller): every CTA adds the
// sum over its tokens of each expert's score (softmax probability or sigmoid
// score) into row (CTA index mod kPsumRows), for the load statistics
cudaError_t launch_route_tcgen05(const moe_config &c, const void *x, const void *W_r,
                                 const float *logit_offset, const float *sel_bias, int32_t *topk_idx,
                                 float *topk_w, float *scores_t, float *psum_rows, void *wr_t, unsigned *err,
                                 cudaStream_t s);
// prob_sum[e] = sum over the kPsumRows rows of rows[r][e], in row order
cudaError_t launch_sum_psum_rows(const moe_config &c, const float *rows, float *prob_sum, cudaStream_t s);
// load statistics from the routing (one CTA); see moe_load_stats
cudaError_t launch_load_stats(const moe_config &c, const int32_t *topk_idx, const int32_t *cnt_raw,
                              const float *prob_sum, float *token_fraction, float *prob_mean, double *summary,
                              cudaStream_t s);
size_t route_tcgen05_scratch_bytes(const moe_config &c);
bool route_tcgen05_supported(const moe_config &c);
int route_tcgen05_launches(const moe_config &c);

int num_sms();
// architecture check and device error word of the current device (set up once per device)
moe_status device_ready(unsigned **err_word);
// limit of the bounded device-side waits (process-wide; moe_set_wait_limit_ns)
uint64_t wait_limit_ns();
// share of L2 that one group of the expert GEMMs' tile order fills with A rows
// (down = 0: x_perm rows of the up projection, 1: H rows of the down projection)
uint64_t tile_group_bytes(int down);
// Per-row E4M3 quantisation of bf16 rows: s[r] = amax_r / 448, q[r][i] = E4M3(x / s[r])
// (fp32 division, round to nearest even, saturated; an all-zero row gets s = 0 and
// zero codes).  rows x d, one warp per row.
cudaError_t launch_quantize_rows(const void *x, int64_t rows, int d, uint8_t *q, float *s, cudaStream_t st);
// one CTA that runs the two bounded-wait routines of the tensor-core kernels (see
// moe_wait_probe); sets kErrWaitTimeout in *err when they give up
cudaError_t launch_wait_probe(const int32_t *flag, int32_t target, uint64_t limit_ns, unsigned *err, cudaStream_t s);

// ----------------------------------------------------------------------------- dependent launches
// The hot kernels (tensor-core GEMMs, split-K select, dispatch plan, gather,
// combine) are launched with programmatic stream serialisation: such a grid may
// start while its predecessor on the stream -- ours or the caller's -- is still
// running, once every CTA of the predecessor has executed pdl_trigger() (or
// exited).  Each of these kernels calls pdl_wait() -- which returns when the
// predecessor grid has completed and its memory writes are visible -- before its
// first access to global memory; only shared-memory and TMEM setup come earlier.
// Without the launch attribute both instructions do nothing.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch with programmatic stream serialisation (and optionally as a cooperative
// launch).  The kernel must follow the pdl_wait() rule above.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             bool cooperative, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// A dependent launch (as above) of thread-block clusters of `cluster` CTAs along x
// (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     int cluster, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ----------------------------------------------------------------------------- device helpers
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Lanes of the warp holding the same 9-bit key (key < 512), from nine ballots:
// a lane matches when it agrees on every bit.  Cheaper than __match_any_sync
// when a warp holds many distinct keys.
__device__ __forceinline__ unsigned warp_peers9(unsigned key) {
    unsigned peers = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 9; ++b) {
        const bool bit = (key >> b) & 1u;
        const unsigned vote = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? vote : ~vote;
    }
    return peers;
}

// Tile table of a grouped problem, built once per CTA in shared memory:
// tile_start[s] = first tile of segment s (tile_start[S] = total tiles).
// The order of a segment's tiles is decode_tile's: N-block-major with the M block
// fastest, or the same inside groups of M blocks (and chunks of N blocks), so that
// the CTAs sharing a weight tile run at the same time.
template <int BM>
__device__ __forceinline__ int build_tile_table(const GroupedShape &g, int *tile_start, int *seg_row0,
                                                int *seg_rows) {
    const int S = g.E + (g.shared_rows > 0 ? 1 : 0);
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        int r0, n;
        if (s < g.E) {
            r0 = g.off[s];
            n = g.off[s + 1] - r0;
        } else {
            r0 = 0;
            n = g.shared_rows;
        }
        seg_row0[s] = r0;
        seg_rows[s] = n;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int s = 0; s < S; ++s) {
            tile_start[s] = acc;
            const int nb = (s < g.E) ? g.nblk_routed : g.nblk_shared;
            acc += ((seg_rows[s] + BM - 1) / BM) * nb;
        }
        tile_start[S] = acc;
    }
    __syncthreads();
    return S;
}

// group_m > 0: the M blocks of a segment are split into ceil(mblk / group_m) groups
// of nearly equal size (the first mblk mod #groups are one block larger), and a
// group's tiles (every N block of it, M fastest) all come before the next group's.
// group_m = 0: the segment's tiles M fastest.
template <int BM>
__device__ __forceinline__ void decode_tile(const GroupedShape &g, const int *tile_start, const int *seg_rows,
                                            int S, int tile, int &s, int &mb, int &nb, int group_m = 0) {
    int lo = 0, hi = S - 1;   // last s with tile_start[s] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    s = lo;
    const int local = tile - tile_start[s];
    const int mblk = (seg_rows[s] + BM - 1) / BM;
    if (group_m > 0 && mblk > group_m) {
        const int nblk = (s < g.E) ? g.nblk_routed : g.nblk_shared;
        const int ng = (mblk + group_m - 1) / group_m;
        const int base = mblk / ng, big = mblk - base * ng;   // big groups of base + 1 blocks first
        const int big_tiles = big * (base + 1) * nblk;
        int gm, m0, rem;
        if (local < big_tiles) {
            gm = base + 1;
            const int grp = local / (gm * nblk);
            rem = local - grp * gm * nblk;
            m0 = grp * gm;
        } else {
            gm = base;
            const int l2 = local - big_tiles, grp = l2 / (gm * nblk);
            rem = l2 - grp * gm * nblk;
            m0 = big * (base + 1) + grp * gm;
        }
        mb = m0 + rem % gm;
        nb = rem / gm;
    } else {
        mb = local % mblk;
        nb = local / mblk;
    }
}

}  // namespace moe
