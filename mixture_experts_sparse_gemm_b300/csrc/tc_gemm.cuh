// Persistent grouped GEMM on the 5th-generation tensor cores (bf16 in, fp32
// accumulate in TMEM), shared by the expert GEMMs and the router.
//
// One CTA per SM, 6 warps (15 with FP8 weights):
//   warp 0      TMA producer: 128x64 A tile + BNx64 B tile per stage, 128-byte
//               swizzle, into a STAGES-deep shared-memory ring (full/empty mbarriers)
//   warp 1      TMEM allocator and MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16)
//               per stage into one of two TMEM accumulators; an expert tile of at
//               most 64 rows uses M=64 (its rows 16 q + i land in TMEM lanes 32 q + i)
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (one row per
//               thread), then the epilogue of the instantiation; it overlaps the
//               next tile's main loop through the second accumulator
//   warps 6..13 (W8 only) converters: an FP8 weight tile of the FP8 ring -> one
//               of two bf16 B buffers, which the MMA reads; the per-column weight
//               scales are applied in the epilogue
//   warp 14     (W8 only) FP8 producer: the weight tiles into their own ring,
//               ahead of the MMA (warp 0 then brings only A, into its own ring)
//   warps 6..15 (split-K router only) selection warps, idle until the tile's
//               partial logits are reduced across the cluster
// F8A instantiations run the tiles of a GEMM marked a_f8 (the up projection) on
// E4M3 operands: kind::f8f6f4 MMAs of K = 32, a k block of 128 one-byte elements
// (the same 128-byte swizzled rows as a bf16 block of 64), and the epilogue scales
// the accumulator by the row's activation scale and the column's weight scale.
// Tiles never straddle segments: the tile table is built on the device from
// off[] (segment s < E = routed expert s, segment E = merged shared experts), and
// a segment's last M tile reads rows past its end (the next segment's rows, or
// zero fill beyond the tensor) whose results are never stored.
//
// Epilogues:
//   kEpiSwiGLU  up projection.  The packed B rows of a tile alternate 64 W1
//               columns and the same 64 W3 columns, so a thread holds gate and up
//               values of the same hidden columns: H = SiLU(gate) * up, bf16.
//   kEpiStore   down projection: bf16 rows of Y.
//   kEpiRoute   router: one row = one token's E logits.  Softmax or sigmoid score,
//               selection-only bias, top-k by insertion in ascending expert order
//               (ties keep the lower index), renormalised weights; or, for Expert
//               Choice, the softmax scores written expert-major.
//   kEpiSplitRoute  router with K split over a cluster: partial logits to shared
//               memory, summed across the cluster's CTAs and selected one warp per
//               token (split_route_select).
#pragma once

#include <cuda_fp16.h>
#include <float.h>

#include "route_common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kBM = 128;
constexpr int kBK = 64;
// Expert GEMM tile order (the ~148 tiles in flight share their operands through L2):
// a segment's M tiles in groups of nearly equal size, at most TcGemm::group_m each,
// every N block of a group (M fastest) before the next group.  A group's A rows
// stay in L2 while its N blocks stream the weights once; the host sizes group_m so
// that a group's A rows fill a set share of L2 (x_perm rows of the up projection,
// H rows of the down projection).
constexpr int kThreads = 192;
constexpr int kEpiSwiGLU = 0;   // up projection (+ SwiGLU)
constexpr int kEpiStore = 1;    // down projection (optionally gated, see TcArgs::gated)
constexpr int kEpiFfn = 2;      // both: up tiles, then down tiles, in one persistent launch
constexpr int kEpiPartial = 3;  // router kinds start here (kEpiRoute.., kEpiSplitRoute..)
// router epilogue keeping the best KMAX candidates: kEpiRoute + KMAX, KMAX in {1, 2, 4, 8}
constexpr int kEpiRoute = 10;
// split-K router reduced inside a thread-block cluster: kEpiSplitRoute + KPL, KPL =
// experts per lane of the selecting warps (E <= 32 KPL).  The cluster is the K
// splits of one token tile: each CTA leaves its partial logits in shared memory,
// and after a cluster barrier CTA q sums the partials of its share of the tile's
// tokens from every CTA's shared memory (in split order) and scores and selects
// them one warp per token.  No partial logits go through global memory.
constexpr int kEpiSplitRoute = 20;
constexpr int kSplitSelectWarps = 10;   // extra warps of a split-K router CTA (16 select in all)

// W8: B arrives as FP8 E4M3 tiles (BN x 64 bytes) in a ring of its own (6 slots),
// brought by an FP8 producer warp and released by eight converter warps as soon as
// they have expanded a tile into one of two bf16 B buffers, which the MMA reads
// and releases.  A has its own ring (3 stages).  The weights thus run up to eight
// k blocks ahead of the MMA, as many weight bytes in flight as the bf16 kernel has.
// Shared memory: stages (bf16: A | B; W8: A) | W8: bf16 B buffers | W8: FP8 slots.
// EXTRA: warps beyond the GEMM roles (the cluster-reduced split-K router adds
// kSplitSelectWarps that only take part in its selection phase).
template <int BN, bool W8 = false, int EXTRA = 0>
struct TcCfg {
    static constexpr int kABytes = kBM * kBK * 2;
    static constexpr int kBBytes = BN * kBK * 2;      // bf16 B tile, as the MMA reads it
    static constexpr int kB8Bytes = BN * kBK;         // FP8 B tile, as the copy brings it (W8)
    static constexpr int kStageBytes = kABytes + (W8 ? 0 : kBBytes);
    static constexpr int kStages = W8 ? 3 : ((BN == 256) ? 4 : (BN == 128 ? 6 : 8));
    static constexpr int kBBufs = W8 ? 3 : 0;         // bf16 B buffers (W8)
    static constexpr int kB8Stages = W8 ? 4 : 0;      // FP8 ring slots
    static constexpr int kConvWarps = W8 ? 12 : 0;
    static constexpr int kB8Warp = kThreads / 32 + kConvWarps;   // W8: warp of the FP8 copies
    static constexpr int kThreadsCta = kThreads + 32 * kConvWarps + (W8 ? 32 : 0) + 32 * EXTRA;
    static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
    static constexpr int kBarBytes = (2 * kStages + 5 + 2 * kBBufs + 2 * kB8Stages) * 8;
    static constexpr int kMiscBytes = 64 + sizeof(int) * (8 * (kMaxE + 2));
    static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + (size_t)kBBufs * kBBytes +
                                    (size_t)kB8Stages * kB8Bytes + kBarBytes + kMiscBytes;
};

struct RouteEpi {
    const float *logit_offset;   // [E] or null
    const float *sel_bias;       // [E] or null
    int32_t *topk_idx;           // [T][k]
    float *topk_w;               // [T][k]
    float *scores_t;             // expert choice: [E][T]
    float *psum_rows;            // [kPsumRows][E] or null: += each CTA's sums of the experts' scores
    int T, E, k, gate, mode, renorm;
};

// One grouped GEMM over the segments: segment s < E is routed expert s (rows
// off[s]..off[s+1] of A and C), segment E (shared_rows > 0) the merged shared experts.
struct TcGemm {
    GroupedShape g;
    int K0, K1;        // reduction width, routed / shared
    int b_rows0;       // B rows per routed segment (tensor-map B)
    // B as tensor-core tile images (tiled_offset layout), one bulk copy per stage;
    // null: B comes through the tensor maps tmB0 / tmB1 instead
    const uint8_t *Bt0;   // routed segments, bt_seg0 bytes each
    const uint8_t *Bt1;   // shared segment
    size_t bt_seg0;
    int img_rows;         // rows of one packed tile image (BN or a multiple: a BN tile is a slice of it)
    void *C0;             // routed output rows (bf16)
    void *C1;             // shared output rows (bf16)
    int ldc0, ldc1;       // output row pitch in elements
    // > 1: the K range is split over ksplit tiles (the N-block index is the split;
    // one N tile of width BN covers all of N; cluster-reduced router only)
    int ksplit;
    // FP8 weights (W8 kernels): fp32 scale of every B row (output column), routed
    // [E][b_rows0] and shared [N]; applied to the accumulator in the epilogue
    const float *sc0, *sc1;
    // B given MN-major through tmB0 / tmB1: a row-major [K][N] matrix read in place,
    // each stage BN / 64 boxes of [64 K rows][64 N] (BN >= 64; router launches only)
    int b_mn;
    // E4M3 A and B (kernels instantiated with F8A): kind::f8f6f4, 128 K per stage;
    // the accumulator is scaled by the row scale of A and the column scale of B
    // (sc0 / sc1).  Row r of a routed segment has scale rs0[rtok0 ? rtok0[r] : r],
    // row r of the shared segment rs1[r].
    int a_f8;
    const float *rs0;
    const int32_t *rtok0;
    const float *rs1;
    // expert GEMMs: M tiles per group of the tile order (0: M fastest over the whole
    // segment; the router keeps 0, its tile order is its K split layout)
    int group_m;
};

struct TcArgs {
    TcGemm p[2];          // p[1]: the down projection of a kEpiFfn launch
    // kEpiFfn: dep[mtile_start(s) + mb] counts the finished up tiles of (segment, M
    // tile); a down tile waits until all of them are done (zeroed before the launch)
    int *dep;
    // down projection with the combine of one expert per token folded in: routed row
    // r is token t = row_token[r] and goes to C0[t] scaled by row_gate[t]
    int gated;
    const int32_t *row_token;
    const float *row_gate;
    RouteEpi route;
    unsigned *err;
    uint64_t wait_ns;     // limit of every bounded wait (set by launch_gemm)
};

// SiLU(z) = z / (1 + e^-z) with the fast exponential and division (the result is
// rounded to bf16 right after; for z < -88 the denominator is inf and SiLU -> -0)
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// ---------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// all threads of every CTA of the cluster; shared-memory writes before it are
// visible to the other CTAs' reads after it
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Keep the best KMAX (key, index, logit) triples in (key desc, index asc) order.
// Candidates arrive in ascending index order and only a strictly larger key
// moves up, so a tie keeps the lower index first.
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tk)[KMAX], int (&ti)[KMAX], float (&tu)[KMAX], float key, int e,
                                            float u) {
    if (key > tk[KMAX - 1]) {
        tk[KMAX - 1] = key;
        ti[KMAX - 1] = e;
        tu[KMAX - 1] = u;
#pragma unroll
        for (int j = KMAX - 1; j > 0; --j) {
            if (tk[j] > tk[j - 1]) {
                const float a = tk[j], b = tu[j];
                const int q = ti[j];
                tk[j] = tk[j - 1];
                tu[j] = tu[j - 1];
                ti[j] = ti[j - 1];
                tk[j - 1] = a;
                tu[j - 1] = b;
                ti[j - 1] = q;
            }
        }
    }
}

// Router epilogue of one token row (all 32 lanes of the warp take part in the
// TMEM loads; `valid` says whether this lane's row is a token).
//   pass 1: u_e = logit + offset.  Softmax: running max, and the top k on u_e
//           itself -- softmax is increasing in the logit, so its order, ties
//           included, is the order of the scores, and fp32 logits resolve it
//           more finely than fp32 scores would.  Sigmoid: key = score + bias.
//   pass 2: softmax normaliser sum_e exp(u_e - max).
//   then the k weights (renormalised when asked), or for Expert Choice every
//   score written expert-major.
// loff / bias: the E logit offsets and selection biases in shared memory (zeros
// where the caller gave none), read from there in every pass.
template <int BN, int KMAX>
__device__ __forceinline__ void route_epilogue(const RouteEpi &r, uint32_t taddr, int t, bool valid,
                                               float *psum_cta, const float *loff, const float *bias) {
    const int E = r.E, T = r.T;
    constexpr int kChunks = BN / 16;
    const bool softmax = r.gate == MOE_GATE_SOFTMAX;
    const bool ec = r.mode == MOE_EXPERT_CHOICE;
    float tk[KMAX], tu[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        tk[j] = -FLT_MAX;
        tu[j] = 0.f;
        ti[j] = 0x7fffffff;
    }
    float mx = -FLT_MAX;
#pragma unroll 1
    for (int c = 0; c < kChunks; ++c) {
        uint32_t v[16];
        tmem_ld16(taddr + c * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int e = c * 16 + i;
            if (e < E) {
                const float u = __uint_as_float(v[i]) + loff[e];
                if (softmax) {
                    mx = fmaxf(mx, u);
                    if (!ec) topk_insert<KMAX>(tk, ti, tu, u, e, u);
                } else {
                    const float s = __fdividef(1.f, 1.f + __expf(-u));
                    topk_insert<KMAX>(tk, ti, tu, s + bias[e], e, u);
                }
            }
        }
    }
    float inv = 1.f;
    if (softmax) {
        float sum = 0.f;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
            uint32_t v[16];
            tmem_ld16(taddr + c * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = c * 16 + i;
                if (e < E) sum += __expf(__uint_as_float(v[i]) + loff[e] - mx);
            }
        }
        inv = 1.f / sum;
    }
    if (r.psum_rows) {
        // every expert's score summed over the warp's 32 token rows into the CTA's
        // shared sums (added to its row of psum_rows once per CTA at the end of the kernel)
        const int lane = threadIdx.x & 31;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
            uint32_t v[16];
            tmem_ld16(taddr + c * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = c * 16 + i;
                float pe = 0.f;
                if (e < E && valid) {
                    const float u = __uint_as_float(v[i]) + loff[e];
                    pe = softmax ? __expf(u - mx) * inv : __fdividef(1.f, 1.f + __expf(-u));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) pe += __shfl_xor_sync(0xffffffffu, pe, o);
                if (lane == 0 && e < E) atomicAdd(psum_cta + e, pe);
            }
        }
    }
    if (ec) {
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
            uint32_t v[16];
            tmem_ld16(taddr + c * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = c * 16 + i;
                if (e < E && valid)
                    r.scores_t[(size_t)e * T + t] =
                        __expf(__uint_as_float(v[i]) + loff[e] - mx) * inv;
            }
        }
        return;
    }
    if (!valid) return;
    const int k = r.k;
    if (ti[k - 1] == 0x7fffffff) {
        // fewer than k keys compared above -FLT_MAX (NaN scores from non-finite
        // inputs): fill the empty slots with the lowest experts not chosen, so every
        // index stays in range
        int e = 0;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < k && ti[j] == 0x7fffffff) {
                for (;; ++e) {
                    bool used = false;
#pragma unroll
                    for (int q = 0; q < KMAX; ++q) used |= (q < k && ti[q] == e);
                    if (!used) break;
                }
                ti[j] = e;
                tu[j] = 0.f;
            }
        }
    }
    float p[KMAX], wsum = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        p[j] = softmax ? __expf(tu[j] - mx) * inv : __fdividef(1.f, 1.f + __expf(-tu[j]));
        if (j < k) wsum += p[j];
    }
    const float scale = r.renorm ? 1.f / wsum : 1.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
            r.topk_idx[(size_t)t * k + j] = ti[j];
            r.topk_w[(size_t)t * k + j] = p[j] * scale;
        }
    }
}

// KPL consecutive floats of another CTA's shared memory (16-byte loads where they fit)
template <int KPL>
__device__ __forceinline__ void ld_dsmem_vec(uint32_t addr, float (&v)[KPL]) {
    if constexpr (KPL % 4 == 0) {
#pragma unroll
        for (int q = 0; q < KPL; q += 4)
            asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v[q]), "=f"(v[q + 1]), "=f"(v[q + 2]), "=f"(v[q + 3])
                         : "r"(addr + 4u * q)
                         : "memory");
    } else if constexpr (KPL == 2) {
        asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v[0]), "=f"(v[1]) : "r"(addr) : "memory");
    } else {
        v[0] = ld_dsmem(addr);
    }
}

// Selection of a cluster-reduced split-K router tile, run by every thread of each
// CTA of the cluster after the cluster barrier.  Every CTA holds its partial
// logits of the tile's rows at red + row * pitch floats; CTA q takes the rows
// [q * ceil(128 / splits), ...) of the tile, and one warp per row sums the
// partials of all CTAs of the cluster in split order (reading the others' shared
// memory; lane l holds experts l * KPL ..), adds the logit offset, and scores and
// selects it (warp_score_select).
template <int KPL>
__device__ __forceinline__ void split_route_select(const RouteEpi &r, const uint8_t *red, int pitch, int splits,
                                                   int T, int mb, float *sacc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int rank = (int)cluster_ctarank();
    const int row0 = mb * kBM;
    const int rows = min(kBM, T - row0);
    const int per = (kBM + splits - 1) / splits;
    const int lo = rank * per, hi = min(rows, lo + per);
    RouteArgs a{};
    a.logit_offset = r.logit_offset;
    a.sel_bias = r.sel_bias;
    a.T = r.T;
    a.E = r.E;
    a.k = r.k;
    a.gate = r.gate;
    a.mode = r.mode;
    a.renorm = r.renorm;
    a.topk_idx = r.topk_idx;
    a.topk_w = r.topk_w;
    a.scores_t = r.scores_t;
    a.psum_rows = r.psum_rows;
    const uint32_t base = smem_u32(red);
    float pacc[KPL], bias[KPL];   // the lane's experts are the same in every row: biases once
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        pacc[i] = 0.f;
        const int e = lane * KPL + i;
        bias[i] = (e < a.E && a.sel_bias) ? a.sel_bias[e] : 0.f;
    }
    for (int rr = lo + warp; rr < hi; rr += nwarps) {
        // every split's values of the row are loaded before the sums (split order kept)
        float pv[kMaxRouteSplits][KPL];
        const uint32_t off = base + (uint32_t)((rr * pitch + lane * KPL) * 4);
#pragma unroll
        for (int q = 0; q < kMaxRouteSplits; ++q)
            if (q < splits) ld_dsmem_vec<KPL>(mapa_shared(off, (uint32_t)q), pv[q]);
        float u[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int e = lane * KPL + i;
            float v = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxRouteSplits; ++q)
                if (q < splits) v += pv[q][i];
            if (e < a.E && a.logit_offset) v += a.logit_offset[e];
            u[i] = (e < a.E) ? v : -FLT_MAX;
        }
        warp_score_select<KPL, true>(a, u, row0 + rr, lane, pacc, bias);
    }
    flush_prob_sum<KPL, true>(a, pacc, lane, sacc);
}

// Tile epilogues (all 32 lanes of each epilogue warp run them; `row` is the
// thread's accumulator row, `rows` the valid rows of the tile).
// sc (FP8 weights, else null): scales of the tile's BN accumulator columns
// rs: scale of the thread's row (E4M3 activations), 1 otherwise
__device__ __forceinline__ void scale16(uint32_t (&v)[16], const float *sc, float rs = 1.f) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = *reinterpret_cast<const float4 *>(sc + 4 * q);
        v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) * (f.x * rs));
        v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) * (f.y * rs));
        v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) * (f.z * rs));
        v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) * (f.w * rs));
    }
}

template <int BN>
__device__ __forceinline__ void epi_swiglu(uint32_t taddr, __nv_bfloat16 *Cp, int ldc, int grow, int row, int rows,
                                           int nb, const float *sc, float rs = 1.f) {
#pragma unroll 1
    for (int grp = 0; grp < BN / 128; ++grp) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t g[16], u[16];
            tmem_ld16(taddr + grp * 128 + c * 16, g);
            tmem_ld16(taddr + grp * 128 + 64 + c * 16, u);
            tmem_ld_wait();
            if (sc) {
                scale16(g, sc + grp * 128 + c * 16, rs);
                scale16(u, sc + grp * 128 + 64 + c * 16, rs);
            }
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                o[i] = pack_bf16x2(h0, h1);
            }
            if (row < rows) {
                uint4 *dst = reinterpret_cast<uint4 *>(Cp + (size_t)grow * ldc + nb * (BN / 2) + grp * 64 + c * 16);
                dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            }
        }
    }
}

template <int BN>
__device__ __forceinline__ void epi_store(uint32_t taddr, __nv_bfloat16 *Cp, int ldc, size_t orow, float scale, int row,
                                          int rows, int nb, const float *sc) {
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(taddr + c * 16, v);
        tmem_ld_wait();
        if (sc) scale16(v, sc + c * 16);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * scale, __uint_as_float(v[2 * i + 1]) * scale);
        if (row < rows) {
            uint4 *dst = reinterpret_cast<uint4 *>(Cp + orow * ldc + nb * BN + c * 16);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
    }
}

// 16 E4M3 codes -> 16 bf16, exactly (every E4M3 value is a bf16 value), without
// conversion instructions: a code s.eeee.mmm is placed as the bf16 bit pattern
// s.0000eeee.mmm0000 -- the value 2^(e-127) (1 + m/8), or for e = 0 the bf16
// subnormal (m/8) 2^-126 -- and one exact bf16 multiply by 2^120 moves the
// exponent bias from 127 to 7: 2^(e-7) (1 + m/8), resp. (m/8) 2^-6, the E4M3 value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t x) {   // x = 0x00bb00aa
    const uint32_t bits = ((x << 4) & 0x07F007F0u) | ((x << 8) & 0x80008000u);
    const uint32_t two120 = 0x7B807B80u;   // bf16 2^120, twice
    const __nv_bfloat162 r = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&bits),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&two120));
    return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 &v, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // bytes 0,1 and 2,3 of the word into the low byte of each 16-bit half
        o[2 * i] = e4m3x2_to_bf16x2(__byte_perm(w[i], 0u, 0x4140));
        o[2 * i + 1] = e4m3x2_to_bf16x2(__byte_perm(w[i], 0u, 0x4342));
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Where a tile lives: phase (GEMM of a kEpiFfn launch), segment, M and N block.
struct TileAt {
    int phase, s, mb, nb;
};

template <int BN, int EPI, bool W8, bool F8A = false>
__global__ void __launch_bounds__(TcCfg<BN, W8, (EPI > kEpiSplitRoute) ? kSplitSelectWarps : 0>::kThreadsCta, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                           const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                           const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA3,
                           TcArgs a) {
    using C = TcCfg<BN, W8, (EPI > kEpiSplitRoute) ? kSplitSelectWarps : 0>;
    constexpr int kPhases = (EPI == kEpiFfn) ? 2 : 1;
    constexpr bool kRouter = EPI >= kEpiPartial;   // router launches may read B (W_r) MN-major
    constexpr bool kFusedRoute = EPI > kEpiRoute && EPI < kEpiSplitRoute;
    constexpr bool kSplitRoute = EPI > kEpiSplitRoute;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *tiles = smem;
    uint8_t *bbuf = tiles + (size_t)C::kStages * C::kStageBytes;   // W8: bf16 B buffers
    uint8_t *b8ring = bbuf + (size_t)C::kBBufs * C::kBBytes;        // W8: FP8 B slots
    uint64_t *bars = reinterpret_cast<uint64_t *>(b8ring + (size_t)C::kB8Stages * C::kB8Bytes);
    uint64_t *full = bars;
    uint64_t *empty = bars + C::kStages;
    uint64_t *tfull = bars + 2 * C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *conv = drain + 1;                 // W8: bf16 B buffer written and fenced (converter warps)
    uint64_t *bempty = conv + C::kBBufs;        // W8: bf16 B buffer read by the MMA
    uint64_t *f8full = bempty + C::kBBufs;      // W8: FP8 slot landed
    uint64_t *f8empty = f8full + C::kB8Stages;  // W8: FP8 slot expanded by all converter warps
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(f8empty + C::kB8Stages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int *tile_start0 = reinterpret_cast<int *>(tmem_holder + 16);   // tiles of phase 0 per segment
    int *tile_start1 = tile_start0 + (kMaxE + 2);                   // tiles of phase 1 per segment
    int *seg_row0 = tile_start1 + (kMaxE + 2);
    int *seg_rows = seg_row0 + (kMaxE + 2);
    int *mtile_start = seg_rows + (kMaxE + 2);                      // first M tile of each segment
    float *psum_cta = reinterpret_cast<float *>(mtile_start + (kMaxE + 2));   // router score sums of this CTA
    float *s_loff = psum_cta + (kMaxE + 2);   // fused router: logit offsets (0 without), staged once
    float *s_bias = s_loff + (kMaxE + 2);     // fused router: selection biases (0 without)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (kFusedRoute) {
        for (int e = threadIdx.x; e < kMaxE; e += C::kThreadsCta) psum_cta[e] = 0.f;   // before the first barrier
    }

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
        if (W8) {
            for (int b = 0; b < C::kBBufs; ++b) {
                mbar_init(smem_u32(&conv[b]), C::kConvWarps);
                mbar_init(smem_u32(&bempty[b]), 1);
            }
            for (int f = 0; f < C::kB8Stages; ++f) {
                mbar_init(smem_u32(&f8full[f]), 1);
                mbar_init(smem_u32(&f8empty[f]), C::kConvWarps);
            }
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tmap(&tmA0);
        prefetch_tmap(&tmA1);
        if (a.p[0].Bt0 == nullptr) {
            prefetch_tmap(&tmB0);
            prefetch_tmap(&tmB1);
        }
        if (kPhases == 2) {
            prefetch_tmap(&tmA2);
            prefetch_tmap(&tmA3);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
        fence_before();
    }
    __syncthreads();
    fence_after();
    pdl_wait();      // the previous kernel's outputs (segment offsets, A rows) are visible from here on
    pdl_trigger();
    if constexpr (kFusedRoute) {   // made visible to the epilogue by the barrier in build_tile_table
        for (int e = threadIdx.x; e < a.route.E; e += C::kThreadsCta) {
            s_loff[e] = a.route.logit_offset ? a.route.logit_offset[e] : 0.f;
            s_bias[e] = a.route.sel_bias ? a.route.sel_bias[e] : 0.f;
        }
    }
    const uint32_t tmem_base = *tmem_holder;
    const int S = build_tile_table<kBM>(a.p[0].g, tile_start0, seg_row0, seg_rows);
    const int total0 = tile_start0[S];
    int total = total0;
    if (kPhases == 2) {
        if (threadIdx.x == 0) {
            int t1 = 0, m = 0;
            for (int s = 0; s < S; ++s) {
                const int mblk = (seg_rows[s] + kBM - 1) / kBM;
                tile_start1[s] = t1;
                mtile_start[s] = m;
                t1 += mblk * ((s < a.p[1].g.E) ? a.p[1].g.nblk_routed : a.p[1].g.nblk_shared);
                m += mblk;
            }
            tile_start1[S] = t1;
            mtile_start[S] = m;
        }
        __syncthreads();
        total += tile_start1[S];
    }
    // Tiles of this CTA: tile0, tile0 + tstep, ...  A cluster-reduced split-K router
    // launch has one CTA per tile, and the CTAs of a cluster (consecutive blocks)
    // take the K splits of one token tile: split = rank, M block = block / splits.
    const int mblk0 = (seg_rows[0] + kBM - 1) / kBM;
    int tile0 = blockIdx.x, tstep = gridDim.x;
    if constexpr (kSplitRoute) {
        const int splits = a.p[0].ksplit;
        tile0 = (int)(blockIdx.x % splits) * mblk0 + (int)(blockIdx.x / splits);
        tstep = total;
    }
    static_assert(!(W8 && F8A), "FP8 weights go through the converters or straight to the MMA, not both");
    // E4M3 operands: a k block holds 128 K (128 bytes per row, as the bf16 block's 64)
    auto tile_f8 = [&](const TileAt &t) { return F8A && a.p[t.phase].a_f8 != 0; };
    // k blocks [kb0, kb0 + nk) of a tile (a K split takes its share of them)
    auto krange = [&](const TileAt &t, const TcGemm &G, int &kb0, int &nk) {
        const int all = ((t.s < G.g.E) ? G.K0 : G.K1) / (tile_f8(t) ? 128 : kBK);
        if (G.ksplit > 1) {
            const int per = (all + G.ksplit - 1) / G.ksplit;
            kb0 = t.nb * per;
            nk = min(all, kb0 + per) - kb0;
        } else {
            kb0 = 0;
            nk = all;
        }
    };
    auto locate = [&](int tile) {
        TileAt t;
        if (kPhases == 2 && tile >= total0) {
            t.phase = 1;
            decode_tile<kBM>(a.p[1].g, tile_start1, seg_rows, S, tile - total0, t.s, t.mb, t.nb, a.p[1].group_m);
        } else {
            t.phase = 0;
            decode_tile<kBM>(a.p[0].g, tile_start0, seg_rows, S, tile, t.s, t.mb, t.nb, a.p[0].group_m);
        }
        return t;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = tile0; tile < total && ok; tile += tstep) {
                const TileAt t = locate(tile);
                const TcGemm &G = a.p[t.phase];
                const bool routed = t.s < G.g.E;
                if (kPhases == 2 && t.phase == 1) {
                    // H rows of this (segment, M tile) come from the up tiles: wait until all
                    // of them have published (release/acquire through dep), bounded
                    const int need = routed ? a.p[0].g.nblk_routed : a.p[0].g.nblk_shared;
                    if (!wait_counter_bounded(a.dep + mtile_start[t.s] + t.mb, need, abort_flag, a.err, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");   // generic writes -> TMA reads
                }
                const CUtensorMap *mA = (t.phase == 0) ? (routed ? &tmA0 : &tmA1) : (routed ? &tmA2 : &tmA3);
                const CUtensorMap *mB = routed ? &tmB0 : &tmB1;
                const int arow = seg_row0[t.s] + t.mb * kBM;
                const int brow = (routed ? t.s * G.b_rows0 : 0) + (G.ksplit > 1 ? 0 : t.nb * BN);
                int kb0, nk;
                krange(t, G, kb0, nk);
                const uint8_t *bt = nullptr;
                size_t img_bytes = 0;
                constexpr int kBCopy = W8 ? C::kB8Bytes : C::kBBytes;   // B bytes per stage
                if (G.Bt0) {
                    // rows [nb*BN, nb*BN + BN) of the N dimension are slice `sub` of image `img`;
                    // image rows are stored consecutively, so a slice is contiguous too
                    const int per = G.img_rows / BN, img = t.nb / per, sub = t.nb % per;
                    img_bytes = (size_t)G.img_rows * kBK * (W8 ? 1 : 2);
                    bt = (routed ? G.Bt0 + (size_t)t.s * G.bt_seg0 : G.Bt1) + (size_t)img * nk * img_bytes +
                         (size_t)sub * kBCopy;
                }
                // router tiles read their token rows once, all CTAs at the same time: each
                // starts at its own k block, so that concurrent requests fall on different
                // column offsets of rows whose stride is a power of two (spread over the
                // DRAM channels); the MMA sums the k blocks in this rotated order
                const int rot = kRouter ? (int)((tile * 5) % nk) : 0;
                for (int kb_ = 0; kb_ < nk; ++kb_) {
                    const int kb = (kb_ + rot) % nk;
                    if (!wait_bounded(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, a.err, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    uint8_t *st = tiles + (size_t)stage * C::kStageBytes;
                    mbar_arrive_expect_tx(fb, C::kABytes + (W8 ? 0 : kBCopy));   // A + B (W8: A only)
                    tma_load_2d(smem_u32(st), mA, (kb0 + kb) * (tile_f8(t) ? 128 : kBK), arow, fb);
                    if (W8)
                        ;   // the FP8 B tiles come through their own ring (B8 producer warp)
                    else if (bt)
                        bulk_load(smem_u32(st + C::kABytes), bt + (size_t)(kb0 + kb) * img_bytes, kBCopy, fb);
                    else if (kRouter && BN >= 64 && G.b_mn)
                        for (int j = 0; j < BN / 64; ++j)   // 64-wide N chunks, 8 KB apart
                            tma_load_2d(smem_u32(st + C::kABytes + j * 8192), mB,
                                        (G.ksplit > 1 ? 0 : t.nb * BN) + 64 * j, (kb0 + kb) * kBK, fb);
                    else
                        tma_load_2d(smem_u32(st + C::kABytes), mB, (kb0 + kb) * kBK, brow, fb);
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
                    while (!mbar_try_wait(fb, ph) && globaltimer() - t0 < kDrainLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
            constexpr uint32_t kIdescF8 = idesc_e4m3_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int bb = 0;           // W8: bf16 B buffer
            uint32_t bph = 0;
            int it = 0;
            bool ok = true;
            for (int tile = tile0; tile < total && ok; tile += tstep, ++it) {
                const TileAt t = locate(tile);
                const TcGemm &G = a.p[t.phase];
                int kb0, nk;
                krange(t, G, kb0, nk);
                const bool f8 = tile_f8(t);
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, a.err, a.wait_ns)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(smem_u32(&full[stage]), phase, abort_flag, a.err, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if constexpr (W8) {
                        if (!wait_bounded(smem_u32(&conv[bb]), bph, abort_flag, a.err, a.wait_ns)) {
                            ok = false;
                            break;
                        }
                    }
                    fence_after();
                    const uint32_t sa = smem_u32(tiles + (size_t)stage * C::kStageBytes);
                    const uint64_t adesc = sdesc_k128(sa);
                    const bool bmn = kRouter && G.b_mn != 0;
                    const uint32_t sb = W8 ? smem_u32(bbuf + (size_t)bb * C::kBBytes) : sa + C::kABytes;
                    const uint64_t bdesc = bmn ? sdesc_mn128(sb, 8192) : sdesc_k128(sb);
                    // K step of 16: 32 bytes inside the K-major swizzle atom, or 16 rows of
                    // the MN-major tile (encoded >> 4)
                    const uint64_t bstep = bmn ? (2048 >> 4) : 2;
                    // an expert tile of at most 64 rows runs M = 64 MMAs on the first half of
                    // its A rows: less energy for the same result, which the power cap
                    // gives back as clock
                    const uint32_t idesc0 = bmn ? (kIdesc | kIdescBMajorMN) : kIdesc;
                    const bool m64 = (EPI <= kEpiFfn) && (seg_rows[t.s] - t.mb * kBM) <= 64;
                    const uint32_t idesc = m64 ? idesc_bf16_f32(64, BN) : idesc0;
                    const uint32_t idesc_f8 = m64 ? idesc_e4m3_f32(64, BN) : kIdescF8;
                    if (F8A && f8) {
                        // four K steps of 32 E4M3 elements, 32 bytes each
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + 2 * kk, idesc_f8, (kb | kk) != 0);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + bstep * kk, idesc,
                                     (kb | kk) != 0);
                    }
                    mma_commit(smem_u32(&empty[stage]));
                    if constexpr (W8) {
                        mma_commit(smem_u32(&bempty[bb]));
                        if (++bb == C::kBBufs) {
                            bb = 0;
                            bph ^= 1u;
                        }
                    }
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
            while (!mbar_try_wait(smem_u32(drain), 0) && globaltimer() - t0 < kDrainLimitNs) {
            }
        }
    } else if (W8 && warp == C::kB8Warp) {
        // ---------------------------------------------------------------- FP8 B producer (W8)
        // The weight tiles of every k block, in the walk's order, into the FP8 ring;
        // a slot is refilled once all converter warps have expanded it.
        if (lane == 0) {
            int f = 0;
            uint32_t fph = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = tile0; tile < total && ok; tile += tstep) {
                const TileAt t = locate(tile);
                const TcGemm &G = a.p[t.phase];
                const bool routed = t.s < G.g.E;
                int kb0, nk;
                krange(t, G, kb0, nk);
                // rows [nb*BN, nb*BN + BN) of the N dimension are slice `sub` of image `img`
                const int per = G.img_rows / BN, img = t.nb / per, sub = t.nb % per;
                const size_t img_bytes = (size_t)G.img_rows * kBK;
                const uint8_t *bt = (routed ? G.Bt0 + (size_t)t.s * G.bt_seg0 : G.Bt1) + (size_t)img * nk * img_bytes +
                                    (size_t)sub * C::kB8Bytes;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bounded(smem_u32(&f8empty[f]), fph ^ 1u, abort_flag, a.err, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&f8full[f]);
                    mbar_arrive_expect_tx(fb, C::kB8Bytes);
                    bulk_load(smem_u32(b8ring + (size_t)f * C::kB8Bytes), bt + (size_t)(kb0 + kb) * img_bytes,
                              C::kB8Bytes, fb);
                    ++issued;
                    if (++f == C::kB8Stages) {
                        f = 0;
                        fph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // leave no copy in flight: wait (bounded) for the last slots issued
                const int n = issued < C::kB8Stages ? issued : C::kB8Stages;
                for (int i = 0; i < n; ++i) {
                    if (--f < 0) {
                        f = C::kB8Stages - 1;
                        fph ^= 1u;
                    }
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(smem_u32(&f8full[f]), fph) && globaltimer() - t0 < kDrainLimitNs) {
                    }
                }
            }
        }
    } else if (W8 && warp >= kThreads / 32) {
        // ---------------------------------------------------------------- converter (W8)
        // k block j: FP8 slot j % kB8Stages -> bf16 B buffer j % kBBufs, once the MMA
        // has released that buffer, in the 128-byte swizzled K-major layout the
        // MMA descriptor expects.  Thread q of 256 converts the 16-byte chunks q,
        // q + 256, ... (contiguous per warp): chunk c is row c / 4, bytes 16 (c % 4).. of
        // the row = K elements 16 (c % 4)..+15, which land in bf16 chunks 2 (c % 4) and
        // 2 (c % 4) + 1, swizzled by row % 8.  Lane 0 polls the barriers; __syncwarp
        // orders the other lanes' accesses after it.
        const int q0 = threadIdx.x - kThreads;
        int bb = 0, f = 0;
        uint32_t bph = 0, fph = 0;
        bool ok = true;
        for (int tile = tile0; tile < total && ok; tile += tstep) {
            const TileAt t = locate(tile);
            int kb0, nk;
            krange(t, a.p[t.phase], kb0, nk);
            for (int kb = 0; kb < nk; ++kb) {
                int okw = 1;
                if (lane == 0)
                    okw = wait_bounded(smem_u32(&f8full[f]), fph, abort_flag, a.err, a.wait_ns) &&
                          wait_bounded(smem_u32(&bempty[bb]), bph ^ 1u, abort_flag, a.err, a.wait_ns);
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = b8ring + (size_t)f * C::kB8Bytes;
                uint8_t *dst = bbuf + (size_t)bb * C::kBBytes;
#pragma unroll
                for (int c = q0; c < C::kB8Bytes / 16; c += 32 * C::kConvWarps) {
                    const int r = c >> 2, c8 = c & 3;
                    const uint4 v = *reinterpret_cast<const uint4 *>(src + (size_t)c * 16);
                    uint4 lo, hi;
                    e4m3x16_to_bf16(v, lo, hi);
                    uint8_t *row = dst + (size_t)r * 128;
                    *reinterpret_cast<uint4 *>(row + (((2 * c8) ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(row + (((2 * c8 + 1) ^ (r & 7)) << 4)) = hi;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // st.shared -> MMA reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&f8empty[f]));   // the FP8 slot has been read
                    mbar_arrive(smem_u32(&conv[bb]));
                }
                if (++f == C::kB8Stages) {
                    f = 0;
                    fph ^= 1u;
                }
                if (++bb == C::kBBufs) {
                    bb = 0;
                    bph ^= 1u;
                }
            }
        }
    } else if (kSplitRoute && warp >= kThreads / 32) {
        // extra warps of the split router: they only take part in the selection
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;   // TMEM lanes [32*quarter, 32*quarter + 32)
        int it = 0;
        for (int tile = tile0; tile < total; tile += tstep, ++it) {
            const TileAt t = locate(tile);
            const TcGemm &G = a.p[t.phase];
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            int ok = 1;
            if (lane == 0) ok = wait_bounded(smem_u32(&tfull[acc]), acc_phase, abort_flag, a.err, a.wait_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            fence_after();
            const bool routed = t.s < G.g.E;
            const int rows = min(kBM, seg_rows[t.s] - t.mb * kBM);
            // M = 64 tiles: row 16 q + i of the accumulator is in TMEM lane 32 q + i (i < 16)
            const bool m64 = (EPI <= kEpiFfn) && rows <= 64;
            const int row = m64 ? (lane < 16 ? quarter * 16 + lane : kBM) : quarter * 32 + lane;
            const int grow = seg_row0[t.s] + t.mb * kBM + row;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
            if constexpr (kFusedRoute) {
                route_epilogue<BN, EPI - kEpiRoute>(a.route, taddr, grow, row < rows, psum_cta, s_loff, s_bias);
            } else if constexpr (kSplitRoute) {
                // this CTA's partial logits of the tile -> shared memory, row r at r * (BN + 4)
                // floats (the stage ring is idle: every MMA of the tile has completed)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                float *red = reinterpret_cast<float *>(tiles) + (size_t)row * (BN + 4);
                const int nchunk = min(BN / 16, (a.route.E + 15) / 16);
#pragma unroll 1
                for (int c = 0; c < nchunk; ++c) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c * 16, v);
                    tmem_ld_wait();
                    uint4 *dst = reinterpret_cast<uint4 *>(red + c * 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            } else {
                __nv_bfloat16 *Cp = static_cast<__nv_bfloat16 *>(routed ? G.C0 : G.C1);
                const int ldc = routed ? G.ldc0 : G.ldc1;
                const bool up = (EPI == kEpiSwiGLU) || (EPI == kEpiFfn && t.phase == 0);
                const bool f8 = tile_f8(t);
                // W8 or E4M3 operands: scales of this tile's BN output columns
                const float *sc = (W8 || f8) ? (routed ? G.sc0 + (size_t)t.s * G.b_rows0 : G.sc1) + (size_t)t.nb * BN
                                             : nullptr;
                if (up) {
                    float rs = 1.f;   // E4M3 activations: the scale of this row's token
                    if (f8 && row < rows) rs = routed ? G.rs0[G.rtok0 ? G.rtok0[grow] : grow] : G.rs1[grow];
                    epi_swiglu<BN>(taddr, Cp, ldc, grow, row, rows, t.nb, sc, rs);
                } else {
                    size_t orow = (size_t)grow;
                    float scale = 1.f;
                    if (a.gated && routed && row < rows) {
                        const int tok = a.row_token[grow];
                        orow = (size_t)tok;
                        scale = a.row_gate[tok];
                    }
                    epi_store<BN>(taddr, Cp, ldc, orow, scale, row, rows, t.nb, sc);
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
            if (EPI == kEpiFfn && t.phase == 0 && warp == 2 && lane == 0) {
                // publish this up tile's H rows to the down tiles (any CTA) that read them:
                // the phase of tempty[acc] completes once all four epilogue warps have
                // stored their rows (this warp cannot fall a phase behind: the next one
                // needs its own arrival), then a GPU-scope release of the counter
                if (wait_bounded(smem_u32(&tempty[acc]), acc_phase, abort_flag, a.err, a.wait_ns)) {
                    __threadfence();
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    int *cnt = a.dep + mtile_start[t.s] + t.mb;
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
                }
            }
        }
    }

    __syncthreads();
    if constexpr (kSplitRoute) {
        cluster_sync();   // every CTA of the cluster holds its partial rows in shared memory
        split_route_select<EPI - kEpiSplitRoute>(a.route, tiles, BN + 4, a.p[0].ksplit, seg_rows[0],
                                                 tile0 % mblk0, psum_cta);
        cluster_sync();   // no CTA leaves while another may still read its rows
    }
    if constexpr (kFusedRoute) {
        if (a.route.psum_rows) {   // this CTA's router score sums into its row: one atomic per expert
            float *row = a.route.psum_rows + (size_t)(blockIdx.x % kPsumRows) * a.route.E;
            for (int e = threadIdx.x; e < a.route.E; e += C::kThreadsCta) atomicAdd(row + e, psum_cta[e]);
        }
    }
    if (warp == 1) {
        __syncwarp();
        fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Persistent launch: one CTA per SM (at most max_tiles).  A kEpiFfn launch has CTAs
// waiting on other CTAs' up tiles, so it is a cooperative launch (all CTAs resident).
// Every CTA waits for the previous kernel on the stream before its first global
// access, so the launch is a dependent one and its setup overlaps that kernel.
template <int BN, int EPI, bool W8 = false, bool F8A = false>
cudaError_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0, const CUtensorMap &b1,
                        const CUtensorMap &a2, const CUtensorMap &a3, const TcArgs &args_in, int64_t max_tiles,
                        cudaStream_t s) {
    auto kern = tc_grouped_gemm_kernel<BN, EPI, W8, F8A>;
    constexpr int kBlock = TcCfg<BN, W8>::kThreadsCta;
    TcArgs args = args_in;
    args.wait_ns = wait_limit_ns();
    const size_t smem = TcCfg<BN, W8>::kSmem;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)(max_tiles > 1 ? max_tiles : 1);
    // always a dependent launch (the kernel waits for its predecessor before reading
    // global memory); a kEpiFfn launch is also cooperative
    err = launch_dependent(kern, dim3(grid), dim3(kBlock), smem, s, EPI == kEpiFfn, a0, a1, b0, b1, a2, a3, args);
    if (err != cudaSuccess && EPI == kEpiFfn) {
        // a runtime that refuses the two attributes together: plain cooperative launch
        (void)cudaGetLastError();
        TcArgs targs = args;
        void *params[] = {const_cast<CUtensorMap *>(&a0), const_cast<CUtensorMap *>(&a1),
                          const_cast<CUtensorMap *>(&b0), const_cast<CUtensorMap *>(&b1),
                          const_cast<CUtensorMap *>(&a2), const_cast<CUtensorMap *>(&a3), &targs};
        err = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid), dim3(kBlock), params,
                                          smem, s);
    }
    return err;
}

// Cluster-reduced split-K router (kEpiSplitRoute + KPL): one CTA per (token tile,
// K split), clusters of `splits` CTAs, each cluster one token tile.
template <int BN, int EPI>
cudaError_t launch_gemm_split_route(const CUtensorMap &a0, const CUtensorMap &b0, const TcArgs &args_in, int tiles,
                                    int splits, cudaStream_t s) {
    static_assert(EPI > kEpiSplitRoute, "cluster launch of the split-K router only");
    auto kern = tc_grouped_gemm_kernel<BN, EPI, false>;
    constexpr int kBlock = TcCfg<BN, false, kSplitSelectWarps>::kThreadsCta;
    static_assert(kBM * (BN + 4) * 4 <= TcCfg<BN, false>::kStages * TcCfg<BN, false>::kStageBytes,
                  "partial rows fit in the stage ring");
    TcArgs args = args_in;
    args.wait_ns = wait_limit_ns();
    const size_t smem = TcCfg<BN, false>::kSmem;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_dependent_cluster(kern, dim3(tiles * splits), dim3(kBlock), smem, s, splits, a0, a0, b0, b0, a0, a0,
                                    args);
}

// Single-GEMM launches pass their A maps again for the unused second phase.
template <int BN, int EPI, bool W8 = false, bool F8A = false>
cudaError_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0, const CUtensorMap &b1,
                        const TcArgs &args, int64_t max_tiles, cudaStream_t s) {
    return launch_gemm<BN, EPI, W8, F8A>(a0, a1, b0, b1, a0, a1, args, max_tiles, s);
}

}  // namespace
}  // namespace moe
