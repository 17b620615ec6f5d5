// Router on CUDA cores: logits, scores, token-choice top-k and the Expert Choice
// column selection.
//
// Follows "技术日报 2026-04-14" (jsqmd.com) §3.1 (KeepTopK / Softmax gating), §3.2
// (softmax score p_i, Switch top-1), §3.3 (Expert Choice: each expert takes the top
// tokens of its column), §3.5 (sigmoid score), §4.3 (bias used for selection only),
// §9.1 (weights renormalised over the selected k).
//
// route_simt_kernel: one CTA computes the logits of 32 tokens for all E experts
// (fp32 FMA over d, x and W_r staged through shared memory), then every warp
// scores 4 tokens and selects their top-k with warp shuffles: each lane holds the
// keys of experts lane, lane+32, ...; k rounds of a warp arg-max on (key, -index)
// give the slots in descending key order with ties to the lower expert index.
#include <float.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTM = 32;    // tokens per CTA
constexpr int kKC = 32;    // d-chunk staged per step
constexpr int kThreads = 256;

struct RouteArgs {
    const void *x;
    const void *Wr;
    const float *logit_offset;
    const float *sel_bias;
    int T, d, E, k, gate, mode, renorm;
    int32_t *topk_idx;
    float *topk_w;
    float *scores_t;   // expert choice: [E][T]
    float *psum_rows;  // [kPsumRows][E] or null: += each block's sums of the experts' scores
};

constexpr int kPerLane = kMaxE / 32;   // experts per lane, the most a warp holds

// Scores and selection of one token by one warp.  u[i] is the logit (offset
// included) of expert lane + 32 i, -FLT_MAX past E.  Softmax (max and sum by warp
// reduction) or sigmoid; Expert Choice writes the scores expert-major; token
// choice takes k rounds of a warp arg-max on (key desc, index asc) over the keys
// score + selection bias, so slots come out in descending key order with ties to
// the lower expert index, and writes indices and (renormalised) weights.
// With a.psum_rows, every score is also added to the lane's running sums pacc
// (expert lane + 32 i), which the caller flushes once.
template <int KPL>
__device__ __forceinline__ void warp_score_select(const RouteArgs &a, const float (&u)[KPL], int t, int lane,
                                                  float (&pacc)[KPL]) {
    constexpr int kPerLane = KPL;
    const int E = a.E;
    float p[kPerLane];
    if (a.gate == MOE_GATE_SIGMOID) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) p[i] = 1.f / (1.f + expf(-u[i]));
    } else {
        float mx = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) mx = fmaxf(mx, u[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            p[i] = (e < E) ? expf(u[i] - mx) : 0.f;
            sum += p[i];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.f / sum;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) p[i] *= inv;
    }
    if (a.psum_rows) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            if (lane + 32 * i < E) pacc[i] += p[i];
    }

    if (a.mode == MOE_EXPERT_CHOICE) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E) a.scores_t[(size_t)e * a.T + t] = p[i];
        }
        return;
    }

    float key[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        key[i] = (e < E) ? p[i] + (a.sel_bias ? a.sel_bias[e] : 0.f) : -FLT_MAX;
    }
    unsigned chosen = 0;     // bit i: expert lane + 32 i already selected
    float wsum = 0.f, wj = 0.f;
    int ij = 0;
    for (int j = 0; j < a.k; ++j) {
        float bk = -FLT_MAX, bp = 0.f;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !(chosen >> i & 1u) && key[i] > bk) {   // ascending e: ties keep the lower
                bk = key[i];
                bi = e;
                bp = p[i];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            const float op = __shfl_xor_sync(0xffffffffu, bp, o);
            if (ok > bk || (ok == bk && oi < bi)) {
                bk = ok;
                bi = oi;
                bp = op;
            }
        }
        if (bi == 0x7fffffff) {
            // no unchosen key compares above -FLT_MAX (NaN scores from non-finite
            // inputs): take the lowest unchosen expert, so every index stays in range
            int low = 0x7fffffff;
#pragma unroll
            for (int i = kPerLane - 1; i >= 0; --i)
                if (lane + 32 * i < E && !(chosen >> i & 1u)) low = lane + 32 * i;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) low = min(low, __shfl_xor_sync(0xffffffffu, low, o));
            bi = low;
            bp = 0.f;
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                if (lane + 32 * i == bi) bp = p[i];
            bp = __shfl_sync(0xffffffffu, bp, bi & 31);   // the owner's score (not finite here)
        }
        if ((bi & 31) == lane) chosen |= 1u << (bi >> 5);
        wsum += bp;
        if (lane == j) {
            ij = bi;
            wj = bp;
        }
    }
    if (lane < a.k) {
        a.topk_idx[(size_t)t * a.k + lane] = ij;
        a.topk_w[(size_t)t * a.k + lane] = a.renorm ? wj / wsum : wj;
    }
}

// Adds the warps' running score sums to the block's row of psum_rows: shared-memory
// sums per block, then one global atomic per expert.  Every thread of the block
// calls it.
template <int KPL>
__device__ __forceinline__ void flush_prob_sum(const RouteArgs &a, const float (&pacc)[KPL], int lane,
                                               float *sacc) {
    if (!a.psum_rows) return;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) sacc[e] = 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int e = lane + 32 * i;
        if (e < a.E && pacc[i] != 0.f) atomicAdd(sacc + e, pacc[i]);
    }
    __syncthreads();
    float *row = a.psum_rows + (size_t)(blockIdx.x % kPsumRows) * a.E;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) atomicAdd(row + e, sacc[e]);
}

template <typename Tin, int NPT>
__global__ void __launch_bounds__(kThreads) route_simt_kernel(RouteArgs a) {
    extern __shared__ float smem[];
    float *xs = smem;                       // [kTM][kKC + 1]
    float *wsm = xs + kTM * (kKC + 1);      // [kKC][E]   later reused as logits [kTM][E]
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *Wr = static_cast<const Tin *>(a.Wr);
    const int E = a.E, d = a.d;
    const int t0 = blockIdx.x * kTM;
    const int tid = threadIdx.x;

    float acc[NPT];
#pragma unroll
    for (int i = 0; i < NPT; ++i) acc[i] = 0.f;

    for (int k0 = 0; k0 < d; k0 += kKC) {
        for (int i = tid; i < kTM * kKC; i += kThreads) {
            const int m = i / kKC, kk = i % kKC;
            const int t = t0 + m;
            xs[m * (kKC + 1) + kk] = (t < a.T && k0 + kk < d) ? to_f32(x[(size_t)t * d + k0 + kk]) : 0.f;
        }
        for (int i = tid; i < kKC * E; i += kThreads) {
            const int kk = i / E, e = i % E;
            wsm[i] = (k0 + kk < d) ? to_f32(Wr[(size_t)(k0 + kk) * E + e]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NPT; ++i) {
            const int o = tid + i * kThreads;
            if (o < kTM * E) {
                const int m = o / E, e = o % E;
                float s = acc[i];
#pragma unroll 8
                for (int kk = 0; kk < kKC; ++kk) s = fmaf(xs[m * (kKC + 1) + kk], wsm[kk * E + e], s);
                acc[i] = s;
            }
        }
        __syncthreads();
    }
    float *lg = wsm;   // [kTM][E]
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
        const int o = tid + i * kThreads;
        if (o < kTM * E) {
            const int e = o % E;
            lg[o] = acc[i] + (a.logit_offset ? a.logit_offset[e] : 0.f);
        }
    }
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    float pacc[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) pacc[i] = 0.f;
    for (int m = warp; m < kTM; m += kThreads / 32) {
        const int t = t0 + m;
        if (t >= a.T) break;
        float u[kPerLane];
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            u[i] = (e < E) ? lg[m * E + e] : -FLT_MAX;
        }
        warp_score_select<kPerLane>(a, u, t, lane, pacc);
    }
    __shared__ float sacc[kMaxE];
    flush_prob_sum<kPerLane>(a, pacc, lane, sacc);
}

// Scoring and selection from split-K partial logits of the tensor-core router:
// one warp per token sums partial[0..splits)[t][e] in split order, adds the logit
// offset, and runs warp_score_select.
// KPL = experts per lane (E <= 32 * KPL); the warps loop over tokens.
template <int KPL>
__global__ void __launch_bounds__(256) route_select_kernel(RouteArgs a, const float *__restrict__ partial, int splits,
                                                           int npad) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    float pacc[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) pacc[i] = 0.f;
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < a.T; t += nwarps) {
        // every partial of the token is loaded before the sums (split order kept)
        float pv[kMaxRouteSplits][KPL];
#pragma unroll
        for (int s = 0; s < kMaxRouteSplits; ++s)
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                const int e = lane + 32 * i;
                pv[s][i] = (s < splits && e < a.E) ? partial[((size_t)s * a.T + t) * npad + e] : 0.f;
            }
        float u[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int e = lane + 32 * i;
            float v = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxRouteSplits; ++s)
                if (s < splits) v += pv[s][i];
            if (e < a.E && a.logit_offset) v += a.logit_offset[e];
            u[i] = (e < a.E) ? v : -FLT_MAX;
        }
        warp_score_select<KPL>(a, u, t, lane, pacc);
    }
    __shared__ float sacc[kMaxE];
    flush_prob_sum<KPL>(a, pacc, lane, sacc);
}

template <typename Tin, int NPT>
cudaError_t launch_npt(const RouteArgs &a, cudaStream_t s) {
    const size_t smem = sizeof(float) * (kTM * (kKC + 1) + kKC * a.E);
    auto kern = route_simt_kernel<Tin, NPT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int grid = (a.T + kTM - 1) / kTM;
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_typed(const RouteArgs &a, cudaStream_t s) {
    const int npt = (kTM * a.E + kThreads - 1) / kThreads;
    if (npt <= 1) return launch_npt<Tin, 1>(a, s);
    if (npt <= 2) return launch_npt<Tin, 2>(a, s);
    if (npt <= 4) return launch_npt<Tin, 4>(a, s);
    if (npt <= 8) return launch_npt<Tin, 8>(a, s);
    if (npt <= 16) return launch_npt<Tin, 16>(a, s);
    return launch_npt<Tin, 32>(a, s);
}

// ----------------------------------------------------------------------------- expert choice
// One CTA per expert.  The column S[:, e] (non-negative floats, so their bit
// patterns order like the values) goes through a 4-pass, 8-bit radix select for
// the cap-th largest key K; every token with key > K is taken, plus the lowest
// token indices among those with key == K until cap are taken.  The taken tokens
// are written in ascending token order with a block-wide ordered compaction.
constexpr int kEcThreads = 1024;
constexpr int kEcSmemMaxT = 49152;   // the column stays in shared memory up to this many tokens (192 KB)
constexpr int kEcBins = 4096;        // widest radix digit (12 bits)

// Exclusive block-wide prefix sum of one int per thread; `total` gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        const int w = (lane < nw) ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nw) warp_tot[32 + lane] = wi - w;
        if (lane == 31) warp_tot[64] = wi;
    }
    __syncthreads();
    const int r = warp_tot[32 + warp] + incl - v;
    total = warp_tot[64];
    __syncthreads();
    return r;
}

// col_cnt (nullable): column e takes min(col_cnt[e], cap) tokens instead of cap
// (the affinity-ordered capacity drop); outputs stay [E][cap].
__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(const float *scores_t, int T, int cap,
                                                                 const int32_t *col_cnt, int32_t *ec_tok,
                                                                 float *ec_w) {
    extern __shared__ unsigned s_col[];   // the expert's column, when it fits
    __shared__ unsigned hist[kEcBins];
    __shared__ int warp_tot[65];
    __shared__ unsigned s_digit;
    __shared__ int s_remaining;
    const int e = blockIdx.x;
    const int take = col_cnt ? min(col_cnt[e], cap) : cap;   // tokens this column keeps
    if (take <= 0) return;                                      // the whole block leaves together
    const unsigned *g = reinterpret_cast<const unsigned *>(scores_t + (size_t)e * T);
    const bool in_smem = T <= kEcSmemMaxT;
    if (in_smem) {
        for (int t = threadIdx.x; t < T; t += blockDim.x) s_col[t] = g[t];
        __syncthreads();
    }
    const unsigned *col = in_smem ? s_col : g;

    // three digits, high to low: 12 bits (sign, exponent and 3 mantissa bits, so the
    // scores of one expert -- which share a few exponents -- spread over many bins),
    // then 10 and 10 bits
    constexpr int kShift[3] = {20, 10, 0};
    constexpr int kBits[3] = {12, 10, 10};
    unsigned prefix = 0, mask = 0;
    int remaining = take;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = kShift[pass];
        const int nb = 1 << kBits[pass];
        const unsigned dmask = (unsigned)nb - 1u;
        for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int t = threadIdx.x; t < T; t += blockDim.x) {
            const unsigned u = col[t];
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & dmask], 1u);
        }
        __syncthreads();
        // find the digit holding the `remaining`-th largest key: thread i sums the
        // bins of digits it owns (digits counted from the top), a block scan gives
        // the keys above them, and the owner of the crossing walks its bins
        const int per = (nb + (int)blockDim.x - 1) / (int)blockDim.x;
        const int b_hi = nb - 1 - (int)threadIdx.x * per;   // this thread's digits: b_hi, b_hi-1, ...
        int mine = 0;
        for (int j = 0; j < per; ++j)
            if (b_hi - j >= 0) mine += (int)hist[b_hi - j];
        int tot;
        const int above = block_exclusive_scan(mine, warp_tot, tot);
        if (above < remaining && above + mine >= remaining) {
            int cum = above;
            for (int j = 0; j < per; ++j) {
                const int b = b_hi - j;
                if (b < 0) break;
                const int h = (int)hist[b];
                if (cum + h >= remaining) {
                    s_digit = (unsigned)b;
                    s_remaining = remaining - cum;
                    break;
                }
                cum += h;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= dmask << shift;
        remaining = s_remaining;
        __syncthreads();
    }
    const unsigned K = prefix;   // the cap-th largest key; `remaining` ties at K are taken

    // ordered compaction: thread i owns tokens [i*per, (i+1)*per), so thread order
    // is token order; ties at K go to the lowest token indices
    const int per = (T + (int)blockDim.x - 1) / (int)blockDim.x;
    const int t0 = threadIdx.x * per, t1 = min(T, t0 + per);
    int gt = 0, eq = 0;
    for (int t = t0; t < t1; ++t) {
        const unsigned u = col[t];
        gt += u > K;
        eq += u == K;
    }
    int tot;
    const int eq_before = block_exclusive_scan(eq, warp_tot, tot);
    const int take_eq = max(0, min(eq, remaining - eq_before));
    const int pos0 = block_exclusive_scan(gt + take_eq, warp_tot, tot);
    int p = pos0, te = 0;
    for (int t = t0; t < t1; ++t) {
        const unsigned u = col[t];
        const bool sel = (u > K) || (u == K && te++ < take_eq);
        if (sel && p < take) {
            ec_tok[(size_t)e * cap + p] = t;
            ec_w[(size_t)e * cap + p] = __uint_as_float(u);
            ++p;
        }
    }
}

}  // namespace

cudaError_t launch_route_simt(const moe_config &c, const void *x, const void *W_r, const float *logit_offset,
                              const float *sel_bias, int32_t *topk_idx, float *topk_w, float *scores_t,
                              float *psum_rows, unsigned *err, cudaStream_t s) {
    (void)err;
    RouteArgs a{};
    a.x = x;
    a.Wr = W_r;
    a.logit_offset = logit_offset;
    a.sel_bias = sel_bias;
    a.T = c.T;
    a.d = c.d;
    a.E = c.E;
    a.k = c.k;
    a.gate = c.gate;
    a.mode = c.mode;
    a.renorm = c.renormalize;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.scores_t = scores_t;
    a.psum_rows = psum_rows;
    if (c.dtype == MOE_F32) return launch_typed<float>(a, s);
    return launch_typed<__nv_bfloat16>(a, s);
}

cudaError_t launch_route_select(const moe_config &c, const float *logit_offset, const float *sel_bias,
                                int32_t *topk_idx, float *topk_w, float *scores_t, float *psum_rows,
                                const float *partial, int splits, int npad, cudaStream_t s) {
    RouteArgs a{};
    a.logit_offset = logit_offset;
    a.sel_bias = sel_bias;
    a.T = c.T;
    a.d = c.d;
    a.E = c.E;
    a.k = c.k;
    a.gate = c.gate;
    a.mode = c.mode;
    a.renorm = c.renormalize;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.scores_t = scores_t;
    a.psum_rows = psum_rows;
    int blocks = (c.T + 7) / 8;
    const int cap = num_sms() * 2;   // warps loop over tokens: the body stays in the instruction cache
    if (blocks > cap) blocks = cap;
    auto kern = c.E <= 32 ? route_select_kernel<1> : c.E <= 64 ? route_select_kernel<2>
              : c.E <= 128 ? route_select_kernel<4> : route_select_kernel<8>;
    return launch_dependent(kern, dim3(blocks), dim3(256), 0, s, false, a, partial, splits, npad);
}

cudaError_t launch_ec_select(const moe_config &c, const float *scores_t, int32_t *ec_tok, float *ec_w,
                             cudaStream_t s) {
    const size_t smem = c.T <= kEcSmemMaxT ? sizeof(unsigned) * (size_t)c.T : 0;
    cudaError_t err = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    ec_select_kernel<<<c.E, kEcThreads, smem, s>>>(scores_t, c.T, c.ec_capacity, nullptr, ec_tok, ec_w);
    return cudaGetLastError();
}

cudaError_t launch_column_select(const moe_config &c, const float *scores_t, int cap, const int32_t *col_cnt,
                                 int32_t *tok, float *w, cudaStream_t s) {
    const size_t smem = c.T <= kEcSmemMaxT ? sizeof(unsigned) * (size_t)c.T : 0;
    cudaError_t err = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    ec_select_kernel<<<c.E, kEcThreads, smem, s>>>(scores_t, c.T, cap, col_cnt, tok, w);
    return cudaGetLastError();
}

}  // namespace moe
