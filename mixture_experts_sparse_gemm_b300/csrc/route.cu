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
// scores 4 tokens and selects their top-k: each lane holds the keys of experts
// lane, lane+32, ...; k rounds of a warp arg-max on (key, -index) -- a warp max
// of the keys, then a warp min of the indices holding it -- give the slots in
// descending key order with ties to the lower expert index.
#include <float.h>

#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kPerLane = kMaxE / 32;   // experts per lane, the most a warp holds
constexpr int kTM = 32;    // tokens per CTA
constexpr int kKC = 32;    // d-chunk staged per step
constexpr int kThreads = 256;


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
