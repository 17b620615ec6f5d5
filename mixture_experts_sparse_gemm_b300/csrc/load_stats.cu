// Load statistics of one routing, the diagnostics of "技术日报 2026-04-14" §4.4
// (token fraction, load imbalance factor, coefficient of variation, router
// entropy) and the balance terms of §4.2 (the Switch auxiliary loss N·Σ f_i·P_i
// and the DeepSeek V1 expert-level balance Σ f'_i·P_i, both without their α).
//
//   f_e  = cnt_raw[e] / Σ cnt_raw          share of the assignments routed to e
//                                          (before any capacity drop)
//   f1_e = share of tokens whose first choice (slot 0) is e; Expert Choice: f_e
//   P_e  = prob_sum[e] / T                 mean router score of e over the tokens
//   LIF  = E·max f        CV = std(f) / mean(f)  (population std)
//   H    = −Σ q ln q, q = P / Σ P          (natural log; q = 0 terms are 0)
//   switch_aux = E·Σ f1·P                  expert_balance = E·Σ f·P
// One CTA: 1024 threads build per-warp slot-0 histograms (eight indices loaded per
// thread before counting; lanes with the same expert add once), then one warp does
// the per-expert arithmetic in fp32 (experts lane + 32 i) with shuffle reductions.
// The results are fp32-accurate (about 1e-6 relative); the summary is returned as
// doubles.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStatThreads = 1024;
constexpr int kStatWarps = kStatThreads / 32;
constexpr int kHistBatch = 8;
constexpr int kPerLane = kMaxE / 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// prob_sum[e] = rows[0][e] + rows[1][e] + ... + rows[kPsumRows - 1][e]
__global__ void sum_psum_rows_kernel(const float *__restrict__ rows, int E, float *prob_sum) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        for (int r = 0; r < kPsumRows; ++r) s += rows[(size_t)r * E + e];
        prob_sum[e] = s;
    }
}

__global__ void __launch_bounds__(kStatThreads)
    load_stats_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ cnt_raw,
                      const float *__restrict__ prob_sum, int T, int E, int k, int ec, float *token_fraction,
                      float *prob_mean, double *summary) {
    __shared__ int hist[kStatWarps][kMaxE];   // per-warp slot-0 histograms
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = lane; e < E; e += 32) hist[warp][e] = 0;
    __syncwarp();
    if (!ec) {
        // warp-uniform trip count: __match_any_sync below needs all 32 lanes
        for (int base = 0; base + (tid & ~31) < T; base += kHistBatch * kStatThreads) {
            int e[kHistBatch];
#pragma unroll
            for (int j = 0; j < kHistBatch; ++j) {
                const int t = base + tid + j * kStatThreads;
                e[j] = t < T ? topk_idx[(size_t)t * k] : -1;
            }
#pragma unroll
            for (int j = 0; j < kHistBatch; ++j) {
                // lanes holding the same expert add once, by the lowest of them
                const unsigned same = __match_any_sync(0xffffffffu, e[j]);
                if ((unsigned)e[j] < (unsigned)E && lane == __ffs(same) - 1) hist[warp][e[j]] += __popc(same);
                __syncwarp();
            }
        }
    }
    __syncthreads();
    if (warp != 0) return;   // one warp finishes: experts lane + 32 i
    float cnt[kPerLane], P[kPerLane], f[kPerLane];
    int first[kPerLane];
    float total = 0.f, psum = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        cnt[i] = e < E ? (float)cnt_raw[e] : 0.f;
        P[i] = e < E ? prob_sum[e] / (float)T : 0.f;
        int n = 0;
        if (e < E && !ec)
            for (int w = 0; w < kStatWarps; ++w) n += hist[w][e];
        first[i] = n;
        total += cnt[i];
        psum += P[i];
    }
    total = warp_sum(total);
    psum = warp_sum(psum);
    float fmax_ = -1.f, fsum = 0.f, sw = 0.f, eb = 0.f, h = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        f[i] = (e < E && total > 0.f) ? cnt[i] / total : 0.f;
        const float f1 = e < E ? (ec ? f[i] : (float)first[i] / (float)T) : 0.f;
        if (e < E) {
            token_fraction[e] = f[i];
            prob_mean[e] = P[i];
            fmax_ = fmaxf(fmax_, f[i]);
            const float q = psum > 0.f ? P[i] / psum : 0.f;
            if (q > 0.f) h -= q * logf(q);
        }
        fsum += f[i];
        sw += f1 * P[i];
        eb += f[i] * P[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fmax_ = fmaxf(fmax_, __shfl_xor_sync(0xffffffffu, fmax_, o));
    const float mean = warp_sum(fsum) / E;
    float dev = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
        if (lane + 32 * i < E) dev += (f[i] - mean) * (f[i] - mean);
    const float var = warp_sum(dev) / E;
    h = warp_sum(h);
    sw = warp_sum(sw);
    eb = warp_sum(eb);
    if (lane == 0) {
        summary[0] = (double)E * fmax_;
        summary[1] = mean > 0.f ? (double)sqrtf(var) / mean : 0.0;
        summary[2] = h;
        summary[3] = (double)E * sw;
        summary[4] = (double)E * eb;
    }
}

}  // namespace

cudaError_t launch_sum_psum_rows(const moe_config &c, const float *rows, float *prob_sum, cudaStream_t s) {
    sum_psum_rows_kernel<<<1, 256, 0, s>>>(rows, c.E, prob_sum);
    return cudaGetLastError();
}

cudaError_t launch_load_stats(const moe_config &c, const int32_t *topk_idx, const int32_t *cnt_raw,
                              const float *prob_sum, float *token_fraction, float *prob_mean, double *summary,
                              cudaStream_t s) {
    load_stats_kernel<<<1, kStatThreads, 0, s>>>(topk_idx, cnt_raw, prob_sum, c.T, c.E, c.k,
                                                 c.mode == MOE_EXPERT_CHOICE ? 1 : 0, token_fraction, prob_mean,
                                                 summary);
    return cudaGetLastError();
}

}  // namespace moe
