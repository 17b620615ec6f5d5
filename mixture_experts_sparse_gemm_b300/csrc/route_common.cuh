// Scoring and top-k selection of one token by one warp, shared by the CUDA-core
// router, the select kernel of the split-K tensor-core router and the
// cluster-reduced split-K router epilogue.
//
// Follows "技术日报 2026-04-14" (jsqmd.com) §3.1 (KeepTopK / Softmax gating), §3.2
// (softmax score p_i), §3.3 (Expert Choice scores), §3.5 (sigmoid score), §4.3
// (bias used for selection only), §9.1 (weights renormalised over the selected k).
#pragma once

#include <float.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

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

// Expert held in slot i of a lane: interleaved (lane + 32 i) or blocked
// (KPL consecutive experts per lane, lane * KPL + i).
template <int KPL, bool BLOCKED>
__device__ __forceinline__ int slot_expert(int lane, int i) {
    return BLOCKED ? lane * KPL + i : lane + 32 * i;
}

// Scores and selection of one token by one warp.  u[i] is the logit (offset
// included) of expert slot_expert(lane, i), -FLT_MAX past E.  Softmax (max and
// sum by warp reduction) or sigmoid, with the fast exponential and division (the
// scores are fp32 and their error stays far below the 1e-4 gaps that the
// selection is checked at); Expert Choice writes the scores expert-major; token
// choice takes k rounds of a warp arg-max on (key desc, index asc) over the keys
// score + selection bias, so slots come out in descending key order with ties to
// the lower expert index, and writes indices and (renormalised) weights.
// With a.psum_rows, every score is also added to the lane's running sums pacc
// (same slots), which the caller flushes once.
// bias (nullable): the lane's selection biases of its KPL slots, loaded once by a
// caller that selects many tokens; null reads them from a.sel_bias here.
template <int KPL, bool BLOCKED = false>
__device__ __forceinline__ void warp_score_select(const RouteArgs &a, const float (&u)[KPL], int t, int lane,
                                                  float (&pacc)[KPL], const float *bias = nullptr) {
    constexpr int kPerLane = KPL;
    const int E = a.E;
    float p[kPerLane];
    if (a.gate == MOE_GATE_SIGMOID) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) p[i] = __fdividef(1.f, 1.f + __expf(-u[i]));
    } else {
        float mx = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) mx = fmaxf(mx, u[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = slot_expert<KPL, BLOCKED>(lane, i);
            p[i] = (e < E) ? __expf(u[i] - mx) : 0.f;
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
            if (slot_expert<KPL, BLOCKED>(lane, i) < E) pacc[i] += p[i];
    }

    if (a.mode == MOE_EXPERT_CHOICE) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = slot_expert<KPL, BLOCKED>(lane, i);
            if (e < E) a.scores_t[(size_t)e * a.T + t] = p[i];
        }
        return;
    }

    // keys as order-preserving unsigned integers (a NaN key counts as -inf), so each
    // round is one warp max over the lanes' best keys and one warp min over the
    // indices holding that maximum: ties go to the lower expert index
    uint32_t key[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = slot_expert<KPL, BLOCKED>(lane, i);
        float kf = (e < E) ? p[i] + (bias ? bias[i] : (a.sel_bias ? a.sel_bias[e] : 0.f)) : -INFINITY;
        if (kf != kf) kf = -INFINITY;
        const uint32_t b = __float_as_uint(kf);
        key[i] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);   // ordered like the floats; -inf > 0
    }
    unsigned chosen = 0;     // bit i: the expert of slot i already selected
    float wsum = 0.f, wj = 0.f;
    int ij = 0;
    for (int j = 0; j < a.k; ++j) {
        uint32_t bk = 0;           // below every key of an expert in range
        int bi = 0x7fffffff;
        float bp = 0.f;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = slot_expert<KPL, BLOCKED>(lane, i);
            if (e < E && !(chosen >> i & 1u) && key[i] > bk) {   // ascending e: ties keep the lower
                bk = key[i];
                bi = e;
                bp = p[i];
            }
        }
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        bi = (int)__reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)bi : 0xffffffffu);
        const int owner = BLOCKED ? bi / KPL : (bi & 31);
        bp = __shfl_sync(0xffffffffu, bp, owner);   // the owner lane's best is the winner
        if (owner == lane) chosen |= 1u << (BLOCKED ? bi % KPL : bi >> 5);
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
template <int KPL, bool BLOCKED = false>
__device__ __forceinline__ void flush_prob_sum(const RouteArgs &a, const float (&pacc)[KPL], int lane,
                                               float *sacc) {
    if (!a.psum_rows) return;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) sacc[e] = 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int e = slot_expert<KPL, BLOCKED>(lane, i);
        if (e < a.E && pacc[i] != 0.f) atomicAdd(sacc + e, pacc[i]);
    }
    __syncthreads();
    float *row = a.psum_rows + (size_t)(blockIdx.x % kPsumRows) * a.E;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) atomicAdd(row + e, sacc[e]);
}

}  // namespace
}  // namespace moe
