// Capacity-limited dispatch: a stable counting sort of the (token, slot)
// assignments by expert, with the capacity drop applied in token order, followed
// by a 16-byte vectorised row gather of x into expert order.
//
// Follows "技术日报 2026-04-14" (jsqmd.com) §3.2 (capacity K_max and overflow drop)
// and "MoE稀疏架构" (cloud.baidu.com) §4 step 3 (inputs distributed to the chosen
// experts).  The kept assignments of expert e are its first cap assignments in
// (token, slot) order; they occupy rows off[e] .. off[e+1]-1 in that order.
//
// Kernels (token choice):
//   count  : one warp per chunk of 256 assignments -> per-chunk expert counts
//   scan   : one CTA; per expert, running base over the chunks, raw count,
//            capped count, and the exclusive scan of capped counts -> off[]
//   rank   : one warp per chunk; __match_any_sync groups the lanes holding the
//            same expert so ranks follow assignment order -> slot_of, row_token
//   gather : one warp per destination row, 16-byte vectors -> x_perm
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kChunk = 256;          // assignments per warp-chunk
constexpr int kWarpsPerCta = 4;

__global__ void __launch_bounds__(32 * kWarpsPerCta)
    dispatch_count_kernel(const int32_t *idx, int64_t n, int E, int nchunks, int32_t *chunk_cnt) {
    extern __shared__ int cnt[];   // [kWarpsPerCta][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x * kWarpsPerCta + warp;
    int *my = cnt + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    if (chunk < nchunks) {
        for (int i = lane; i < kChunk; i += 32) {
            const int64_t a = (int64_t)chunk * kChunk + i;
            if (a < n) {
                const int e = idx[a];
                if ((unsigned)e < (unsigned)E) atomicAdd(&my[e], 1);
            }
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) chunk_cnt[(size_t)chunk * E + e] = my[e];
    }
}

__global__ void __launch_bounds__(256)
    dispatch_scan_kernel(int32_t *chunk_cnt, int nchunks, int E, int cap, int32_t *cnt_raw, int32_t *off) {
    __shared__ int kept[kMaxE];
    const int e = threadIdx.x;
    if (e < E) {
        int run = 0;
        for (int c = 0; c < nchunks; ++c) {
            const int v = chunk_cnt[(size_t)c * E + e];
            chunk_cnt[(size_t)c * E + e] = run;   // base of this chunk inside expert e
            run += v;
        }
        cnt_raw[e] = run;
        kept[e] = (cap < 0) ? run : min(run, cap);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int i = 0; i < E; ++i) {
            off[i] = acc;
            acc += kept[i];
        }
        off[E] = acc;
    }
}

__global__ void __launch_bounds__(32 * kWarpsPerCta)
    dispatch_rank_kernel(const int32_t *idx, int64_t n, int k, int E, int nchunks, const int32_t *chunk_base,
                         const int32_t *off, int cap, int32_t *slot_of, int32_t *row_token, unsigned *err) {
    extern __shared__ int run[];   // [kWarpsPerCta][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x * kWarpsPerCta + warp;
    if (chunk >= nchunks) return;
    int *my = run + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = chunk_base[(size_t)chunk * E + e];
    __syncwarp();
    for (int step = 0; step < kChunk / 32; ++step) {
        const int64_t a = (int64_t)chunk * kChunk + step * 32 + lane;
        const int e_in = (a < n) ? idx[a] : -1;
        const bool valid = (unsigned)e_in < (unsigned)E;   // out-of-range ids are dropped and flagged
        if (a < n && !valid) {
            slot_of[a] = -1;
            atomicOr(err, kErrBadIndex);
        }
        const int e = valid ? e_in : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank_in = __popc(peers & ((1u << lane) - 1u));
        const int base = valid ? my[e] : 0;
        __syncwarp();
        if (valid && rank_in == 0) my[e] = base + __popc(peers);
        __syncwarp();
        if (valid) {
            const int r = base + rank_in;
            const int slot = (cap < 0 || r < cap) ? off[e] + r : -1;
            slot_of[a] = slot;
            if (slot >= 0) row_token[slot] = (int32_t)(a / k);
        }
    }
}

// The same three steps in one launch of a thread-block cluster of Q CTAs (Q = 1,
// 2, 4 or 8: one per 2048 assignments) of 32 warps each, for up to kPlanMax assignments.  The
// 32 Q warps own consecutive segments of the assignments (warp order = assignment
// order) and hold them in registers: lane l keeps assignments a0 + 32 q + l,
// q < PER, all loaded at once.  Pass 1: each warp counts its segment per expert
// into its own shared-memory counters; thread e turns its CTA's 32 per-warp counts
// of expert e into per-warp rank bases and the CTA's count.  After a cluster
// barrier every CTA reads the other CTAs' counts (distributed shared memory): the
// sum over the CTAs before it is its base, the sum over all the raw count; warp 0
// caps and scans the counts into off[] (every CTA the same; CTA 0 writes them).
// Pass 2: each warp ranks its segment in order from its bases; lanes holding the
// same expert are found with ballots (warp_peers9); slot_of and row_token are
// written directly.
constexpr int kPlanWarps = 32;
constexpr int64_t kPlanMax = 32 * kPlanWarps * 32;   // the multi-kernel path above this
constexpr int kPlanMaxCtas = 8;

size_t plan_smem_bytes(int E) { return sizeof(int) * ((size_t)kPlanWarps * E + 3 * (size_t)E + 1); }

__device__ __forceinline__ uint32_t plan_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void plan_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the int at shared-memory address `p` of this CTA, in CTA `rank` of the cluster
__device__ __forceinline__ int plan_ld_remote(const int *p, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p)), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    int v;
    asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(r) : "memory");
    return v;
}

template <int PER>
__global__ void __launch_bounds__(32 * kPlanWarps)
    dispatch_plan_kernel(const int32_t *idx, int n, int k, int E, int cap, int32_t *cnt_raw, int32_t *off,
                         int32_t *slot_of, int32_t *row_token, unsigned *err) {
    extern __shared__ int sm[];
    int *wcnt = sm;                        // [kPlanWarps][E]: counts, then rank bases
    int *ctot = wcnt + kPlanWarps * E;     // [E]: this CTA's count per expert
    int *cbase = ctot + E;                 // [E]: the counts of the CTAs before this one
    int *offs = cbase + E;                 // [E + 1]
    pdl_wait();
    pdl_trigger();
    const int Q = (int)gridDim.x;          // the whole grid is one cluster (or one CTA)
    const int rank = Q > 1 ? (int)plan_ctarank() : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gwarps = kPlanWarps * Q;
    const int seg = ((n + gwarps - 1) / gwarps + 31) & ~31;   // <= 32 * PER
    const int a0 = min(n, (rank * kPlanWarps + warp) * seg), a1 = min(n, a0 + seg);
    int *my = wcnt + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    int ev[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const int a = a0 + q * 32 + lane;
        ev[q] = (a < a1) ? idx[a] : -1;
    }
    __syncwarp();
#pragma unroll
    for (int q = 0; q < PER; ++q)   // counts: fire-and-forget shared adds
        if ((unsigned)ev[q] < (unsigned)E) atomicAdd(&my[ev[q]], 1);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {   // per-warp bases in segment order
        int s = 0;
#pragma unroll
        for (int w = 0; w < kPlanWarps; ++w) {
            const int c = wcnt[w * E + e];
            wcnt[w * E + e] = s;
            s += c;
        }
        ctot[e] = s;
    }
    if (Q > 1) plan_cluster_sync();   // every CTA's counts are visible to the cluster
    else __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int before = 0, all = 0;
        for (int c = 0; c < Q; ++c) {
            const int v = (c == rank) ? ctot[e] : plan_ld_remote(ctot + e, (uint32_t)c);
            if (c < rank) before += v;
            all += v;
        }
        cbase[e] = before;
        offs[e] = all;   // raw count, scanned below
    }
    if (Q > 1) plan_cluster_sync();   // no CTA's counts are read after this (a CTA may leave)
    else __syncthreads();
    if (warp == 0) {   // kept counts and their exclusive scan, 32 experts per step
        int carry = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            int kept = 0;
            if (e < E) {
                const int raw = offs[e];
                if (rank == 0) cnt_raw[e] = raw;
                kept = (cap < 0) ? raw : min(raw, cap);
            }
            int incl = kept;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e < E) offs[e] = carry + incl - kept;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) offs[E] = carry;
    }
    __syncthreads();
    if (rank == 0)
        for (int e = tid; e <= E; e += blockDim.x) off[e] = offs[e];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        if (a0 + q * 32 >= a1) break;   // warp-uniform
        const int a = a0 + q * 32 + lane;
        const bool valid = (unsigned)ev[q] < (unsigned)E;
        if (a < a1 && !valid) {
            slot_of[a] = -1;
            atomicOr(err, kErrBadIndex);
        }
        const int e = valid ? ev[q] : 0;
        const unsigned peers = warp_peers9(valid ? (unsigned)e : 511u);   // invalid lanes group apart
        const int rank_in = __popc(peers & ((1u << lane) - 1u));
        const int base = valid ? my[e] : 0;
        __syncwarp();
        if (valid && rank_in == 0) my[e] = base + __popc(peers);
        __syncwarp();
        if (valid) {
            const int r = cbase[e] + base + rank_in;
            const int slot = (cap < 0 || r < cap) ? offs[e] + r : -1;
            slot_of[a] = slot;
            if (slot >= 0) row_token[slot] = a / k;
        }
    }
}

template <int PER>
cudaError_t launch_plan(const int32_t *idx, int n, int k, int E, int cap, int32_t *cnt_raw, int32_t *off,
                        int32_t *slot_of, int32_t *row_token, unsigned *err, int ctas, cudaStream_t s) {
    const size_t smem = plan_smem_bytes(E);
    cudaError_t ce = cudaFuncSetAttribute(dispatch_plan_kernel<PER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smem);
    if (ce != cudaSuccess) return ce;
    if (ctas == 1)
        return launch_dependent(dispatch_plan_kernel<PER>, dim3(1), dim3(32 * kPlanWarps), smem, s, false, idx, n, k, E,
                                cap, cnt_raw, off, slot_of, row_token, err);
    return launch_dependent_cluster(dispatch_plan_kernel<PER>, dim3(ctas), dim3(32 * kPlanWarps), smem, s, ctas, idx,
                                    n, k, E, cap, cnt_raw, off, slot_of, row_token, err);
}

// x_perm[row] = x[row_token[row]] for row < *rows (read on the device).  One warp
// per (row, span of the row), four 16-byte vectors per lane in flight; a span is
// the whole row unless there are fewer rows than 16 warps per SM.
// With z.slot_of, the same launch zeroes the output rows of dropped tokens and
// the dependency counters of the fused expert launch (see GatherZero).
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint4 *__restrict__ x, int vecs, int span, const int32_t *__restrict__ row_token,
                       const int32_t *__restrict__ rows_dev, int64_t rows_host, uint4 *__restrict__ x_perm,
                       GatherZero z) {
    pdl_wait();
    pdl_trigger();
    const int64_t rows = rows_dev ? (int64_t)*rows_dev : rows_host;
    const int nch = (vecs + span - 1) / span;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int64_t it = gw; it < rows * nch; it += nwarps) {
        const int64_t r = it / nch;
        const int c = (int)(it - r * nch);
        const uint4 *src = x + (size_t)row_token[r] * vecs;
        uint4 *dst = x_perm + (size_t)r * vecs;
        const int vend = min(vecs, (c + 1) * span);
        for (int v = c * span + lane; v < vend; v += 128) {
            uint4 t[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (v + 32 * q < vend) t[q] = src[v + 32 * q];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (v + 32 * q < vend) dst[v + 32 * q] = t[q];
        }
    }
    if (z.slot_of) {
        for (int64_t t0 = gw * 32; t0 < z.T; t0 += nwarps * 32) {   // warp-uniform bound
            const int64_t t = t0 + lane;
            unsigned m = __ballot_sync(0xffffffffu, t < z.T && z.slot_of[t] < 0);
            while (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                uint4 *row = z.y + (size_t)(t0 + b) * z.y_vecs;
                for (int v = lane; v < z.y_vecs; v += 32) row[v] = make_uint4(0, 0, 0, 0);
            }
        }
        if (blockIdx.x == 0)
            for (int i = threadIdx.x; i < z.ndep; i += blockDim.x) z.dep[i] = 0;
    }
}

cudaError_t launch_gather(const void *x, int vecs, const int32_t *row_token, const int32_t *rows_dev,
                          int64_t rows_host, void *x_perm, const GatherZero &z_in, cudaStream_t s) {
    GatherZero z = z_in;
    if (z.y_vecs == 0) z.y_vecs = vecs;
    constexpr int kSpanStep = 128;   // vectors of one warp step (four per lane)
    const int64_t target = (int64_t)num_sms() * 16;   // rows split only below 16 warps per SM
    const int max_ch = (vecs + kSpanStep - 1) / kSpanStep;
    int64_t nch = rows_host > 0 ? (target + rows_host - 1) / rows_host : 1;
    nch = nch < 1 ? 1 : (nch > max_ch ? max_ch : nch);
    const int span = (int)(((vecs + nch - 1) / nch + kSpanStep - 1) / kSpanStep * kSpanStep);
    const int64_t items = rows_host * ((vecs + span - 1) / span);
    int64_t blocks = (items + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_dependent(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, s, false,
                            static_cast<const uint4 *>(x), vecs, span, row_token, rows_dev, rows_host,
                            static_cast<uint4 *>(x_perm), z);
}

// Expert choice: off[e] = e*cap, cnt_raw[e] = cap, slot_of[t][e] = e*cap + r.
__global__ void ec_slots_kernel(const int32_t *ec_tok, int T, int E, int cap, int32_t *off, int32_t *cnt_raw,
                                int32_t *slot_of, unsigned *err) {
    const int64_t n = (int64_t)E * cap;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t e = first; e <= E; e += stride) {
        off[e] = (int32_t)(e * cap);
        if (e < E) cnt_raw[e] = cap;
    }
    for (int64_t i = first; i < n; i += stride) {
        const int e = (int)(i / cap);
        const int t = ec_tok[i];
        if ((unsigned)t < (unsigned)T) slot_of[(size_t)t * E + e] = (int32_t)i;
        else atomicOr(err, kErrBadIndex);
    }
}

// ----------------------------------------------------------------------------- affinity-ordered drop
// DeepSeek-V2 drop ("技术日报 2026-04-14" §5.2: over-capacity tokens dropped by
// descending affinity): an expert over capacity keeps the `cap` assignments with
// the largest gate weights, ties to the lower token.  The weights go into a dense
// S[E][T] (0 where the token did not choose the expert; weights are positive), the
// column select of the Expert Choice path takes min(cnt_raw[e], cap) per column in
// ascending token order, and the rows are placed from there.

// S[e][t] = topk_w[t][j] for every assignment (t, j) -> e; cnt_raw[e] += 1
__global__ void affinity_scatter_kernel(const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
                                        int64_t n, int k, int T, int E, float *S, int32_t *cnt_raw, unsigned *err) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int e = topk_idx[i];
        if ((unsigned)e >= (unsigned)E) {
            atomicOr(err, kErrBadIndex);
            continue;
        }
        S[(size_t)e * T + i / k] = topk_w[i];
        atomicAdd(&cnt_raw[e], 1);
    }
}

// One block per expert: off[e] = sum over e' < e of min(cnt_raw[e'], cap); the kept
// tokens kept[e][r] (ascending) get rows off[e] + r: row_token, and slot_of of the
// slot j with topk_idx[t][j] == e.
__global__ void affinity_rows_kernel(const int32_t *__restrict__ kept, const int32_t *__restrict__ cnt_raw, int cap,
                                     const int32_t *__restrict__ topk_idx, int k, int E, int32_t *off, int32_t *slot_of,
                                     int32_t *row_token) {
    __shared__ int s_off;
    const int e = blockIdx.x;
    if (threadIdx.x < 32) {
        int part = 0;
        for (int q = threadIdx.x; q < e; q += 32) part += min(cnt_raw[q], cap);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (threadIdx.x == 0) {
            s_off = part;
            off[e] = part;
            if (e == E - 1) off[E] = part + min(cnt_raw[e], cap);
        }
    }
    __syncthreads();
    const int take = min(cnt_raw[e], cap), base = s_off;
    for (int r = threadIdx.x; r < take; r += blockDim.x) {
        const int t = kept[(size_t)e * cap + r];
        row_token[base + r] = t;
        for (int j = 0; j < k; ++j)
            if (topk_idx[(size_t)t * k + j] == e) slot_of[(size_t)t * k + j] = base + r;
    }
}


}  // namespace

int dispatch_tc_launches(int64_t assignments) { return assignments <= kPlanMax ? 2 : 4; }

size_t dispatch_tc_scratch_ints(int64_t assignments, int E) {
    const int64_t nchunks = (assignments + kChunk - 1) / kChunk;
    return (size_t)(nchunks * E) + (size_t)assignments;   // chunk counts + row_token
}

cudaError_t launch_dispatch_tc(const moe_config &c, int32_t cap, const int32_t *topk_idx, const void *x,
                               int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm,
                               int32_t *chunk_cnt, int32_t *row_token, unsigned *err, cudaStream_t s,
                               const GatherZero &zero, int row_bytes) {
    const int64_t n = (int64_t)c.T * c.k;
    if (n <= kPlanMax) {
        // one CTA per 2048 assignments, up to a cluster of eight
        const int ctas = n <= 2048 ? 1 : n <= 4096 ? 2 : n <= 8192 ? 4 : kPlanMaxCtas;
        const int per = (int)((n + 32 * kPlanWarps * ctas - 1) / (32 * kPlanWarps * ctas));   // per lane
        auto pick = [](int p) {
            return p <= 1 ? launch_plan<1> : p <= 2 ? launch_plan<2> : p <= 4 ? launch_plan<4>
                 : p <= 8 ? launch_plan<8> : p <= 16 ? launch_plan<16> : launch_plan<32>;
        };
        cudaError_t ce = pick(per)(topk_idx, (int)n, c.k, c.E, cap, cnt_raw, off, slot_of, row_token, err, ctas, s);
        if (ce != cudaSuccess && ctas > 1) {
            // a device that cannot place the cluster (SMs held elsewhere): one CTA does it all
            (void)cudaGetLastError();
            const int per1 = (int)((n + 32 * kPlanWarps - 1) / (32 * kPlanWarps));
            ce = pick(per1)(topk_idx, (int)n, c.k, c.E, cap, cnt_raw, off, slot_of, row_token, err, 1, s);
        }
        if (ce != cudaSuccess) return ce;
    } else {
        const int nchunks = (int)((n + kChunk - 1) / kChunk);
        const int blocks = (nchunks + kWarpsPerCta - 1) / kWarpsPerCta;
        const size_t smem = sizeof(int) * kWarpsPerCta * c.E;
        dispatch_count_kernel<<<blocks, 32 * kWarpsPerCta, smem, s>>>(topk_idx, n, c.E, nchunks, chunk_cnt);
        dispatch_scan_kernel<<<1, 256, 0, s>>>(chunk_cnt, nchunks, c.E, cap, cnt_raw, off);
        dispatch_rank_kernel<<<blocks, 32 * kWarpsPerCta, smem, s>>>(topk_idx, n, c.k, c.E, nchunks, chunk_cnt, off,
                                                                     cap, slot_of, row_token, err);
    }
    const int vecs = (row_bytes ? row_bytes : c.d * (c.dtype == MOE_F32 ? 4 : 2)) / 16;
    return launch_gather(x, vecs, row_token, off + c.E, n, x_perm, zero, s);
}

cudaError_t launch_dispatch_affinity(const moe_config &c, int32_t cap, const int32_t *topk_idx, const float *topk_w,
                                     const void *x, int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm,
                                     float *S, int32_t *kept, float *kept_w, int32_t *row_token, unsigned *err,
                                     cudaStream_t s, const GatherZero &zero, int row_bytes) {
    const int64_t n = (int64_t)c.T * c.k;
    cudaError_t ce = cudaMemsetAsync(S, 0, sizeof(float) * (size_t)c.E * c.T, s);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(cnt_raw, 0, sizeof(int32_t) * c.E, s);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(slot_of, 0xff, sizeof(int32_t) * (size_t)n, s);
    if (ce != cudaSuccess) return ce;
    int blocks = (int)((n + 255) / 256);
    if (blocks > num_sms() * 4) blocks = num_sms() * 4;
    affinity_scatter_kernel<<<blocks, 256, 0, s>>>(topk_idx, topk_w, n, c.k, c.T, c.E, S, cnt_raw, err);
    ce = launch_column_select(c, S, cap, cnt_raw, kept, kept_w, s);
    if (ce != cudaSuccess) return ce;
    affinity_rows_kernel<<<c.E, 256, 0, s>>>(kept, cnt_raw, cap, topk_idx, c.k, c.E, off, slot_of, row_token);
    const int vecs = (row_bytes ? row_bytes : c.d * (c.dtype == MOE_F32 ? 4 : 2)) / 16;
    return launch_gather(x, vecs, row_token, off + c.E, n, x_perm, zero, s);
}

cudaError_t launch_dispatch_ec(const moe_config &c, const int32_t *ec_tok, const void *x, int32_t *off,
                               int32_t *cnt_raw, int32_t *slot_of, void *x_perm, unsigned *err, cudaStream_t s,
                               int row_bytes) {
    const int64_t n = (int64_t)c.E * c.ec_capacity;
    cudaError_t ce = cudaMemsetAsync(slot_of, 0xff, sizeof(int32_t) * (size_t)c.T * c.E, s);
    if (ce != cudaSuccess) return ce;
    int blocks = (int)((n + 255) / 256);
    if (blocks > num_sms() * 4) blocks = num_sms() * 4;
    ec_slots_kernel<<<blocks, 256, 0, s>>>(ec_tok, c.T, c.E, c.ec_capacity, off, cnt_raw, slot_of, err);
    const int vecs = (row_bytes ? row_bytes : c.d * (c.dtype == MOE_F32 ? 4 : 2)) / 16;
    return launch_gather(x, vecs, ec_tok, nullptr, n, x_perm, GatherZero{}, s);
}

}  // namespace moe
