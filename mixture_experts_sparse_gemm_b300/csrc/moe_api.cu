// C ABI of the MoE layer: argument checks, workspace carving and the launch
// sequence route -> dispatch -> grouped experts -> combine.  Every argument check
// runs before any CUDA call, so a rejected call touches no device state.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "tc_common.cuh"

namespace moe {

// Device error word: bounded waits and index checks OR their bits in here.
__device__ unsigned g_moe_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s
constexpr uint64_t kMinWaitNs = 1000ull;             // 1 us
constexpr uint64_t kMaxWaitNs = 60000000000ull;      // 60 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
constexpr uint64_t kDefaultGroupBytes[2] = {40ull << 20, 64ull << 20};   // up, down
constexpr uint64_t kMaxGroupBytes = 1ull << 40;
std::atomic<uint64_t> g_group_bytes[2] = {kDefaultGroupBytes[0], kDefaultGroupBytes[1]};
int g_sm_count[kMaxDevices];
int g_arch_ok[kMaxDevices];   // 0 unknown, 1 sm_103, -1 other
unsigned *g_err_ptr[kMaxDevices];
std::mutex g_mu;

cudaError_t current_device(int &dev) {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    return cudaSuccess;
}

// Per-device set-up: SM count, architecture check, address of the error word.
moe_status device_setup(unsigned **err_ptr) {
    int dev = 0;
    if (current_device(dev) != cudaSuccess) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        g_sm_count[dev] = sms;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_arch_ok[dev] == 1) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_moe_error_word) != cudaSuccess) {
                g_arch_ok[dev] = 0;
                return MOE_ERR_CUDA;
            }
            g_err_ptr[dev] = static_cast<unsigned *>(p);
        }
    }
    if (g_arch_ok[dev] != 1) return MOE_ERR_UNSUPPORTED;
    if (err_ptr) *err_ptr = g_err_ptr[dev];
    return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- workspace layouts
struct Carver {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    }
};

struct RouteWs {
    size_t scores_t, wr_t, psum_rows, total;
};
RouteWs route_ws(const moe_config &c) {
    Carver k;
    RouteWs w{};
    w.scores_t = k.take(c.mode == MOE_EXPERT_CHOICE ? sizeof(float) * (size_t)c.E * c.T : 0);
    w.psum_rows = k.take(sizeof(float) * kPsumRows * (size_t)c.E);   // router score sums, see moe_route
    w.wr_t = k.take(bf16_acts(c) && route_tcgen05_supported(c) ? route_tcgen05_scratch_bytes(c) : 0);
    w.total = k.off;
    return w;
}

// the affinity-ordered capacity drop applies (token choice, a capacity limit)
bool affinity_drop(const moe_config &c) {
    return c.mode == MOE_TOKEN_CHOICE && c.drop_policy == MOE_DROP_AFFINITY && sizes_of(c).cap >= 0;
}

struct DispatchWs {
    size_t chunk, row_token, aff_S, aff_kept, aff_w, total;
};
DispatchWs dispatch_ws(const moe_config &c) {
    Carver k;
    DispatchWs w{};
    if (c.mode == MOE_TOKEN_CHOICE) {
        const int64_t n = (int64_t)c.T * c.k;
        const size_t ints = dispatch_tc_scratch_ints(n, c.E);
        w.chunk = k.take(sizeof(int32_t) * (ints - (size_t)n));
        w.row_token = k.take(sizeof(int32_t) * (size_t)n);
        if (affinity_drop(c)) {   // dense weights S[E][T], kept tokens and weights [E][cap]
            const size_t cap = (size_t)sizes_of(c).cap;
            w.aff_S = k.take(sizeof(float) * (size_t)c.E * c.T);
            w.aff_kept = k.take(sizeof(int32_t) * (size_t)c.E * cap);
            w.aff_w = k.take(sizeof(float) * (size_t)c.E * cap);
        }
    }
    w.total = k.off;
    return w;
}

// the two expert GEMMs run as one persistent launch when both use 256-wide tiles
bool ffn_fused(const moe_config &c) { return bf16_acts(c) && ffn_fused_supported(c); }

// FP8 up projection: aq / asc = E4M3 codes and scales of the x_perm rows (the
// grouped-FFN stage quantises its input), xq / xsc = those of the T token rows (the
// shared experts' input; in moe_forward also the rows the dispatch gathers).
struct FfnWs {
    size_t H, Hs, dep, aq, asc, xq, xsc, total;
};
FfnWs ffn_ws(const moe_config &c) {
    const Sizes z = sizes_of(c);
    Carver k;
    FfnWs w{};
    w.H = k.take((size_t)z.rows_routed * c.f * z.elt);
    w.Hs = k.take((size_t)(c.n_shared > 0 ? c.T : 0) * z.fs_tot * z.elt);
    w.dep = k.take(ffn_fused(c) ? sizeof(int) * ffn_dep_counters(c) : 0);
    const bool q = fp8_up(c);
    w.aq = k.take(q ? (size_t)z.rows_routed * c.d : 0);
    w.asc = k.take(q ? sizeof(float) * (size_t)z.rows_routed : 0);
    w.xq = k.take(q ? (size_t)c.T * c.d : 0);
    w.xsc = k.take(q ? sizeof(float) * (size_t)c.T : 0);
    w.total = k.off;
    return w;
}

struct ForwardWs {
    size_t idx, w, off, cnt_raw, slot_of, x_perm, Y, route, dispatch, ffn, total;
};
ForwardWs forward_ws(const moe_config &c) {
    const Sizes z = sizes_of(c);
    const size_t n_sel = c.mode == MOE_EXPERT_CHOICE ? (size_t)c.E * c.ec_capacity : (size_t)c.T * c.k;
    const size_t n_slot = c.mode == MOE_EXPERT_CHOICE ? (size_t)c.T * c.E : (size_t)c.T * c.k;
    Carver k;
    ForwardWs w{};
    w.idx = k.take(sizeof(int32_t) * n_sel);
    w.w = k.take(sizeof(float) * n_sel);
    w.off = k.take(sizeof(int32_t) * (c.E + 1));
    w.cnt_raw = k.take(sizeof(int32_t) * c.E);
    w.slot_of = k.take(sizeof(int32_t) * n_slot);
    w.x_perm = k.take((size_t)z.rows_routed * c.d * z.elt);
    w.Y = k.take((size_t)z.rows_total * c.d * z.elt);
    w.route = k.take(route_ws(c).total);
    w.dispatch = k.take(dispatch_ws(c).total);
    w.ffn = k.take(ffn_ws(c).total);
    w.total = k.off;
    return w;
}

// ---------------------------------------------------------------- stage bodies (validated input)
// prob_sum (nullable): the router CTAs add their score sums into kPsumRows rows of
// the workspace (row = CTA index mod kPsumRows, so few CTAs share an address),
// then one small kernel sums the rows in order into prob_sum[E].
moe_status do_route(const moe_config &c, const void *x, const void *W_r, const float *lo, const float *sb,
                    int32_t *idx, float *w, char *ws, unsigned *err, cudaStream_t s, float *prob_sum = nullptr) {
    const RouteWs L = route_ws(c);
    float *scores_t = c.mode == MOE_EXPERT_CHOICE ? reinterpret_cast<float *>(ws + L.scores_t) : nullptr;
    float *rows = prob_sum ? reinterpret_cast<float *>(ws + L.psum_rows) : nullptr;
    cudaError_t e;
    if (rows && cudaMemsetAsync(rows, 0, sizeof(float) * kPsumRows * (size_t)c.E, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (bf16_acts(c) && route_tcgen05_supported(c))
        e = launch_route_tcgen05(c, x, W_r, lo, sb, idx, w, scores_t, rows, ws + L.wr_t, err, s);
    else
        e = launch_route_simt(c, x, W_r, lo, sb, idx, w, scores_t, rows, err, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (rows && launch_sum_psum_rows(c, rows, prob_sum, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (c.mode == MOE_EXPERT_CHOICE) return from_cuda(launch_ec_select(c, scores_t, idx, w, s));
    return MOE_OK;
}

// row_bytes: bytes of a row of x (0: d in the activation type; E4M3 rows: d)
moe_status do_dispatch(const moe_config &c, const int32_t *idx, const float *topk_w, const void *x, int32_t *off,
                       int32_t *cnt_raw, int32_t *slot_of, void *x_perm, char *ws, unsigned *err, cudaStream_t s,
                       const GatherZero &zero = GatherZero{}, int row_bytes = 0) {
    if (c.mode == MOE_EXPERT_CHOICE)
        return from_cuda(launch_dispatch_ec(c, idx, x, off, cnt_raw, slot_of, x_perm, err, s, row_bytes));
    const DispatchWs L = dispatch_ws(c);
    const Sizes z = sizes_of(c);
    if (affinity_drop(c))
        return from_cuda(launch_dispatch_affinity(
            c, z.cap, idx, topk_w, x, off, cnt_raw, slot_of, x_perm, reinterpret_cast<float *>(ws + L.aff_S),
            reinterpret_cast<int32_t *>(ws + L.aff_kept), reinterpret_cast<float *>(ws + L.aff_w),
            reinterpret_cast<int32_t *>(ws + L.row_token), err, s, zero, row_bytes));
    return from_cuda(launch_dispatch_tc(c, z.cap, idx, x, off, cnt_raw, slot_of, x_perm,
                                        reinterpret_cast<int32_t *>(ws + L.chunk),
                                        reinterpret_cast<int32_t *>(ws + L.row_token), err, s, zero, row_bytes));
}

moe_status do_ffn(const moe_config &c, const void *x_perm, const int32_t *off, const void *packed, const void *x,
                  void *Y, char *ws, unsigned *err, cudaStream_t s) {
    const FfnWs L = ffn_ws(c);
    const Sizes z = sizes_of(c);
    void *H = ws + L.H;
    void *Hs = ws + L.Hs;
    if (fp8_up(c)) {
        // quantise the rows to E4M3 per row, then the fused launch on them
        uint8_t *aq = reinterpret_cast<uint8_t *>(ws + L.aq), *xq = reinterpret_cast<uint8_t *>(ws + L.xq);
        float *asc = reinterpret_cast<float *>(ws + L.asc), *xsc = reinterpret_cast<float *>(ws + L.xsc);
        if (launch_quantize_rows(x_perm, z.rows_routed, c.d, aq, asc, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (c.n_shared > 0 && launch_quantize_rows(x, c.T, c.d, xq, xsc, s) != cudaSuccess) return MOE_ERR_CUDA;
        F8Rows f8;
        f8.rs0 = asc;
        f8.rs1 = xsc;
        return from_cuda(launch_ffn_fused_tcgen05(c, z, aq, off, packed, c.n_shared > 0 ? xq : nullptr, H, Hs, Y,
                                                  reinterpret_cast<int *>(ws + L.dep), err, s, nullptr, nullptr,
                                                  false, &f8));
    }
    if (ffn_fused(c))
        return from_cuda(launch_ffn_fused_tcgen05(c, z, x_perm, off, packed, x, H, Hs, Y,
                                                  reinterpret_cast<int *>(ws + L.dep), err, s));
    cudaError_t e = bf16_acts(c) ? launch_ffn_up_tcgen05(c, z, x_perm, off, packed, x, H, Hs, err, s)
                                          : launch_ffn_up_simt(c, z, x_perm, off, packed, x, H, Hs, s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = bf16_acts(c) ? launch_ffn_down_tcgen05(c, z, H, Hs, off, packed, Y, err, s)
                              : launch_ffn_down_simt(c, z, H, Hs, off, packed, Y, s);
    return from_cuda(e);
}

// kernels enqueued per stage; mirrors the launch sequence of the do_* bodies above
int ffn_launches(const moe_config &c) {
    if (fp8_up(c)) return 1 + (c.n_shared > 0 ? 1 : 0) + 1;   // quantise x_perm (and x), fused launch
    return ffn_fused(c) ? 1 : 2;
}
int route_launches(const moe_config &c) {
    const int base = (bf16_acts(c) && route_tcgen05_supported(c)) ? route_tcgen05_launches(c) : 1;
    return base + (c.mode == MOE_EXPERT_CHOICE ? 1 : 0);
}
int dispatch_launches(const moe_config &c) {
    if (affinity_drop(c)) return 4;   // scatter, column select, rows, gather
    return c.mode == MOE_EXPERT_CHOICE ? 2 : dispatch_tc_launches((int64_t)c.T * c.k);
}

// moe_forward folds the combine into the down GEMM when every token has one
// expert and there are no shared experts (the row -> token map is a permutation)
bool gated_down(const moe_config &c) {
    return bf16_acts(c) && c.mode == MOE_TOKEN_CHOICE && c.k == 1 && c.n_shared == 0;
}

}  // namespace

// ---------------------------------------------------------------- internal shared helpers
Sizes sizes_of(const moe_config &c) {
    Sizes z{};
    z.elt = c.dtype == MOE_F32 ? 4 : 2;
    z.fs_tot = c.n_shared > 0 ? c.n_shared * c.f_shared : 0;
    if (c.mode == MOE_EXPERT_CHOICE) {
        z.rows_routed = (int64_t)c.E * c.ec_capacity;
        z.cap = c.ec_capacity;
    } else {
        z.rows_routed = (int64_t)c.T * c.k;
        z.cap = c.capacity_factor > 0.f
                    ? (int32_t)std::floor((double)c.capacity_factor * (double)c.T * (double)c.k / (double)c.E)
                    : -1;
    }
    z.rows_total = z.rows_routed + (c.n_shared > 0 ? c.T : 0);
    return z;
}

PackedLayout packed_layout(const moe_config &c) {
    const Sizes z = sizes_of(c);
    Carver k;
    PackedLayout L{};
    const size_t we = fp8_weights(c) ? 1 : z.elt;   // bytes per stored weight
    const size_t we13 = (fp8_weights(c) || fp8_up(c)) ? 1 : z.elt;   // the up projection's
    L.w13 = k.take((size_t)c.E * 2 * c.f * c.d * we13);
    L.w2 = k.take((size_t)c.E * c.d * c.f * we);
    L.w13s = k.take((size_t)2 * z.fs_tot * c.d * we13);
    L.w2s = k.take((size_t)c.d * z.fs_tot * we);
    const bool sc = fp8_weights(c), sc13 = sc || fp8_up(c);
    L.sc13 = k.take(sc13 ? sizeof(float) * (size_t)c.E * 2 * c.f : 0);
    L.sc2 = k.take(sc ? sizeof(float) * (size_t)c.E * c.d : 0);
    L.sc13s = k.take(sc13 ? sizeof(float) * (size_t)2 * z.fs_tot : 0);
    L.sc2s = k.take(sc ? sizeof(float) * (size_t)c.d : 0);
    L.total = k.off;
    return L;
}

moe_status device_ready(unsigned **err_word) { return device_setup(err_word); }

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

uint64_t tile_group_bytes(int down) { return g_group_bytes[down ? 1 : 0].load(std::memory_order_relaxed); }

int num_sms() {
    int dev = 0;
    if (current_device(dev) != cudaSuccess || g_sm_count[dev] <= 0) return 148;
    return g_sm_count[dev];
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tmap_encoder() {
    static EncodeTiledFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return encode;
}
}  // namespace

bool make_tmap_u8(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const EncodeTiledFn encode = tmap_encoder();
    if (!encode) return false;
    if (rows == 0) rows = 1;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        encode = reinterpret_cast<EncodeFn>(fn);
    }
    if (rows == 0) rows = 1;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status moe_validate_config(const moe_config *cfg) {
    if (!cfg) return MOE_ERR_INVALID_ARG;
    const moe_config &c = *cfg;
    if (c.T < 0 || c.d <= 0 || c.f <= 0 || c.E <= 0) return MOE_ERR_INVALID_ARG;
    if (c.gate != MOE_GATE_SOFTMAX && c.gate != MOE_GATE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (c.mode != MOE_TOKEN_CHOICE && c.mode != MOE_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (c.dtype != MOE_F32 && c.dtype != MOE_BF16 && c.dtype != MOE_BF16_FP8W && c.dtype != MOE_BF16_FP8UP)
        return MOE_ERR_INVALID_ARG;
    if (c.drop_policy != MOE_DROP_TOKEN_ORDER && c.drop_policy != MOE_DROP_AFFINITY) return MOE_ERR_INVALID_ARG;
    if (c.n_shared < 0 || (c.n_shared > 0 && c.f_shared <= 0)) return MOE_ERR_INVALID_ARG;
    if (std::isnan(c.capacity_factor)) return MOE_ERR_INVALID_ARG;
    if (c.E > kMaxE) return MOE_ERR_UNSUPPORTED;
    if (c.mode == MOE_TOKEN_CHOICE) {
        if (c.k <= 0 || c.k > c.E) return MOE_ERR_INVALID_ARG;
        if (c.k > kMaxK) return MOE_ERR_UNSUPPORTED;
        if ((int64_t)c.T * c.k > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    } else {
        if (c.ec_capacity <= 0 || (c.T > 0 && c.ec_capacity > c.T)) return MOE_ERR_INVALID_ARG;
        if (c.gate != MOE_GATE_SOFTMAX) return MOE_ERR_UNSUPPORTED;
        if ((int64_t)c.T * c.E > INT32_MAX || (int64_t)c.E * c.ec_capacity > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    }
    const int64_t fs = c.n_shared > 0 ? (int64_t)c.n_shared * c.f_shared : 0;
    if (fs > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (c.dtype == MOE_BF16) {
        if (c.d % 128 != 0 || c.f % 64 != 0 || fs % 64 != 0) return MOE_ERR_UNSUPPORTED;
    } else if (c.dtype == MOE_BF16_FP8W || c.dtype == MOE_BF16_FP8UP) {   // 256-wide tiles (one fused launch)
        if (c.d % 256 != 0 || c.f % 128 != 0 || fs % 128 != 0) return MOE_ERR_UNSUPPORTED;
    } else {
        if (c.d % 64 != 0 || c.f % 64 != 0 || fs % 64 != 0) return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

moe_status moe_expert_capacity(const moe_config *cfg, int32_t *cap) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!cap) return MOE_ERR_INVALID_ARG;
    *cap = sizes_of(*cfg).cap;
    return MOE_OK;
}

moe_status moe_buffer_rows(const moe_config *cfg, int64_t *rows_routed, int64_t *rows_total) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const Sizes z = sizes_of(*cfg);
    if (rows_routed) *rows_routed = z.rows_routed;
    if (rows_total) *rows_total = z.rows_total;
    return MOE_OK;
}

moe_status moe_workspace_size(const moe_config *cfg, moe_stage stage, size_t *bytes) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    switch (stage) {
        case MOE_STAGE_ROUTE: *bytes = route_ws(*cfg).total; break;
        case MOE_STAGE_DISPATCH: *bytes = dispatch_ws(*cfg).total; break;
        case MOE_STAGE_GROUPED_FFN: *bytes = ffn_ws(*cfg).total; break;
        case MOE_STAGE_COMBINE: *bytes = 0; break;
        case MOE_STAGE_FORWARD: *bytes = forward_ws(*cfg).total; break;
        default: return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

moe_status moe_packed_weights_size(const moe_config *cfg, size_t *bytes) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = packed_layout(*cfg).total;
    return MOE_OK;
}

#define MOE_REQUIRE(cond, code) \
    do {                        \
        if (!(cond)) return code; \
    } while (0)

static moe_status check_ws(const void *ws, size_t ws_bytes, size_t need) {
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    if (need > 0 && !ws) return MOE_ERR_INVALID_ARG;
    if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

moe_status moe_pack_weights(const moe_config *cfg, const void *W1, const void *W3, const void *W2, const void *W1s,
                            const void *W3s, const void *W2s, void *packed, size_t packed_bytes, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(W1 && W3 && W2 && packed, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.n_shared == 0 || (W1s && W3s && W2s), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(packed_bytes >= packed_layout(c).total, MOE_ERR_WORKSPACE);
    MOE_REQUIRE(aligned16(W1) && aligned16(W3) && aligned16(W2) && aligned16(packed), MOE_ERR_MISALIGNED);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(packed) & 255u) == 0, MOE_ERR_MISALIGNED);
    st = device_setup(nullptr);
    if (st != MOE_OK) return st;
    return from_cuda(launch_pack(c, W1, W3, W2, W1s, W3s, W2s, packed, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const moe_config *cfg, const void *x, const void *W_r, const float *logit_offset,
                     const float *sel_bias, int32_t *topk_idx, float *topk_w, float *prob_sum, void *ws,
                     size_t ws_bytes, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(x && W_r && topk_idx && topk_w, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.mode == MOE_TOKEN_CHOICE || !sel_bias, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(x) && aligned16(W_r), MOE_ERR_MISALIGNED);
    MOE_REQUIRE(aligned4(topk_idx) && aligned4(topk_w) && aligned4(logit_offset) && aligned4(sel_bias) &&
                    aligned4(prob_sum),
                MOE_ERR_MISALIGNED);
    st = check_ws(ws, ws_bytes, route_ws(c).total);
    if (st != MOE_OK) return st;
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c.T == 0) {   // no tokens: zero score sums
        if (prob_sum && cudaMemsetAsync(prob_sum, 0, sizeof(float) * c.E, s) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    return do_route(c, x, W_r, logit_offset, sel_bias, topk_idx, topk_w, static_cast<char *>(ws), err, s, prob_sum);
}

moe_status moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const float *topk_w, const void *x,
                        int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm, void *ws, size_t ws_bytes,
                        void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(topk_idx && x && off && cnt_raw && slot_of && x_perm, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(topk_w || !affinity_drop(c), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(x) && aligned16(x_perm), MOE_ERR_MISALIGNED);
    MOE_REQUIRE(aligned4(topk_idx) && aligned4(off) && aligned4(cnt_raw) && aligned4(slot_of) && aligned4(topk_w),
                MOE_ERR_MISALIGNED);
    st = check_ws(ws, ws_bytes, dispatch_ws(c).total);
    if (st != MOE_OK) return st;
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c.T == 0) {   // empty batch: every expert segment is empty
        if (cudaMemsetAsync(off, 0, sizeof(int32_t) * (c.E + 1), s) != cudaSuccess ||
            cudaMemsetAsync(cnt_raw, 0, sizeof(int32_t) * c.E, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    return do_dispatch(c, topk_idx, topk_w, x, off, cnt_raw, slot_of, x_perm, static_cast<char *>(ws), err, s);
}

moe_status moe_grouped_ffn(const moe_config *cfg, const void *x_perm, const int32_t *off, const void *packed,
                           const void *x, void *Y, void *ws, size_t ws_bytes, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(x_perm && off && packed && Y, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.n_shared == 0 || x, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(x_perm) && aligned16(Y) && aligned16(x) && aligned4(off), MOE_ERR_MISALIGNED);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(packed) & 255u) == 0, MOE_ERR_MISALIGNED);
    st = check_ws(ws, ws_bytes, ffn_ws(c).total);
    if (st != MOE_OK) return st;
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK || c.T == 0) return st;
    return do_ffn(c, x_perm, off, packed, x, Y, static_cast<char *>(ws), err, static_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_ffn_up(const moe_config *cfg, const void *x_perm, const int32_t *off, const void *packed,
                              const void *x, void *H, void *Hs, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(!fp8_up(c), MOE_ERR_UNSUPPORTED);   // needs a workspace for its E4M3 rows
    MOE_REQUIRE(x_perm && off && packed && H, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.n_shared == 0 || (x && Hs), MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(x_perm) && aligned16(x) && aligned16(H) && aligned16(Hs) && aligned4(off),
                MOE_ERR_MISALIGNED);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(packed) & 255u) == 0, MOE_ERR_MISALIGNED);
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK || c.T == 0) return st;
    const Sizes z = sizes_of(c);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(bf16_acts(c) ? launch_ffn_up_tcgen05(c, z, x_perm, off, packed, x, H, Hs, err, s)
                                         : launch_ffn_up_simt(c, z, x_perm, off, packed, x, H, Hs, s));
}

moe_status moe_grouped_ffn_down(const moe_config *cfg, const void *H, const void *Hs, const int32_t *off,
                                const void *packed, void *Y, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(!fp8_up(c), MOE_ERR_UNSUPPORTED);   // the halves of the FP8 layer run fused
    MOE_REQUIRE(H && off && packed && Y, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.n_shared == 0 || Hs, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(H) && aligned16(Hs) && aligned16(Y) && aligned4(off), MOE_ERR_MISALIGNED);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(packed) & 255u) == 0, MOE_ERR_MISALIGNED);
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK || c.T == 0) return st;
    const Sizes z = sizes_of(c);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(bf16_acts(c) ? launch_ffn_down_tcgen05(c, z, H, Hs, off, packed, Y, err, s)
                                         : launch_ffn_down_simt(c, z, H, Hs, off, packed, Y, s));
}

moe_status moe_launch_count(const moe_config *cfg, moe_stage stage, int32_t *kernels) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!kernels) return MOE_ERR_INVALID_ARG;
    const moe_config &c = *cfg;
    const int empty = c.T == 0;
    switch (stage) {
        case MOE_STAGE_ROUTE: *kernels = empty ? 0 : route_launches(c); break;
        case MOE_STAGE_DISPATCH: *kernels = empty ? 0 : dispatch_launches(c); break;
        case MOE_STAGE_GROUPED_FFN: *kernels = empty ? 0 : ffn_launches(c); break;
        case MOE_STAGE_COMBINE: *kernels = empty ? 0 : 1; break;
        case MOE_STAGE_FORWARD:
            // the FP8 up projection quantises x once (before the dispatch gathers its rows)
            *kernels = empty ? 0
                             : route_launches(c) + dispatch_launches(c) + (fp8_up(c) ? 2 : (ffn_fused(c) ? 1 : 2)) +
                                   (gated_down(c) ? 0 : 1);
            break;
        default: return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

moe_status moe_load_stats(const moe_config *cfg, const int32_t *topk_idx, const int32_t *cnt_raw,
                          const float *prob_sum, float *token_fraction, float *prob_mean, double *summary,
                          void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(topk_idx && cnt_raw && prob_sum && token_fraction && prob_mean && summary, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned4(topk_idx) && aligned4(cnt_raw) && aligned4(prob_sum) && aligned4(token_fraction) &&
                    aligned4(prob_mean) && (reinterpret_cast<uintptr_t>(summary) & 7u) == 0,
                MOE_ERR_MISALIGNED);
    st = device_setup(nullptr);
    if (st != MOE_OK || c.T == 0) return st;
    return from_cuda(launch_load_stats(c, topk_idx, cnt_raw, prob_sum, token_fraction, prob_mean, summary,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const moe_config *cfg, const void *Y, const int32_t *slot_of, const float *topk_w, void *y,
                       void *ws, size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(Y && slot_of && topk_w && y, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(Y) && aligned16(y) && aligned4(slot_of) && aligned4(topk_w), MOE_ERR_MISALIGNED);
    st = device_setup(nullptr);
    if (st != MOE_OK || c.T == 0) return st;
    return from_cuda(launch_combine(c, sizes_of(c), Y, slot_of, topk_w, y, static_cast<cudaStream_t>(stream)));
}

moe_status moe_forward(const moe_config *cfg, const void *x, const void *W_r, const float *logit_offset,
                       const float *sel_bias, const void *packed, void *y, void *ws, size_t ws_bytes, void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    MOE_REQUIRE(x && W_r && packed && y, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(c.mode == MOE_TOKEN_CHOICE || !sel_bias, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned16(x) && aligned16(W_r) && aligned16(y), MOE_ERR_MISALIGNED);
    MOE_REQUIRE(aligned4(logit_offset) && aligned4(sel_bias), MOE_ERR_MISALIGNED);
    MOE_REQUIRE((reinterpret_cast<uintptr_t>(packed) & 255u) == 0, MOE_ERR_MISALIGNED);
    const ForwardWs L = forward_ws(c);
    st = check_ws(ws, ws_bytes, L.total);
    if (st != MOE_OK) return st;
    unsigned *err = nullptr;
    st = device_setup(&err);
    if (st != MOE_OK || c.T == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *w = static_cast<char *>(ws);
    int32_t *idx = reinterpret_cast<int32_t *>(w + L.idx);
    float *gw = reinterpret_cast<float *>(w + L.w);
    int32_t *off = reinterpret_cast<int32_t *>(w + L.off);
    int32_t *cnt_raw = reinterpret_cast<int32_t *>(w + L.cnt_raw);
    int32_t *slot_of = reinterpret_cast<int32_t *>(w + L.slot_of);
    void *x_perm = w + L.x_perm;
    void *Y = w + L.Y;
    st = do_route(c, x, W_r, logit_offset, sel_bias, idx, gw, w + L.route, err, s);
    if (st != MOE_OK) return st;
    if (fp8_up(c)) {
        // the tokens to E4M3 once: the dispatch gathers their codes into x_perm and the
        // shared experts read them; the up tiles look up each row's scale by its token
        const Sizes z = sizes_of(c);
        const FfnWs F = ffn_ws(c);
        uint8_t *xq = reinterpret_cast<uint8_t *>(w + L.ffn + F.xq);
        float *xsc = reinterpret_cast<float *>(w + L.ffn + F.xsc);
        int *dep = reinterpret_cast<int *>(w + L.ffn + F.dep);
        if (launch_quantize_rows(x, c.T, c.d, xq, xsc, s) != cudaSuccess) return MOE_ERR_CUDA;
        const int32_t *row_token = c.mode == MOE_EXPERT_CHOICE
                                       ? idx
                                       : reinterpret_cast<const int32_t *>(w + L.dispatch + dispatch_ws(c).row_token);
        const bool gated = gated_down(c);
        GatherZero zero;
        if (gated) {
            zero.slot_of = slot_of;
            zero.T = c.T;
            zero.y = static_cast<uint4 *>(y);
            zero.y_vecs = c.d * 2 / 16;
            zero.dep = dep;
            zero.ndep = (int)ffn_dep_counters(c);
        }
        st = do_dispatch(c, idx, gw, xq, off, cnt_raw, slot_of, x_perm, w + L.dispatch, err, s, zero, c.d);
        if (st != MOE_OK) return st;
        F8Rows f8;
        f8.rs0 = xsc;
        f8.rtok0 = row_token;
        f8.rs1 = xsc;
        if (gated)
            return from_cuda(launch_ffn_fused_tcgen05(c, z, x_perm, off, packed, xq, w + L.ffn + F.H, nullptr, y, dep,
                                                      err, s, row_token, gw, /*dep_zeroed=*/true, &f8));
        if (launch_ffn_fused_tcgen05(c, z, x_perm, off, packed, c.n_shared > 0 ? xq : nullptr, w + L.ffn + F.H,
                                     w + L.ffn + F.Hs, Y, dep, err, s, nullptr, nullptr, false, &f8) != cudaSuccess)
            return MOE_ERR_CUDA;
        return from_cuda(launch_combine(c, z, Y, slot_of, gw, y, s));
    }
    if (gated_down(c)) {
        // one expert per token and no shared experts: the down GEMM writes each kept
        // row straight to its token's output, scaled by the gate; the dispatch gather
        // zeroes the output rows of dropped tokens (and the fused launch's counters)
        const Sizes z = sizes_of(c);
        const FfnWs F = ffn_ws(c);
        const int32_t *row_token = reinterpret_cast<const int32_t *>(w + L.dispatch + dispatch_ws(c).row_token);
        const bool fused = ffn_fused(c);
        GatherZero zero;
        zero.slot_of = slot_of;
        zero.T = c.T;
        zero.y = static_cast<uint4 *>(y);
        zero.dep = fused ? reinterpret_cast<int *>(w + L.ffn + F.dep) : nullptr;
        zero.ndep = fused ? (int)ffn_dep_counters(c) : 0;
        st = do_dispatch(c, idx, gw, x, off, cnt_raw, slot_of, x_perm, w + L.dispatch, err, s, zero);
        if (st != MOE_OK) return st;
        if (fused)
            return from_cuda(launch_ffn_fused_tcgen05(c, z, x_perm, off, packed, x, w + L.ffn + F.H, nullptr, y,
                                                      reinterpret_cast<int *>(w + L.ffn + F.dep), err, s, row_token,
                                                      gw, /*dep_zeroed=*/true));
        cudaError_t e = launch_ffn_up_tcgen05(c, z, x_perm, off, packed, x, w + L.ffn + F.H, nullptr, err, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        return from_cuda(launch_ffn_down_tcgen05(c, z, w + L.ffn + F.H, nullptr, off, packed, y, err, s, row_token,
                                                 gw));
    }
    st = do_dispatch(c, idx, gw, x, off, cnt_raw, slot_of, x_perm, w + L.dispatch, err, s);
    if (st != MOE_OK) return st;
    st = do_ffn(c, x_perm, off, packed, x, Y, w + L.ffn, err, s);
    if (st != MOE_OK) return st;
    return from_cuda(launch_combine(c, sizes_of(c), Y, slot_of, gw, y, s));
}

moe_status moe_set_wait_limit_ns(uint64_t limit_ns) {
    if (limit_ns == 0) limit_ns = kDefaultWaitNs;
    if (limit_ns < kMinWaitNs || limit_ns > kMaxWaitNs) return MOE_ERR_INVALID_ARG;
    g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed);
    return MOE_OK;
}

moe_status moe_set_tile_group_bytes(uint64_t up_bytes, uint64_t down_bytes) {
    if (up_bytes > kMaxGroupBytes || down_bytes > kMaxGroupBytes) return MOE_ERR_INVALID_ARG;
    g_group_bytes[0].store(up_bytes ? up_bytes : kDefaultGroupBytes[0], std::memory_order_relaxed);
    g_group_bytes[1].store(down_bytes ? down_bytes : kDefaultGroupBytes[1], std::memory_order_relaxed);
    return MOE_OK;
}

moe_status moe_get_tile_group_bytes(uint64_t *up_bytes, uint64_t *down_bytes) {
    if (!up_bytes || !down_bytes) return MOE_ERR_INVALID_ARG;
    *up_bytes = tile_group_bytes(0);
    *down_bytes = tile_group_bytes(1);
    return MOE_OK;
}

moe_status moe_get_wait_limit_ns(uint64_t *limit_ns) {
    if (!limit_ns) return MOE_ERR_INVALID_ARG;
    *limit_ns = wait_limit_ns();
    return MOE_OK;
}

moe_status moe_wait_probe(const int32_t *flag, int32_t target, void *stream) {
    MOE_REQUIRE(flag, MOE_ERR_INVALID_ARG);
    MOE_REQUIRE(aligned4(flag), MOE_ERR_MISALIGNED);
    unsigned *err = nullptr;
    moe_status st = device_setup(&err);
    if (st != MOE_OK) return st;
    return from_cuda(launch_wait_probe(flag, target, wait_limit_ns(), err, static_cast<cudaStream_t>(stream)));
}

moe_status moe_check_device_error(void *stream) {
    unsigned *err = nullptr;
    moe_status st = device_setup(&err);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (host == 0) return MOE_OK;
    if (cudaMemsetAsync(err, 0, sizeof(unsigned), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return (host & kErrWaitTimeout) ? MOE_ERR_TIMEOUT : MOE_ERR_INVALID_ARG;
}

}  // extern "C"
