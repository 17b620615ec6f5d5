// moe_dispatch_noalloc: the capacity-limited dispatch for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin inside a
// host framework that owns every device allocation and passes in only the
// layer's input and output buffers, or a latency-critical serving loop where a
// cudaMalloc could synchronise the device and stall every stream.  For them this
// entry point runs the same kernels as moe_dispatch, with the scratch those
// kernels need (per-chunk expert counts and the row -> token table) taken from a
// fixed array compiled into the library instead of from `ws`.
//
// The array holds kNoAllocScratchInts int32 (512 KiB) on every GPU that loads the
// library, for the life of the process.  It bounds a call to
// MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS token-choice assignments (T * k); larger
// calls are rejected with MOE_ERR_UNSUPPORTED before anything is launched.
// Expert Choice dispatch needs no scratch and runs as in moe_dispatch.
//
// The first call on each device looks up the array's device address there
// (cudaGetSymbolAddress) and keeps it; make that first call before any stream
// capture.
//
// All calls share the one array and it keeps the previous call's contents.  The
// kernels overwrite every entry they read before reading it (each chunk's counts
// and every kept row's token), so nothing needs clearing between calls.  Calls
// whose work overlaps on the GPU -- on different streams, or from different host
// threads -- race on the array and give wrong results; serialise them.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int64_t kNoAllocMaxAssignments = MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS;
constexpr size_t kNoAllocScratchInts = 131072;   // >= dispatch_tc_scratch_ints(65536, 256)
static_assert(kNoAllocMaxAssignments == 65536, "scratch size is derived for 65536 assignments");

static __device__ __align__(256) int32_t g_noalloc_dispatch_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
int32_t *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
moe_status scratch_address(int32_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                                           int32_t *off, int32_t *cnt_raw, int32_t *slot_of, void *x_perm,
                                           void *stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (!topk_idx || !x || !off || !cnt_raw || !slot_of || !x_perm) return MOE_ERR_INVALID_ARG;
    if (c.mode == MOE_TOKEN_CHOICE && c.drop_policy == MOE_DROP_AFFINITY && c.capacity_factor > 0.f)
        return MOE_ERR_UNSUPPORTED;   // the affinity order needs the gate weights and a workspace
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x_perm);
    const uintptr_t a4 = reinterpret_cast<uintptr_t>(topk_idx) | reinterpret_cast<uintptr_t>(off) |
                         reinterpret_cast<uintptr_t>(cnt_raw) | reinterpret_cast<uintptr_t>(slot_of);
    if ((a16 & 15u) || (a4 & 3u)) return MOE_ERR_MISALIGNED;
    const int64_t n = (c.mode == MOE_TOKEN_CHOICE) ? (int64_t)c.T * c.k : 0;
    if (n > kNoAllocMaxAssignments) return MOE_ERR_UNSUPPORTED;
    if (dispatch_tc_scratch_ints(n, c.E) > kNoAllocScratchInts) return MOE_ERR_UNSUPPORTED;
    unsigned *err = nullptr;
    st = device_ready(&err);
    if (st != MOE_OK) return st;
    int32_t *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (c.T == 0) {
        if (cudaMemsetAsync(off, 0, sizeof(int32_t) * (c.E + 1), s) != cudaSuccess ||
            cudaMemsetAsync(cnt_raw, 0, sizeof(int32_t) * c.E, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    cudaError_t e;
    if (c.mode == MOE_EXPERT_CHOICE) {
        e = launch_dispatch_ec(c, topk_idx, x, off, cnt_raw, slot_of, x_perm, err, s);
    } else {
        const Sizes z = sizes_of(c);
        const size_t chunk_ints = dispatch_tc_scratch_ints(n, c.E) - (size_t)n;
        e = launch_dispatch_tc(c, z.cap, topk_idx, x, off, cnt_raw, slot_of, x_perm, scratch, scratch + chunk_ints,
                               err, s);
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
