"""ctypes binding of the C ABI in include/moe_b300.h.

Argument marshalling only: every function forwards to the entry point of the same
name in libmoe_b300.so, passing raw device pointers (torch tensors are accepted
and their data_ptr() is passed) and the current torch CUDA stream.  All compute
happens in the library's CUDA kernels; there is no other code path.  A missing or
unloadable library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_MISALIGNED = 0, 1, 2, 3
MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_GATE_SOFTMAX, MOE_GATE_SIGMOID = 0, 1
MOE_TOKEN_CHOICE, MOE_EXPERT_CHOICE = 0, 1
MOE_F32, MOE_BF16, MOE_BF16_FP8W, MOE_BF16_FP8UP = 0, 1, 2, 3
MOE_DROP_TOKEN_ORDER, MOE_DROP_AFFINITY = 0, 1
MOE_STAGE_ROUTE, MOE_STAGE_DISPATCH, MOE_STAGE_GROUPED_FFN, MOE_STAGE_COMBINE, MOE_STAGE_FORWARD = range(5)

EXPORTS = ("moe_status_string", "moe_validate_config", "moe_expert_capacity", "moe_buffer_rows",
           "moe_workspace_size", "moe_packed_weights_size", "moe_pack_weights", "moe_route", "moe_dispatch",
           "moe_grouped_ffn", "moe_grouped_ffn_up", "moe_grouped_ffn_down", "moe_combine", "moe_forward",
           "moe_launch_count", "moe_check_device_error", "moe_dispatch_noalloc", "moe_load_stats",
           "moe_set_wait_limit_ns", "moe_get_wait_limit_ns", "moe_wait_probe", "moe_set_tile_group_bytes",
           "moe_get_tile_group_bytes")
MOE_DISPATCH_NOALLOC_MAX_ASSIGNMENTS = 65536


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("f", ctypes.c_int32),
                ("k", ctypes.c_int32), ("gate", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
                ("ec_capacity", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("f_shared", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("drop_policy", ctypes.c_int32)]


_lib = None


def lib():
    """Load libmoe_b300.so (build it first with mixture_experts_sparse_gemm_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run `python -m mixture_experts_sparse_gemm_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, cfgp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(moe_config)
        i32p, i64p, szp = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_size_t)
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        sigs = {
            "moe_validate_config": [cfgp],
            "moe_expert_capacity": [cfgp, i32p],
            "moe_buffer_rows": [cfgp, i64p, i64p],
            "moe_workspace_size": [cfgp, ctypes.c_int, szp],
            "moe_packed_weights_size": [cfgp, szp],
            "moe_pack_weights": [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_route": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_dispatch": [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_grouped_ffn": [cfgp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_grouped_ffn_up": [cfgp, vp, vp, vp, vp, vp, vp, vp],
            "moe_grouped_ffn_down": [cfgp, vp, vp, vp, vp, vp, vp],
            "moe_launch_count": [cfgp, ctypes.c_int, i32p],
            "moe_combine": [cfgp, vp, vp, vp, vp, vp, sz, vp],
            "moe_forward": [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
            "moe_check_device_error": [vp],
            "moe_dispatch_noalloc": [cfgp, vp, vp, vp, vp, vp, vp, vp],
            "moe_load_stats": [cfgp, vp, vp, vp, vp, vp, vp, vp],
            "moe_set_wait_limit_ns": [ctypes.c_uint64],
            "moe_get_wait_limit_ns": [ctypes.POINTER(ctypes.c_uint64)],
            "moe_set_tile_group_bytes": [ctypes.c_uint64, ctypes.c_uint64],
            "moe_get_tile_group_bytes": [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)],
            "moe_wait_probe": [vp, ctypes.c_int32, vp],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _p(t):
    """Device pointer of a tensor (or an int address, or None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def config(T, d, E, f, k=1, gate="softmax", mode="tc", renormalize=True, capacity_factor=0.0, ec_capacity=0,
           n_shared=0, f_shared=0, dtype="bf16", drop_policy="token") -> moe_config:
    return moe_config(T, d, E, f, k, MOE_GATE_SIGMOID if gate == "sigmoid" else MOE_GATE_SOFTMAX,
                      MOE_EXPERT_CHOICE if mode == "ec" else MOE_TOKEN_CHOICE, int(bool(renormalize)),
                      float(capacity_factor), int(ec_capacity), int(n_shared), int(f_shared),
                      _DTYPES[dtype], MOE_DROP_AFFINITY if drop_policy == "affinity" else MOE_DROP_TOKEN_ORDER)


# run dtype names: "fp8w" = bf16 activations with FP8 E4M3 expert weights; "fp8up" =
# the up projection on E4M3 activations and weights (H, W2, Y bf16)
_DTYPES = {"f32": MOE_F32, "fp32": MOE_F32, "float32": MOE_F32, "bf16": MOE_BF16, "bfloat16": MOE_BF16,
           "fp8w": MOE_BF16_FP8W, "fp8up": MOE_BF16_FP8UP}


def config_from_workload(w, T=None) -> moe_config:
    return config(T if T is not None else w.T, w.d, w.E, w.f, w.k if w.mode == "tc" else 0, w.gate, w.mode,
                  w.renorm, w.capacity_factor, w.ec_capacity, w.n_shared, w.f_shared, w.dtype, w.drop_policy)


# ------------------------------------------------------------------ host queries (no CUDA call)
def moe_validate_config(cfg) -> int:
    return lib().moe_validate_config(ctypes.byref(cfg))


def moe_expert_capacity(cfg) -> int:
    cap = ctypes.c_int32()
    _check(lib().moe_expert_capacity(ctypes.byref(cfg), ctypes.byref(cap)), "moe_expert_capacity")
    return cap.value


def moe_buffer_rows(cfg):
    r, t = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().moe_buffer_rows(ctypes.byref(cfg), ctypes.byref(r), ctypes.byref(t)), "moe_buffer_rows")
    return r.value, t.value


def moe_workspace_size(cfg, stage=MOE_STAGE_FORWARD) -> int:
    b = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), int(stage), ctypes.byref(b)), "moe_workspace_size")
    return b.value


def moe_packed_weights_size(cfg) -> int:
    b = ctypes.c_size_t()
    _check(lib().moe_packed_weights_size(ctypes.byref(cfg), ctypes.byref(b)), "moe_packed_weights_size")
    return b.value


# ------------------------------------------------------------------ device entry points
def moe_pack_weights(cfg, W1, W3, W2, W1s, W3s, W2s, packed, stream=None):
    _check(lib().moe_pack_weights(ctypes.byref(cfg), _p(W1), _p(W3), _p(W2), _p(W1s), _p(W3s), _p(W2s), _p(packed),
                                  _nbytes(packed), _stream(stream)), "moe_pack_weights")


def moe_route(cfg, x, W_r, logit_offset, sel_bias, topk_idx, topk_w, ws, stream=None, prob_sum=None):
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(W_r), _p(logit_offset), _p(sel_bias), _p(topk_idx),
                           _p(topk_w), _p(prob_sum), _p(ws), _nbytes(ws), _stream(stream)), "moe_route")


def moe_load_stats(cfg, topk_idx, cnt_raw, prob_sum, token_fraction, prob_mean, summary, stream=None):
    _check(lib().moe_load_stats(ctypes.byref(cfg), _p(topk_idx), _p(cnt_raw), _p(prob_sum), _p(token_fraction),
                                _p(prob_mean), _p(summary), _stream(stream)), "moe_load_stats")


def moe_dispatch(cfg, topk_idx, x, off, cnt_raw, slot_of, x_perm, ws, stream=None, topk_w=None):
    """topk_w: the gate weights, read for the affinity-ordered capacity drop only."""
    _check(lib().moe_dispatch(ctypes.byref(cfg), _p(topk_idx), _p(topk_w), _p(x), _p(off), _p(cnt_raw), _p(slot_of),
                              _p(x_perm), _p(ws), _nbytes(ws), _stream(stream)), "moe_dispatch")


def moe_dispatch_noalloc(cfg, topk_idx, x, off, cnt_raw, slot_of, x_perm, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate device
    memory; scratch comes from a fixed array inside the library (see the header)."""
    _check(lib().moe_dispatch_noalloc(ctypes.byref(cfg), _p(topk_idx), _p(x), _p(off), _p(cnt_raw), _p(slot_of),
                                      _p(x_perm), _stream(stream)), "moe_dispatch_noalloc")


def moe_grouped_ffn(cfg, x_perm, off, packed, x, Y, ws, stream=None):
    _check(lib().moe_grouped_ffn(ctypes.byref(cfg), _p(x_perm), _p(off), _p(packed), _p(x), _p(Y), _p(ws),
                                 _nbytes(ws), _stream(stream)), "moe_grouped_ffn")


def moe_grouped_ffn_up(cfg, x_perm, off, packed, x, H, Hs, stream=None):
    _check(lib().moe_grouped_ffn_up(ctypes.byref(cfg), _p(x_perm), _p(off), _p(packed), _p(x), _p(H), _p(Hs),
                                    _stream(stream)), "moe_grouped_ffn_up")


def moe_grouped_ffn_down(cfg, H, Hs, off, packed, Y, stream=None):
    _check(lib().moe_grouped_ffn_down(ctypes.byref(cfg), _p(H), _p(Hs), _p(off), _p(packed), _p(Y),
                                      _stream(stream)), "moe_grouped_ffn_down")


def moe_launch_count(cfg, stage=MOE_STAGE_FORWARD) -> int:
    n = ctypes.c_int32()
    _check(lib().moe_launch_count(ctypes.byref(cfg), int(stage), ctypes.byref(n)), "moe_launch_count")
    return n.value


def moe_combine(cfg, Y, slot_of, topk_w, y, ws=None, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(Y), _p(slot_of), _p(topk_w), _p(y), _p(ws), _nbytes(ws),
                             _stream(stream)), "moe_combine")


def moe_forward(cfg, x, W_r, logit_offset, sel_bias, packed, y, ws, stream=None):
    _check(lib().moe_forward(ctypes.byref(cfg), _p(x), _p(W_r), _p(logit_offset), _p(sel_bias), _p(packed), _p(y),
                             _p(ws), _nbytes(ws), _stream(stream)), "moe_forward")


def moe_set_wait_limit_ns(limit_ns: int):
    _check(lib().moe_set_wait_limit_ns(int(limit_ns)), "moe_set_wait_limit_ns")


def moe_get_wait_limit_ns() -> int:
    v = ctypes.c_uint64()
    _check(lib().moe_get_wait_limit_ns(ctypes.byref(v)), "moe_get_wait_limit_ns")
    return int(v.value)


def moe_set_tile_group_bytes(up_bytes: int, down_bytes: int):
    _check(lib().moe_set_tile_group_bytes(int(up_bytes), int(down_bytes)), "moe_set_tile_group_bytes")


def moe_get_tile_group_bytes() -> tuple[int, int]:
    u, d = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().moe_get_tile_group_bytes(ctypes.byref(u), ctypes.byref(d)), "moe_get_tile_group_bytes")
    return int(u.value), int(d.value)


def moe_wait_probe(flag, target=1, stream=None):
    _check(lib().moe_wait_probe(_p(flag), int(target), _stream(stream)), "moe_wait_probe")


def moe_check_device_error(stream=None):
    _check(lib().moe_check_device_error(_stream(stream)), "moe_check_device_error")
