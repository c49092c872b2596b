"""Python binding of libmoe_ffn.so (the GB300 routed FP4 MoE expert-FFN library).

Argument marshalling only: every function forwards to the C entry point of the
same name in include/moe_ffn.h.  Pointers may be given as ints or as torch
tensors (their data_ptr() is passed); streams as ints, torch streams or None
(the legacy default stream).  A nonzero return code raises MoeError.  There is
no fallback: if the CUDA library cannot be built or loaded, importing the
binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_CUDA = -2
MOE_ERR_OOM = -3
MOE_ERR_UNSUPPORTED = -4
MOE_ERR_BAD_INDEX = -5
MOE_ERR_DEVICE_TIMEOUT = -6

MOE_ACT_BF16 = 0
MOE_ACT_E4M3_UE8M0_128 = 1
MOE_ACT_E2M1_UE8M0_32 = 2
MOE_OUT_BF16 = 0
MOE_OUT_F32 = 1
DEFAULT_GEMM_MIN_TOKENS = 16   # MOE_DEFAULT_GEMM_MIN_TOKENS

EXPORTS = [
    "moe_ffn_packed_expert_bytes", "moe_ffn_create",
    "moe_ffn_pack_expert", "moe_ffn_forward", "moe_ffn_forward_host", "moe_ffn_route",
    "moe_ffn_act_quant", "moe_stack_forward", "moe_stack_forward_host", "moe_ffn_profile_enable",
    "moe_ffn_profile_read",
    "moe_ffn_status", "moe_ffn_strerror", "moe_ffn_destroy", "moe_ffn_forward_noalloc",
    "moe_router_topk", "moe_router_select", "moe_batch_plan", "moe_batch_distinct",
    "moe_expert_cache_create", "moe_expert_cache_fetch", "moe_expert_cache_prefetch", "moe_expert_cache_slot",
    "moe_expert_cache_stats", "moe_expert_cache_destroy", "moe_ffn_test_set_wait", "moe_ffn_test_fail_allocs",
    "moe_ffn_test_copy_h",
    "moe_ffn_set_mma_kind", "moe_ffn_set_routing_wait",
    "moe_ffn_profile_layer_only",
]

MOE_MMA_AUTO = 0
MOE_MMA_MXF4_PIECES = 1
MOE_MMA_MXF8F6F4 = 2

MOE_PHASE_PREP = 0
MOE_PHASE_GATE_UP = 1
MOE_PHASE_DOWN = 2
MOE_PHASE_ROUTE = 3
MOE_PHASE_ACT_QUANT = 4
MOE_PHASE_ROUTER = 5
MOE_NUM_PHASES = 8


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class moe_ffn_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_experts", "hidden", "inter", "topk", "max_tokens", "act_mode", "out_dtype",
        "gemm_min_tokens")]


class moe_expert_table(ctypes.Structure):
    _fields_ = [("experts", ctypes.c_void_p)]


_lib = None


def build(force: bool = False) -> str:
    """Compile libmoe_ffn.so for sm_103a (in-tree)."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        cfgp = ctypes.POINTER(moe_ffn_config)
        tblp = ctypes.POINTER(moe_expert_table)
        sig = {
            "moe_ffn_packed_expert_bytes": (S, [cfgp]),
            "moe_ffn_create": (I, [ctypes.POINTER(P), cfgp, I]),
            "moe_ffn_pack_expert": (I, [P, P, P, P, P]),
            "moe_ffn_forward": (I, [P, P, P, P, tblp, P, I, P]),
            "moe_ffn_forward_host": (I, [P, P, P, P, tblp, P, I, P]),
            "moe_ffn_route": (I, [P, P, I, P, P, P, P, P]),
            "moe_ffn_act_quant": (I, [P, P, I, I, P, P, P]),
            "moe_stack_forward": (I, [P, P, tblp, P, P, I, I, P]),
            "moe_stack_forward_host": (I, [P, P, tblp, P, P, I, I, P]),
            "moe_ffn_profile_enable": (I, [P, I]),
            "moe_ffn_profile_read": (I, [P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I)]),
            "moe_ffn_status": (I, [P, P]),
            "moe_ffn_strerror": (ctypes.c_char_p, [I]),
            "moe_ffn_destroy": (None, [P]),
            "moe_ffn_forward_noalloc": (I, [cfgp, I, P, P, P, tblp, P, I, P, P]),
            "moe_router_topk": (I, [P, P, P, I, P, P, P, P]),
            "moe_router_select": (I, [P, P, I, P, P, P]),
            "moe_batch_plan": (I, [P, I, I, I, I, I, P]),
            "moe_batch_distinct": (I, [P, P, I, I, I, I, I, P]),
            "moe_expert_cache_create": (I, [cfgp, I, P, I, ctypes.POINTER(P)]),
            "moe_expert_cache_fetch": (I, [P, P, I, P, tblp]),
            "moe_expert_cache_prefetch": (I, [P, P, I, P]),
            "moe_expert_cache_slot": (I, [P, I]),
            "moe_expert_cache_stats": (I, [P, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(ctypes.c_longlong),
                                           ctypes.POINTER(ctypes.c_longlong)]),
            "moe_expert_cache_destroy": (None, [P]),
            "moe_ffn_test_set_wait": (I, [P, ctypes.c_ulonglong, I]),
            "moe_ffn_test_fail_allocs": (None, [I]),
            "moe_ffn_test_copy_h": (I, [P, P, P, I, P]),
            "moe_ffn_set_mma_kind": (I, [P, I]),
            "moe_ffn_set_routing_wait": (I, [P, I]),
            "moe_ffn_profile_layer_only": (I, [P, I]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def library_path() -> str:
    return os.path.abspath(_build.LIB)


def _p(x) -> int | None:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, ctypes.Array):
        return ctypes.addressof(x)
    return int(x)


def _s(stream) -> int | None:
    if stream is None:
        return None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int, where: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, where)


def strerror(code: int) -> str:
    return lib().moe_ffn_strerror(int(code)).decode()


moe_ffn_strerror = strerror


def config(num_experts, hidden, inter, topk, max_tokens, act_mode=MOE_ACT_BF16,
           out_dtype=MOE_OUT_F32, gemm_min_tokens=0) -> moe_ffn_config:
    return moe_ffn_config(num_experts, hidden, inter, topk, max_tokens, act_mode, out_dtype,
                          gemm_min_tokens)


def moe_ffn_packed_expert_bytes(cfg: moe_ffn_config) -> int:
    return lib().moe_ffn_packed_expert_bytes(ctypes.byref(cfg))


def moe_ffn_create(cfg: moe_ffn_config, device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(lib().moe_ffn_create(ctypes.byref(h), ctypes.byref(cfg), int(device)), "moe_ffn_create")
    return h.value


def moe_ffn_pack_expert(h, canon_codes, canon_scales, packed, stream=None):
    _check(lib().moe_ffn_pack_expert(h, _p(canon_codes), _p(canon_scales), _p(packed), _s(stream)),
           "moe_ffn_pack_expert")


def expert_table(expert_ptrs) -> moe_expert_table:
    """expert_ptrs: a device array (e.g. a torch int64 tensor on the GPU)
    holding one device pointer per expert, each to a packed blob."""
    return moe_expert_table(_p(expert_ptrs))


def moe_ffn_forward(h, x, topk_idx, topk_w, table: moe_expert_table, y, T: int, stream=None):
    _check(lib().moe_ffn_forward(h, _p(x), _p(topk_idx), _p(topk_w), ctypes.byref(table), _p(y),
                                 int(T), _s(stream)), "moe_ffn_forward")


def moe_ffn_forward_host(h, x, topk_idx, topk_w, table: moe_expert_table, y, T: int, stream=None):
    _check(lib().moe_ffn_forward_host(h, _p(x), _p(topk_idx), _p(topk_w), ctypes.byref(table),
                                      _p(y), int(T), _s(stream)), "moe_ffn_forward_host")


def moe_ffn_route(h, topk_idx, T: int, counts, offsets, perm, inv, stream=None):
    _check(lib().moe_ffn_route(h, _p(topk_idx), int(T), _p(counts), _p(offsets), _p(perm), _p(inv),
                               _s(stream)), "moe_ffn_route")


def moe_ffn_act_quant(h, x, rows: int, n: int, codes, scales, stream=None):
    _check(lib().moe_ffn_act_quant(h, _p(x), int(rows), int(n), _p(codes), _p(scales), _s(stream)),
           "moe_ffn_act_quant")


def moe_stack_forward(h, x, tables, topk_idx, topk_w, L: int, T: int, stream=None):
    """tables: a sequence of moe_expert_table, one per layer."""
    arr = (moe_expert_table * len(tables))(*tables)
    _check(lib().moe_stack_forward(h, _p(x), arr, _p(topk_idx), _p(topk_w), int(L), int(T),
                                   _s(stream)), "moe_stack_forward")


def moe_stack_forward_host(h, x_host, tables, topk_idx_host, topk_w_host, L: int, T: int, stream=None):
    """Host buffers (CPU tensors or ints holding host addresses): x fp32 [T][H]
    updated in place, topk_idx int32 / topk_w fp32 [L][T][k]; waits for the
    stream.  tables: a sequence of moe_expert_table, one per layer."""
    arr = (moe_expert_table * len(tables))(*tables)
    _check(lib().moe_stack_forward_host(h, _p(x_host), arr, _p(topk_idx_host), _p(topk_w_host), int(L), int(T),
                                        _s(stream)), "moe_stack_forward_host")


def moe_ffn_profile_enable(h, on: bool = True) -> None:
    _check(lib().moe_ffn_profile_enable(h, 1 if on else 0), "moe_ffn_profile_enable")


def moe_ffn_profile_read(h):
    """Returns (ms, launches): per-phase summed milliseconds and launch counts."""
    ms = (ctypes.c_double * MOE_NUM_PHASES)()
    n = (ctypes.c_int * MOE_NUM_PHASES)()
    _check(lib().moe_ffn_profile_read(h, ms, n), "moe_ffn_profile_read")
    return list(ms), list(n)


def moe_ffn_profile_layer_only(h, on: bool = True) -> None:
    """Measurement mode: slot-major forwards launch the layer kernel alone,
    reusing the last full call's activation pieces (see include/moe_ffn.h)."""
    _check(lib().moe_ffn_profile_layer_only(h, 1 if on else 0), "moe_ffn_profile_layer_only")


def moe_ffn_set_mma_kind(h, kind: int) -> None:
    """The expert-major path's MMA in the E4M3 mode (MOE_MMA_*)."""
    _check(lib().moe_ffn_set_mma_kind(h, int(kind)), "moe_ffn_set_mma_kind")


def moe_ffn_set_routing_wait(h, on: int) -> None:
    """1: the layer's kernels read the routing only after their dependency wait."""
    _check(lib().moe_ffn_set_routing_wait(h, int(on)), "moe_ffn_set_routing_wait")


def moe_ffn_status(h, stream=None) -> int:
    """Returns the (cleared) sticky device status code; does not raise."""
    return lib().moe_ffn_status(h, _s(stream))


def moe_ffn_forward_noalloc(cfg: moe_ffn_config, device: int, x, topk_idx, topk_w,
                            table: moe_expert_table, y, T: int, status=None, stream=None):
    """The layer without a handle, using the library's fixed device scratch
    array instead of allocating (see include/moe_ffn.h)."""
    _check(lib().moe_ffn_forward_noalloc(ctypes.byref(cfg), int(device), _p(x), _p(topk_idx),
                                         _p(topk_w), ctypes.byref(table), _p(y), int(T),
                                         _p(status), _s(stream)), "moe_ffn_forward_noalloc")


def moe_ffn_test_copy_h(h, n: int, inter: int, stream=None):
    """Test hook: (h [n][inter] fp32, perm [n] int32) of the last kind::mxf8f6f4
    expert-major call, as device tensors (see include/moe_ffn.h)."""
    import torch

    hd = torch.empty((n, inter), dtype=torch.float32, device="cuda")
    pd = torch.empty(n, dtype=torch.int32, device="cuda")
    _check(lib().moe_ffn_test_copy_h(h, hd.data_ptr(), pd.data_ptr(), int(n), _s(stream)), "moe_ffn_test_copy_h")
    return hd, pd


def moe_ffn_test_set_wait(h, wait_ns: int, withhold: bool) -> None:
    """Test hook: bounded-wait limit of the slot-major kernel and the withheld
    partial sums that make its waits run out (see include/moe_ffn.h)."""
    _check(lib().moe_ffn_test_set_wait(h, int(wait_ns), 1 if withhold else 0), "moe_ffn_test_set_wait")


def moe_ffn_test_fail_allocs(n: int) -> None:
    """Test hook: the library's next n allocations fail as if out of memory."""
    lib().moe_ffn_test_fail_allocs(int(n))


def moe_ffn_destroy(h) -> None:
    lib().moe_ffn_destroy(h)


def moe_router_topk(h, x, router_w, T: int, topk_idx, topk_w, logits=None, stream=None):
    _check(lib().moe_router_topk(h, _p(x), _p(router_w), int(T), _p(logits), _p(topk_idx), _p(topk_w),
                                 _s(stream)), "moe_router_topk")


def moe_router_select(h, logits, T: int, topk_idx, topk_w, stream=None):
    _check(lib().moe_router_select(h, _p(logits), int(T), _p(topk_idx), _p(topk_w), _s(stream)),
           "moe_router_select")


def _host_i32(a, ndim):
    import numpy as np

    a = np.ascontiguousarray(a, dtype=np.int32)
    if a.ndim != ndim:
        raise ValueError(f"expected a {ndim}-d int32 array, got shape {a.shape}")
    return a


def moe_batch_plan(sig, E: int, B: int):
    """Batch order of N sequences from their signatures sig [N][L][topk] (host
    int32 expert ids, -1 for none): returns order [N] (host int32)."""
    import numpy as np

    sig = _host_i32(sig, 3)
    N, L, k = sig.shape
    order = np.empty(N, np.int32)
    _check(lib().moe_batch_plan(sig.ctypes.data, N, L, k, int(E), int(B), order.ctypes.data), "moe_batch_plan")
    return order


def moe_batch_distinct(routing, order, E: int, B: int):
    """Distinct experts per (batch, layer) [ceil(N/B)][L] of routing [N][L][topk]
    cut into batches of B in the given order."""
    import numpy as np

    routing = _host_i32(routing, 3)
    order = _host_i32(order, 1)
    N, L, k = routing.shape
    if order.size != N:
        raise ValueError("order must hold N entries")
    out = np.empty(((N + B - 1) // B, L), np.int32)
    _check(lib().moe_batch_distinct(routing.ctypes.data, order.ctypes.data, N, L, k, int(E), int(B),
                                    out.ctypes.data), "moe_batch_distinct")
    return out


# ------------------------------------------------------ host-resident experts

def moe_expert_cache_create(cfg, device: int, host_ptrs, slots: int):
    """Cache of `slots` device slots over experts whose packed blobs sit at the
    host addresses host_ptrs [E] (page-locked)."""
    arr = (ctypes.c_void_p * len(host_ptrs))(*[int(p) for p in host_ptrs])
    out = ctypes.c_void_p()
    _check(lib().moe_expert_cache_create(ctypes.byref(cfg), int(device), arr, int(slots), ctypes.byref(out)),
           "moe_expert_cache_create")
    return out.value


def moe_expert_cache_fetch(c, ids, stream=None):
    """Makes the experts of ids (host int32) resident; returns the layer's table."""
    import numpy as np

    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    tbl = moe_expert_table()
    _check(lib().moe_expert_cache_fetch(c, ids.ctypes.data, ids.size, _s(stream), ctypes.byref(tbl)),
           "moe_expert_cache_fetch")
    return tbl


def moe_expert_cache_prefetch(c, ids, stream=None):
    import numpy as np

    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    _check(lib().moe_expert_cache_prefetch(c, ids.ctypes.data, ids.size, _s(stream)), "moe_expert_cache_prefetch")


def moe_expert_cache_slot(c, expert: int) -> int:
    return int(lib().moe_expert_cache_slot(c, int(expert)))


def moe_expert_cache_stats(c):
    h, m, b = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
    _check(lib().moe_expert_cache_stats(c, ctypes.byref(h), ctypes.byref(m), ctypes.byref(b)),
           "moe_expert_cache_stats")
    return h.value, m.value, b.value


def moe_expert_cache_destroy(c) -> None:
    lib().moe_expert_cache_destroy(c)
