"""CPU reference (oracle) of the routed FP4 MoE expert FFN -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product library never does; the two share no
code.  The arithmetic lives in ``oracle.c`` (plain C, fp64); this module only
builds it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ACT_BF16 = 0
ACT_E4M3_UE8M0_128 = 1
ACT_E2M1_UE8M0_32 = 2

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (portable C, no target-specific flags).

    -ffp-contract=off keeps every multiply and add separately rounded, so the
    results are the same on x86-64 and aarch64 hosts.
    """
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared",
             "-pthread", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, dbl = ctypes.c_int, ctypes.c_double
        L.orc_e2m1_value.restype = dbl
        L.orc_e2m1_value.argtypes = [i32]
        L.orc_ue8m0_value.restype = dbl
        L.orc_ue8m0_value.argtypes = [i32]
        L.orc_bf16_value.restype = dbl
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_bf16_rne.restype = ctypes.c_uint16
        L.orc_bf16_rne.argtypes = [dbl]
        L.orc_e4m3_value.restype = dbl
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_rne.restype = ctypes.c_uint8
        L.orc_e4m3_rne.argtypes = [dbl]
        L.orc_ue8m0_for_amax.restype = i32
        L.orc_ue8m0_for_amax.argtypes = [dbl]
        L.orc_act_quant_e4m3.restype = None
        L.orc_act_quant_e4m3.argtypes = [P, i32, i32, P, P]
        L.orc_e2m1_rne.restype = i32
        L.orc_e2m1_rne.argtypes = [dbl]
        L.orc_ue8m0_for_amax_e2m1.restype = i32
        L.orc_ue8m0_for_amax_e2m1.argtypes = [dbl]
        L.orc_act_quant_e2m1.restype = None
        L.orc_act_quant_e2m1.argtypes = [P, i32, i32, P, P]
        L.orc_silu.restype = dbl
        L.orc_silu.argtypes = [dbl]
        L.orc_matvec.restype = i32
        L.orc_matvec.argtypes = [P, P, i32, i32, P, P]
        L.orc_expert_ffn.restype = i32
        L.orc_expert_ffn.argtypes = [P, P, i32, i32, P, i32, P]
        L.orc_moe_ffn.restype = i32
        L.orc_moe_ffn.argtypes = [P, P, i32, i32, P, P, i32, P, i32]
        L.orc_route.restype = i32
        L.orc_route.argtypes = [P, i32, i32, i32, P, P, P, P]
        L.orc_rmsnorm_bf16.restype = None
        L.orc_rmsnorm_bf16.argtypes = [P, i32, dbl, P]
        L.orc_moe_stack.restype = i32
        L.orc_moe_stack.argtypes = [P, i32, P, i32, i32, P, P, i32, dbl, i32]
        L.orc_router_logits.argtypes = [P, P, i32, i32, i32, P]
        L.orc_router_logits.restype = None
        L.orc_topk_softmax.argtypes = [P, i32, i32, i32, P, P]
        L.orc_topk_softmax.restype = i32
        _lib = L
    return _lib


class _Layer(ctypes.Structure):
    _fields_ = [
        ("num_experts", ctypes.c_int),
        ("hidden", ctypes.c_int),
        ("inter", ctypes.c_int),
        ("codes", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
    ]


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def ue8m0_value(s: int) -> float:
    return lib().orc_ue8m0_value(int(s))


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(int(bits))


def bf16_rne(v: float) -> int:
    return int(lib().orc_bf16_rne(float(v)))


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def e4m3_rne(v: float) -> int:
    return int(lib().orc_e4m3_rne(float(v)))


def ue8m0_for_amax(amax: float) -> int:
    return int(lib().orc_ue8m0_for_amax(float(amax)))


def silu(g: float) -> float:
    return lib().orc_silu(float(g))


def act_quant_e4m3(v, block: int = 128):
    v = _c(v, np.float64)
    n = v.size
    codes = np.zeros(n, np.uint8)
    scales = np.zeros((n + block - 1) // block, np.uint8)
    lib().orc_act_quant_e4m3(_ptr(v), n, block, _ptr(codes), _ptr(scales))
    return codes, scales


def e2m1_rne(v: float) -> int:
    """Nearest E2M1 code to v (ties to the even mantissa, saturating)."""
    return int(lib().orc_e2m1_rne(float(v)))


def ue8m0_for_amax_e2m1(amax: float) -> int:
    """Scale byte k + 127 of an E2M1 block: the least k with amax <= 6 * 2^k."""
    return int(lib().orc_ue8m0_for_amax_e2m1(float(amax)))


def act_quant_e2m1(v, block: int = 32):
    """Per-block E2M1 codes (one per byte) and ue8m0 scale bytes of v."""
    v = _c(v, np.float64)
    n = v.size
    codes = np.zeros(n, np.uint8)
    scales = np.zeros((n + block - 1) // block, np.uint8)
    lib().orc_act_quant_e2m1(_ptr(v), n, block, _ptr(codes), _ptr(scales))
    return codes, scales


def matvec(codes, scales, rows: int, k: int, v) -> np.ndarray:
    codes, scales, v = _c(codes, np.uint8), _c(scales, np.uint8), _c(v, np.float64)
    out = np.zeros(rows, np.float64)
    rc = lib().orc_matvec(_ptr(codes), _ptr(scales), rows, k, _ptr(v), _ptr(out))
    if rc:
        raise ValueError(f"orc_matvec failed ({rc})")
    return out


def expert_ffn(codes, scales, hidden: int, inter: int, x, act_mode: int = ACT_BF16) -> np.ndarray:
    codes, scales, x = _c(codes, np.uint8), _c(scales, np.uint8), _c(x, np.float64)
    o = np.zeros(hidden, np.float64)
    rc = lib().orc_expert_ffn(_ptr(codes), _ptr(scales), hidden, inter, _ptr(x), act_mode, _ptr(o))
    if rc:
        raise ValueError(f"orc_expert_ffn failed ({rc})")
    return o


def _layer_struct(codes_list, scales_list, hidden, inter, keep):
    E = len(codes_list)
    cptr = (ctypes.c_void_p * E)()
    sptr = (ctypes.c_void_p * E)()
    for e in range(E):
        if codes_list[e] is not None:
            c = _c(codes_list[e], np.uint8)
            s = _c(scales_list[e], np.uint8)
            keep += [c, s]
            cptr[e] = _ptr(c)
            sptr[e] = _ptr(s)
    keep += [cptr, sptr]
    return _Layer(E, hidden, inter, ctypes.cast(cptr, ctypes.c_void_p), ctypes.cast(sptr, ctypes.c_void_p))


def moe_ffn(codes_list, scales_list, hidden: int, inter: int, x_bf16, topk_idx, topk_w,
            act_mode: int = ACT_BF16, nthreads: int = 1) -> np.ndarray:
    """codes_list[e] / scales_list[e]: canonical blobs (None for unused experts);
    x_bf16: uint16 [T, H] bf16 bit patterns; topk_idx int32 [T, k]; topk_w f32 [T, k].
    Returns y as float64 [T, H]."""
    keep: list = []
    layer = _layer_struct(codes_list, scales_list, hidden, inter, keep)
    x = _c(x_bf16, np.uint16)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float32)
    T, k = idx.shape
    y = np.zeros((T, hidden), np.float64)
    rc = lib().orc_moe_ffn(ctypes.addressof(layer), _ptr(x), T, k, _ptr(idx), _ptr(w),
                           act_mode, _ptr(y), int(nthreads))
    if rc:
        raise ValueError(f"orc_moe_ffn failed ({rc})")
    return y


def route(topk_idx, num_experts: int):
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(num_experts, np.int32)
    offsets = np.zeros(num_experts + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    inv = np.zeros(T * k, np.int32)
    rc = lib().orc_route(_ptr(idx), T, k, num_experts, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv))
    if rc:
        raise ValueError(f"orc_route failed ({rc})")
    return counts, offsets, perm, inv


def rmsnorm_bf16(x, eps: float = 1e-6) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.zeros(x.shape, np.uint16)
    n = x.shape[-1]
    for t in range(x.size // n):
        lib().orc_rmsnorm_bf16(_ptr(x) + 8 * t * n, n, eps, _ptr(out) + 2 * t * n)
    return out


def moe_stack(layers, x, topk_idx, topk_w, act_mode: int = ACT_BF16, eps: float = 1e-6,
              nthreads: int = 1) -> np.ndarray:
    """layers: list of (codes_list, scales_list, hidden, inter); x float64 [T, H]
    (the residual, returned updated); topk_idx int32 [L, T, k]; topk_w f32 [L, T, k]."""
    keep: list = []
    L = len(layers)
    arr = (_Layer * L)()
    for l, (cl, sl, H, I) in enumerate(layers):
        arr[l] = _layer_struct(cl, sl, H, I, keep)
    x = np.array(x, dtype=np.float64, order="C", copy=True)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_w, np.float32)
    _, T, k = idx.shape
    rc = lib().orc_moe_stack(ctypes.addressof(arr), L, _ptr(x), T, k, _ptr(idx), _ptr(w),
                             act_mode, float(eps), int(nthreads))
    if rc:
        raise ValueError(f"orc_moe_stack failed ({rc})")
    return x


def router_logits(x_bf16, w_bf16) -> np.ndarray:
    """fp64 logits [T][E] of bf16 activations x [T][H] and router weights W [E][H]."""
    x = _c(x_bf16, np.uint16)
    w = _c(w_bf16, np.uint16)
    T, H = x.shape
    E = w.shape[0]
    assert w.shape[1] == H
    out = np.zeros((T, E), np.float64)
    lib().orc_router_logits(_ptr(x), _ptr(w), T, H, E, _ptr(out))
    return out


def topk_softmax(logits, k: int):
    """(idx int32 [T][k], w float64 [T][k]) of the k largest logits per row."""
    l = _c(logits, np.float64)
    T, E = l.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    rc = lib().orc_topk_softmax(_ptr(l), T, E, k, _ptr(idx), _ptr(w))
    assert rc == 0, "orc_topk_softmax failed"
    return idx, w


# ------------------------------------------------ expert-sharing batching

def batch_distinct(routing, order, B: int) -> np.ndarray:
    """Distinct experts touched per (batch, layer) when the sequences, taken in
    `order`, are cut into batches of B: |union of the batch's expert ids| with
    -1 meaning none.  routing [N][L][k]; returns [ceil(N/B)][L]."""
    routing = np.asarray(routing)
    N, L, _ = routing.shape
    nb = (N + B - 1) // B
    out = np.zeros((nb, L), np.int64)
    for b in range(nb):
        members = [int(i) for i in order[b * B:(b + 1) * B]]
        for l in range(L):
            experts = set()
            for i in members:
                experts |= {int(e) for e in routing[i, l] if e >= 0}
            out[b, l] = len(experts)
    return out


def batch_plan_greedy(sig, B: int) -> np.ndarray:
    """The greedy expert-sharing plan, step by step: a batch starts from the
    lowest-numbered sequence not yet placed; while it holds fewer than B, it
    takes the unplaced sequence that adds the fewest experts not yet in the
    batch, summed over the layers (the lowest number among equals).  Reading
    (the pages report the effect -- 216 -> 156 distinct experts in a layer
    when alike prompts share a batch -- and no algorithm)."""
    sig = np.asarray(sig)
    N, L, _ = sig.shape
    rows = [[{int(e) for e in sig[i, l] if e >= 0} for l in range(L)] for i in range(N)]
    placed = [False] * N
    order = []
    while len(order) < N:
        seed = placed.index(False)
        batch_sets = [set(s) for s in rows[seed]]
        placed[seed] = True
        order.append(seed)
        size = 1
        while size < B and len(order) < N:
            best, best_cost = None, None
            for i in range(N):
                if placed[i]:
                    continue
                cost = sum(len(rows[i][l] - batch_sets[l]) for l in range(L))
                if best_cost is None or cost < best_cost:
                    best, best_cost = i, cost
            placed[best] = True
            order.append(best)
            for l in range(L):
                batch_sets[l] |= rows[best][l]
            size += 1
    return np.array(order, np.int32)
