"""Seeded synthetic inputs shaped like the routed FP4 MoE decode workload.

This module only draws inputs; it holds none of the method's arithmetic.  It
serves both the oracle and the CUDA path, and nothing else is shared between
them.

Every random quantity comes from one counter-based generator, SplitMix64
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014): the n-th output of stream s under seed S is

    key      = mix64(S * GAMMA + s)                 (mod 2^64)
    u64(n)   = mix64(key + (n + 1) * GAMMA)         (mod 2^64)
    mix64(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)

with GAMMA = 0x9E3779B97F4A7C15.  Being counter-based, any slice of any stream
can be regenerated independently: the host draws single experts with numpy,
and ``synth_fill.cu`` fills whole expert sets on the device with the same
function (a test checks the two agree byte for byte).

Recipes (all seed 0 unless a test says otherwise):
  * E2M1 codes: byte j of a code stream is byte (j mod 8) (little-endian) of
    u64(j div 8): both nibbles uniform over the 16 codes.
  * ue8m0 scales: byte j = lo + floor((u64(j) >> 32) * (hi - lo + 1) / 2^32),
    lo = 119, hi = 127 (Lemire's multiply-shift reduction).
  * x ~ N(0,1): Box-Muller in fp64 on two outputs per element, rounded to
    fp32 then to bf16 (round to nearest even at each step).
  * routing: per token, draws (u64 >> 32) * E >> 32, rejecting repeats until
    top-k distinct experts (uniform without replacement); Zipf(s) routing
    draws expert e with probability proportional to (e + 1)^-s by inverse CDF.
  * topk_w: softmax (fp64) of top-k N(0,1) logits, stored as fp32.
  * clustered routing (alike prompts route alike): sequence i belongs to
    cluster (u64(i) >> 32) * C >> 32; cluster c has, per layer, a hot set of
    `hot` distinct experts drawn uniformly; at decode step s each (sequence,
    layer) draws k distinct experts, each draw from the hot set with
    probability p_hot (uniform within it) and otherwise uniform over all E.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# stream ids
S_CODES, S_SCALES = 0, 1
S_X, S_ROUTE, S_LOGIT = 0x10, 0x11, 0x12
S_ROUTER_W = 0x13
S_CLUSTER, S_HOT, S_CROUTE = 0x14, 0x15, 0x16


def mix64_int(z: int) -> int:
    z &= _M64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    return mix64_int((seed * GAMMA + stream) & _M64)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def u64(seed: int, stream: int, n0: int, count: int) -> np.ndarray:
    """Outputs n0 .. n0+count-1 of the stream, as uint64."""
    key = np.uint64(stream_key(seed, stream))
    with np.errstate(over="ignore"):
        ctr = np.arange(n0 + 1, n0 + count + 1, dtype=np.uint64)
        return _mix64(key + ctr * np.uint64(GAMMA))


def random_bytes(seed: int, stream: int, nbytes: int, offset: int = 0) -> np.ndarray:
    """Bytes offset .. offset+nbytes-1 of a byte stream (8 bytes per output)."""
    w0 = offset // 8
    w1 = (offset + nbytes + 7) // 8
    words = u64(seed, stream, w0, w1 - w0)
    b = words.astype("<u8").view(np.uint8)
    s = offset - 8 * w0
    return b[s:s + nbytes].copy()


def random_range_bytes(seed: int, stream: int, nbytes: int, lo: int, hi: int,
                       offset: int = 0) -> np.ndarray:
    r = u64(seed, stream, offset, nbytes) >> np.uint64(32)
    return (np.uint64(lo) + ((r * np.uint64(hi - lo + 1)) >> np.uint64(32))).astype(np.uint8)


def uniforms(seed: int, stream: int, n0: int, count: int) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (u64(seed, stream, n0, count) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def normals(seed: int, stream: int, count: int, n0: int = 0) -> np.ndarray:
    """Box-Muller standard normals; element i uses outputs 2(n0+i) and 2(n0+i)+1."""
    u = uniforms(seed, stream, 2 * n0, 2 * count)
    u1 = 1.0 - u[0::2]                       # (0, 1]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = r.astype(np.uint16)
    nan = np.isnan(np.asarray(a, dtype=np.float32))
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------- experts

def expert_sizes(hidden: int, inter: int):
    """Canonical blob sizes: codes (gate|up|down, 2 codes per byte) and
    scales (one byte per 32 weights)."""
    n = 3 * hidden * inter
    return n // 2, n // 32


def expert_stream(layer: int, expert: int, which: int) -> int:
    return (layer << 24) | (expert << 2) | which


def expert_canonical(hidden: int, inter: int, expert: int, layer: int = 0, seed: int = 0,
                     scale_lo: int = 119, scale_hi: int = 127):
    """Canonical (codes, scales) of one expert as uint8 numpy arrays."""
    nc, ns = expert_sizes(hidden, inter)
    codes = random_bytes(seed, expert_stream(layer, expert, S_CODES), nc)
    scales = random_range_bytes(seed, expert_stream(layer, expert, S_SCALES), ns, scale_lo, scale_hi)
    return codes, scales


# -------------------------------------------------------------- activations

def activations_bf16(T: int, hidden: int, seed: int = 0, stream: int = S_X, n0: int = 0) -> np.ndarray:
    """x ~ N(0,1) as bf16 bit patterns, shape [T, hidden]."""
    z = normals(seed, stream, T * hidden, n0)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(T, hidden)


def router_weights_bf16(E: int, hidden: int, layer: int = 0, seed: int = 0) -> np.ndarray:
    """Router weights W ~ N(0, 1/hidden) as bf16 bit patterns, shape [E, hidden]
    (logits of unit-variance activations then have unit variance)."""
    z = normals(seed, S_ROUTER_W + 0x100 * layer, E * hidden) / np.sqrt(hidden)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(E, hidden)


def activations_f32(T: int, hidden: int, seed: int = 0, stream: int = S_X, n0: int = 0) -> np.ndarray:
    return normals(seed, stream, T * hidden, n0).astype(np.float32).reshape(T, hidden)


# ------------------------------------------------------------------ routing

def _distinct_draws(draw, T: int, k: int, E: int, avoid=None) -> np.ndarray:
    out = np.zeros((T, k), np.int32)
    for t in range(T):
        chosen: list = []
        j = 0
        while len(chosen) < k:
            e = draw(t, j)
            j += 1
            if e in chosen or (avoid is not None and e in avoid):
                continue
            chosen.append(e)
        out[t] = chosen
    return out


def routing_uniform(T: int, E: int, k: int, seed: int = 0, stream: int = S_ROUTE,
                    avoid=None) -> np.ndarray:
    """topk_idx [T, k]: per token k distinct experts, uniform without replacement.
    `avoid` (a set) excludes experts, used to make consecutive benchmark steps
    share no expert."""
    if avoid is not None and E - len(avoid) < k:
        avoid = None
    ndraw = 1024

    def draw(t, j):
        r = int(u64(seed, stream, t * ndraw + (j % ndraw), 1)[0] >> np.uint64(32))
        return (r * E) >> 32

    return _distinct_draws(draw, T, k, E, avoid)


def zipf_cdf(E: int, s: float) -> np.ndarray:
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def routing_zipf(T: int, E: int, k: int, s: float = 1.1, seed: int = 0,
                 stream: int = S_ROUTE) -> np.ndarray:
    """topk_idx [T, k]: expert e drawn with probability proportional to
    (e + 1)^-s (rank r = e + 1), repeats rejected until k are distinct."""
    cdf = zipf_cdf(E, s)
    ndraw = 4096
    uu = uniforms(seed, stream, 0, T * ndraw).reshape(T, ndraw)
    idx = np.minimum(np.searchsorted(cdf, uu, side="right"), E - 1).astype(np.int64)

    def draw(t, j):
        return int(idx[t, j % ndraw])

    return _distinct_draws(draw, T, k, E)


def routing_clustered(N: int, L: int, E: int, k: int, clusters: int = 8, hot: int = 32, p_hot: float = 0.6,
                      seed: int = 0, step: int = 0):
    """(routing [N][L][k] int32, cluster [N]) of N sequences at decode step
    `step` under the clustered recipe; the clusters and their hot sets depend
    on the seed only, so consecutive steps of a sequence route alike."""
    cl = ((u64(seed, S_CLUSTER, 0, N) >> np.uint64(32)) * np.uint64(clusters)) >> np.uint64(32)
    cl = cl.astype(np.int64)
    ndraw = 256
    hot_sets = {}

    def hot_set(c, l):
        if (c, l) not in hot_sets:
            base = (c * L + l) * ndraw
            hu = u64(seed, S_HOT, base, ndraw) >> np.uint64(32)
            hot_sets[(c, l)] = _distinct_draws(lambda t, j: int((int(hu[j % ndraw]) * E) >> 32), 1, hot, E)[0]
        return hot_sets[(c, l)]

    out = np.zeros((N, L, k), np.int32)
    for i in range(N):
        for l in range(L):
            hs = hot_set(int(cl[i]), l)
            base = ((step * N + i) * L + l) * 2 * ndraw
            uu = u64(seed, S_CROUTE, base, 2 * ndraw) >> np.uint64(32)

            def draw(t, j, uu=uu, hs=hs):
                a, b = int(uu[(2 * j) % (2 * ndraw)]), int(uu[(2 * j + 1) % (2 * ndraw)])
                if a < int(p_hot * 2 ** 32):
                    return int(hs[(b * len(hs)) >> 32])
                return (b * E) >> 32

            out[i, l] = _distinct_draws(draw, 1, k, E)[0]
    return out, cl


def routing_weights(T: int, k: int, seed: int = 0, stream: int = S_LOGIT, n0: int = 0) -> np.ndarray:
    """topk_w [T, k] fp32: softmax of N(0,1) logits (computed in fp64)."""
    z = normals(seed, stream, T * k, n0).reshape(T, k)
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


# ------------------------------------------------------- device-side filling

_HERE = os.path.dirname(os.path.abspath(__file__))
_CU = os.path.join(_HERE, "synth_fill.cu")
_SO = os.path.join(_HERE, "libsynth.so")
_dev = None


def build(nvcc: str = "nvcc", force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_CU):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc, "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-Xcompiler", "-fPIC", "-shared", _CU, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


def _devlib():
    global _dev
    if _dev is None:
        build()
        L = ctypes.CDLL(_SO)
        P, U64 = ctypes.c_void_p, ctypes.c_uint64
        L.synth_fill_bytes.restype = ctypes.c_int
        L.synth_fill_bytes.argtypes = [P, U64, U64, U64, U64, P]
        L.synth_fill_range.restype = ctypes.c_int
        L.synth_fill_range.argtypes = [P, U64, U64, U64, U64, ctypes.c_int, ctypes.c_int, P]
        _dev = L
    return _dev


def device_fill_bytes(dptr: int, nbytes: int, seed: int, stream: int, offset: int = 0,
                      cuda_stream: int = 0) -> None:
    """Device memory [dptr, dptr+nbytes) <- random_bytes(seed, stream, nbytes, offset)."""
    rc = _devlib().synth_fill_bytes(dptr, nbytes, seed, stream, offset, cuda_stream)
    if rc:
        raise RuntimeError(f"synth_fill_bytes failed ({rc})")


def device_fill_range(dptr: int, nbytes: int, seed: int, stream: int, lo: int, hi: int,
                      offset: int = 0, cuda_stream: int = 0) -> None:
    rc = _devlib().synth_fill_range(dptr, nbytes, seed, stream, offset, lo, hi, cuda_stream)
    if rc:
        raise RuntimeError(f"synth_fill_range failed ({rc})")


def device_fill_expert(codes_ptr: int, scales_ptr: int, hidden: int, inter: int, expert: int,
                       layer: int = 0, seed: int = 0, cuda_stream: int = 0,
                       scale_lo: int = 119, scale_hi: int = 127) -> None:
    nc, ns = expert_sizes(hidden, inter)
    device_fill_bytes(codes_ptr, nc, seed, expert_stream(layer, expert, S_CODES), 0, cuda_stream)
    device_fill_range(scales_ptr, ns, seed, expert_stream(layer, expert, S_SCALES), scale_lo, scale_hi,
                      0, cuda_stream)
