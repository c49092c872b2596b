"""Pins of the CPU oracle against facts fixed outside it: the pages' printed
values, closed forms, textbook/library routines and brute force.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import golden

TINY = dict(E=8, k=2, H=256, I=128)


# -------------------------------------------------------------- helpers

def e2m1_bitfield(code):
    """E2M1 from its bit fields (1 sign, 2 exponent, 1 mantissa bit, bias 1):
    exponent 0 is subnormal m * 0.5, else 2^(e-1) * (1 + m/2)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -mag if s else mag


def dequant_bitfield(codes, scales, rows, k):
    """Dense fp64 matrix [rows][k] from packed codes (low nibble first) and
    per-32 ue8m0 scales, via the bit-field definition and numpy ldexp."""
    c = np.asarray(codes, np.uint8).reshape(rows, k // 2)
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(rows, k).astype(np.int64)
    tab = np.array([e2m1_bitfield(i) for i in range(16)])
    w = tab[nib]
    sc = np.asarray(scales, np.uint8).reshape(rows, k // 32).astype(np.int64)
    return w * np.ldexp(1.0, np.repeat(sc, 32, axis=1) - 127)


def tiny_experts(E, H, I, seed=0):
    return [synth.expert_canonical(H, I, e, seed=seed) for e in range(E)]


def split_expert(codes, scales, H, I):
    gc, gs = I * H // 2, I * H // 32
    Wg = dequant_bitfield(codes[:gc], scales[:gs], I, H)
    Wu = dequant_bitfield(codes[gc:2 * gc], scales[gs:2 * gs], I, H)
    Wd = dequant_bitfield(codes[2 * gc:], scales[2 * gs:], H, I)
    return Wg, Wu, Wd


# ---------------------------------------------------------------- E2M1

def test_e2m1_doubled_values_match_pages():
    page = sorted(int(r[0]) for r in golden("e2m1_doubled_values.txt"))
    doubled = [2 * oracle.e2m1_value(c) for c in range(16)]
    assert all(float(d).is_integer() for d in doubled)
    assert sorted({abs(int(d)) for d in doubled}) == page
    # each magnitude appears once with each sign (0 as +0 and -0)
    assert sorted(int(d) for d in doubled) == sorted([-v for v in page] + page)


def test_e2m1_table_equals_bitfield_definition():
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert v == e2m1_bitfield(c)
        assert math.copysign(1.0, v) == (-1.0 if c >= 8 else 1.0)


def test_e2m1_all_256_products_brute_force():
    page = [int(r[0]) for r in golden("e2m1_doubled_values.txt")]
    allowed = {a * b for a in page for b in page}
    seen = set()
    for a in range(16):
        for b in range(16):
            p = oracle.e2m1_value(a) * oracle.e2m1_value(b)
            q = 4 * p
            assert q.is_integer() and -144 <= q <= 144
            assert abs(int(q)) in allowed
            assert p == e2m1_bitfield(a) * e2m1_bitfield(b)
            seen.add(int(q))
    assert max(seen) == 144 and min(seen) == -144


# ---------------------------------------------------------------- ue8m0

def test_ue8m0_powers_of_two():
    assert oracle.ue8m0_value(127) == 1.0
    assert oracle.ue8m0_value(128) == 2.0
    assert oracle.ue8m0_value(119) == 2.0 ** -8
    assert oracle.ue8m0_value(0) == math.ldexp(1.0, -127)
    assert math.isnan(oracle.ue8m0_value(255))
    for s in range(254):
        assert oracle.ue8m0_value(s + 1) == 2 * oracle.ue8m0_value(s)


# ------------------------------------------------------------ bf16, E4M3

def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                           [0.0, -0.0, 1.0, 3.0e38, 1e-40, -2.5e-39]]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)
    # exact ties in fp64 that are not fp32 values: 1 + 2^-8 -> 1, 1 + 3*2^-8 -> 1 + 2^-6
    assert oracle.bf16_rne(1 + 2.0 ** -8) == 0x3F80
    assert oracle.bf16_rne(1 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.bf16_rne(1 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert oracle.e4m3_value(0x7E) == 448.0


def _e4m3_brute(v):
    """Nearest finite E4M3 by search over all codes; ties to the even code;
    saturating at 448; sign kept."""
    a = abs(v)
    best, bd = None, None
    for c in range(0x7F):                    # all non-negative finite codes
        d = abs(oracle.e4m3_value(c) - a)
        if bd is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best | (0x80 if math.copysign(1.0, v) < 0 else 0)


def test_e4m3_rne_equals_brute_force_on_all_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = synth.bf16_bits_to_f32(bits).astype(np.float64)
    finite = np.isfinite(vals) & (np.abs(vals) < 1e4)
    big = np.isfinite(vals) & (np.abs(vals) >= 1e4)
    # saturation: every finite value at or beyond the largest code maps to +-448
    assert all(oracle.e4m3_rne(float(v)) == (0xFE if v < 0 else 0x7E) for v in vals[big])
    grid = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    # vectorised brute force: nearest grid point, ties to even code
    a = np.abs(vals[finite])[:, None]
    d = np.abs(grid[None, :] - a)
    dmin = d.min(axis=1, keepdims=True)
    cand = (d == dmin)
    even = cand & (np.arange(0x7F)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    ref = pick | np.where(np.signbit(vals[finite]), 0x80, 0)
    got = np.array([oracle.e4m3_rne(float(v)) for v in vals[finite]])
    assert np.array_equal(got, ref)
    # spot-check the scalar brute force on a few values, including saturation
    for v in [0.0, -0.0, 1e-9, -1e-9, 2.0 ** -10, 3 * 2.0 ** -10, 447.9, 449.0, 470.0, 1e6, -1e6]:
        assert oracle.e4m3_rne(v) == _e4m3_brute(v)


def test_e4m3_rne_matches_torch_in_range():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 9, 20000)).astype(np.float32)
    v = v[np.abs(v) < 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_rne(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, ref)


def test_ue8m0_for_amax_boundaries():
    assert oracle.ue8m0_for_amax(0.0) == 127
    for k in range(-40, 41):
        edge = math.ldexp(448.0, k)
        assert oracle.ue8m0_for_amax(edge) == 127 + k
        assert oracle.ue8m0_for_amax(math.nextafter(edge, math.inf)) == 128 + k
        assert oracle.ue8m0_for_amax(math.ldexp(448.0, k - 1) * 1.0000001) == 127 + k
    assert oracle.ue8m0_for_amax(math.inf) == 255


def test_act_quant_scale_is_minimal_and_codes_fit():
    rng = np.random.default_rng(3)
    for n in (1, 17, 300, 1024, 2880):
        v = rng.standard_normal(n) * 2.0 ** rng.integers(-20, 20)
        codes, scales = oracle.act_quant_e4m3(v, 128)
        for b, s in enumerate(scales):
            blk = v[b * 128:(b + 1) * 128]
            k = int(s) - 127
            amax = np.abs(blk).max()
            assert amax <= 448.0 * 2.0 ** k and amax > 448.0 * 2.0 ** (k - 1)
            for i, x in enumerate(blk):
                assert codes[b * 128 + i] == _e4m3_brute(x / 2.0 ** k) or abs(x / 2.0 ** k) > 440


# ------------------------------------------------ E2M1 activations (MXFP4)

E2M1_GRID = np.array([e2m1_bitfield(c) for c in range(8)])     # 0, .5, 1, 1.5, 2, 3, 4, 6


def _e2m1_brute(v):
    """Nearest E2M1 code by brute force over the bit-field grid: ties to the
    code whose mantissa bit is 0, magnitudes above 6 saturate."""
    a = abs(v)
    if a >= 6.0:
        return 7 | (8 if math.copysign(1.0, v) < 0 else 0)
    d = np.abs(E2M1_GRID - a)
    best = [c for c in range(8) if d[c] == d.min()]
    c = best[0] if len(best) == 1 else [b for b in best if b & 1 == 0][0]
    return c | (8 if math.copysign(1.0, v) < 0 else 0)


def _e2m1_qd_numpy(v, block=32):
    """Independent MXFP4 quantize-dequantize: per block the least k with
    amax <= 6 * 2^k (log2 then exact correction), vectorised nearest grid
    value with ties to the even mantissa."""
    out = np.empty_like(v)
    for b0 in range(0, v.size, block):
        blk = v[b0:b0 + block]
        amax = np.abs(blk).max()
        k = 0 if amax == 0 else math.ceil(math.log2(amax / 6.0))
        while amax > 6.0 * 2.0 ** k:
            k += 1
        while amax != 0 and amax <= 6.0 * 2.0 ** (k - 1):
            k -= 1
        a = np.abs(blk) / 2.0 ** k
        d = np.abs(a[:, None] - E2M1_GRID[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = (d == dmin)
        even = cand & ((np.arange(8) & 1) == 0)[None, :]
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        out[b0:b0 + block] = np.sign(blk) * E2M1_GRID[pick] * 2.0 ** k
    return out


def test_e2m1_rne_equals_brute_force_on_all_bf16():
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(vals)
    for v in vals[finite]:
        assert oracle.e2m1_rne(float(v)) == _e2m1_brute(float(v)), v


def test_e2m1_rne_ties_and_saturation():
    # the midpoints of the grid go to the even mantissa
    for v, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert oracle.e2m1_rne(v) == c and oracle.e2m1_rne(-v) == c | 8
    assert oracle.e2m1_rne(6.0) == 7 and oracle.e2m1_rne(1e30) == 7 and oracle.e2m1_rne(-7.0) == 15


def test_ue8m0_for_amax_e2m1_boundaries():
    assert oracle.ue8m0_for_amax_e2m1(0.0) == 127
    for k in range(-40, 41):
        edge = math.ldexp(6.0, k)
        assert oracle.ue8m0_for_amax_e2m1(edge) == 127 + k
        assert oracle.ue8m0_for_amax_e2m1(math.nextafter(edge, math.inf)) == 128 + k
        assert oracle.ue8m0_for_amax_e2m1(math.ldexp(6.0, k - 1) * 1.0000001) == 127 + k
    assert oracle.ue8m0_for_amax_e2m1(math.inf) == 255


def test_act_quant_e2m1_scale_is_minimal_and_codes_are_nearest():
    rng = np.random.default_rng(4)
    for n in (1, 31, 64, 300, 2880):
        v = rng.standard_normal(n) * 2.0 ** rng.integers(-20, 20)
        codes, scales = oracle.act_quant_e2m1(v, 32)
        for b, s in enumerate(scales):
            blk = v[b * 32:(b + 1) * 32]
            k = int(s) - 127
            amax = np.abs(blk).max()
            assert amax <= 6.0 * 2.0 ** k and amax > 6.0 * 2.0 ** (k - 1)
            for i, x in enumerate(blk):
                assert codes[b * 32 + i] == _e2m1_brute(x / 2.0 ** k)


def test_act_quant_e2m1_fixed_points():
    # a block of E2M1 values times 2^k (holding +-6 * 2^k) quantizes to itself
    rng = np.random.default_rng(5)
    for k in (-9, -1, 0, 3, 17):
        c = rng.integers(0, 16, 32)
        c[7] = 7
        v = np.array([e2m1_bitfield(int(x)) for x in c]) * 2.0 ** k
        codes, scales = oracle.act_quant_e2m1(v, 32)
        assert scales[0] == 127 + k
        assert np.array_equal(np.array([e2m1_bitfield(int(x)) for x in codes]) * 2.0 ** k, v)


# --------------------------------------------------------------- SiLU

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    for g in [0.1, 1.0, 3.7, 20.0]:
        # g*sigmoid(g) - (-g)*sigmoid(-g) = g
        assert abs(oracle.silu(g) - oracle.silu(-g) - g) < 1e-15 * max(1.0, g)
    assert oracle.silu(800.0) == 800.0
    assert oracle.silu(-800.0) == 0.0


# ------------------------------------------------------------ bytes

def test_expert_byte_sizes_match_pages():
    g = {r[0]: float(r[1]) for r in golden("expert_bytes.txt")}
    nc, ns = synth.expert_sizes(4096, 2880)
    assert round(nc / 1e6, 1) == g["expert_codes"]
    assert round(ns / 1e6, 1) == g["expert_scales"]
    assert round((nc + ns) / 2 ** 20, 2) == g["expert_total"]
    per_token = g["layers"] * g["topk"] * (nc + ns)
    assert round(per_token / 2 ** 30, 1) == g["per_token"]
    total = g["layers"] * g["experts_per_layer"] * (nc + ns)
    assert round(total / 2 ** 30) == g["expert_set"]
    # one ue8m0 byte per 16 code bytes, i.e. per 32 weights
    assert nc == 16 * ns


# ------------------------------------------------------------ matvec/FFN

def test_matvec_one_hot_reads_dequantized_column():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 3, seed=5)
    gc, gs = I * H // 2, I * H // 32
    W = dequant_bitfield(codes[:gc], scales[:gs], I, H)
    for j in (0, 1, 31, 32, 77, 255):
        x = np.zeros(H)
        x[j] = 1.0
        assert np.array_equal(oracle.matvec(codes[:gc], scales[:gs], I, H, x), W[:, j])


def test_matvec_equals_dense_matmul():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 1, seed=7)
    Wg, Wu, Wd = split_expert(codes, scales, H, I)
    x = np.random.default_rng(0).standard_normal(H)
    gc, gs = I * H // 2, I * H // 32
    ref = Wu @ x
    got = oracle.matvec(codes[gc:2 * gc], scales[gs:2 * gs], I, H, x)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())
    h = np.random.default_rng(1).standard_normal(I)
    got = oracle.matvec(codes[2 * gc:], scales[2 * gs:], H, I, h)
    assert np.allclose(got, Wd @ h, rtol=1e-13, atol=1e-13 * np.abs(Wd @ h).max())


def test_expert_ffn_zero_input_gives_exact_zero():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 0)
    for mode in (oracle.ACT_BF16, oracle.ACT_E4M3_UE8M0_128, oracle.ACT_E2M1_UE8M0_32):
        o = oracle.expert_ffn(codes, scales, H, I, np.zeros(H), mode)
        assert np.all(o == 0.0)


def test_expert_ffn_one_hot_closed_form():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 2)
    Wg, Wu, Wd = split_expert(codes, scales, H, I)
    j = 41
    x = np.zeros(H)
    x[j] = 1.0
    g, u = Wg[:, j], Wu[:, j]
    h = g / (1 + np.exp(-g)) * u
    ref = Wd @ h
    got = oracle.expert_ffn(codes, scales, H, I, x)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_expert_ffn_equals_dense_definition():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 4)
    Wg, Wu, Wd = split_expert(codes, scales, H, I)
    x = synth.bf16_bits_to_f32(synth.activations_bf16(1, H)[0]).astype(np.float64)
    g, u = Wg @ x, Wu @ x
    ref = Wd @ (g / (1 + np.exp(-g)) * u)
    got = oracle.expert_ffn(codes, scales, H, I, x)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_expert_ffn_e4m3_mode_equals_dense_definition():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 5)
    Wg, Wu, Wd = split_expert(codes, scales, H, I)
    x = synth.bf16_bits_to_f32(synth.activations_bf16(1, H)[0]).astype(np.float64)

    def qd(v):
        out = np.empty_like(v)
        for b0 in range(0, v.size, 128):
            blk = v[b0:b0 + 128]
            amax = np.abs(blk).max()
            k = 0 if amax == 0 else math.ceil(math.log2(amax / 448.0))
            while amax > 448.0 * 2.0 ** k:
                k += 1
            while amax <= 448.0 * 2.0 ** (k - 1):
                k -= 1
            q = torch.from_numpy((blk / 2.0 ** k).astype(np.float32)).to(torch.float8_e4m3fn)
            out[b0:b0 + 128] = q.to(torch.float64).numpy() * 2.0 ** k
        return out

    xq = qd(x)
    g, u = Wg @ xq, Wu @ xq
    h = qd(g / (1 + np.exp(-g)) * u)
    ref = Wd @ h
    got = oracle.expert_ffn(codes, scales, H, I, x, oracle.ACT_E4M3_UE8M0_128)
    # h crosses an fp32 rounding in the torch quantizer; allow rare rounding flips
    err = np.abs(got - ref).max() / np.sqrt(np.mean(ref ** 2))
    assert err < 1e-3


def test_expert_ffn_e2m1_mode_equals_dense_definition():
    H, I = 256, 128
    codes, scales = synth.expert_canonical(H, I, 6)
    Wg, Wu, Wd = split_expert(codes, scales, H, I)
    x = synth.bf16_bits_to_f32(synth.activations_bf16(1, H, seed=8)[0]).astype(np.float64)
    xq = _e2m1_qd_numpy(x)
    g, u = Wg @ xq, Wu @ xq
    ref = Wd @ _e2m1_qd_numpy(g / (1 + np.exp(-g)) * u)
    got = oracle.expert_ffn(codes, scales, H, I, x, oracle.ACT_E2M1_UE8M0_32)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # and the mode does quantize: it differs from the bf16 path
    assert not np.allclose(got, oracle.expert_ffn(codes, scales, H, I, x), rtol=1e-3)


def _tiny_layer(seed=0):
    E, H, I = TINY["E"], TINY["H"], TINY["I"]
    ex = tiny_experts(E, H, I, seed)
    return [c for c, _ in ex], [s for _, s in ex]


def test_moe_ffn_combine_linear_and_one_hot():
    E, k, H, I = TINY["E"], TINY["k"], TINY["H"], TINY["I"]
    cl, sl = _tiny_layer()
    T = 3
    x = synth.activations_bf16(T, H)
    idx = synth.routing_uniform(T, E, k)
    w1 = synth.routing_weights(T, k)
    w2 = synth.routing_weights(T, k, seed=9)
    y1 = oracle.moe_ffn(cl, sl, H, I, x, idx, w1)
    y2 = oracle.moe_ffn(cl, sl, H, I, x, idx, w2)
    y12 = oracle.moe_ffn(cl, sl, H, I, x, idx, (w1.astype(np.float64) + w2).astype(np.float32))
    scale = np.abs(y12).max()
    # w1 + w2 is rounded to fp32; the difference is at most 2^-24 relative per weight
    assert np.abs(y12 - (y1 + y2)).max() <= 1e-6 * scale
    # one-hot topk_w picks out a single expert
    onehot = np.zeros((T, k), np.float32)
    onehot[:, 1] = 1.0
    y = oracle.moe_ffn(cl, sl, H, I, x, idx, onehot)
    for t in range(T):
        xt = synth.bf16_bits_to_f32(x[t]).astype(np.float64)
        e = idx[t, 1]
        assert np.array_equal(y[t], oracle.expert_ffn(cl[e], sl[e], H, I, xt))


def test_moe_ffn_slot_order_invariance_and_dense_reference():
    E, k, H, I = TINY["E"], TINY["k"], TINY["H"], TINY["I"]
    cl, sl = _tiny_layer(seed=3)
    T = 2
    x = synth.activations_bf16(T, H, seed=3)
    idx = synth.routing_uniform(T, E, k, seed=3)
    w = synth.routing_weights(T, k, seed=3)
    y = oracle.moe_ffn(cl, sl, H, I, x, idx, w)
    yp = oracle.moe_ffn(cl, sl, H, I, x, idx[:, ::-1], w[:, ::-1])
    assert np.allclose(y, yp, rtol=0, atol=1e-12 * np.abs(y).max())
    # dense reference with numpy matmuls, a different summation order
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            Wg, Wu, Wd = split_expert(cl[idx[t, j]], sl[idx[t, j]], H, I)
            g, u = Wg @ xf[t], Wu @ xf[t]
            ref[t] += float(w[t, j]) * (Wd @ (g / (1 + np.exp(-g)) * u))
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_moe_ffn_threads_do_not_change_result():
    E, k, H, I = TINY["E"], TINY["k"], TINY["H"], TINY["I"]
    cl, sl = _tiny_layer()
    x = synth.activations_bf16(4, H)
    idx = synth.routing_uniform(4, E, k)
    w = synth.routing_weights(4, k)
    a = oracle.moe_ffn(cl, sl, H, I, x, idx, w, nthreads=1)
    b = oracle.moe_ffn(cl, sl, H, I, x, idx, w, nthreads=3)
    assert np.array_equal(a, b)


def test_moe_ffn_rejects_bad_expert():
    E, k, H, I = TINY["E"], TINY["k"], TINY["H"], TINY["I"]
    cl, sl = _tiny_layer()
    x = synth.activations_bf16(1, H)
    with pytest.raises(ValueError):
        oracle.moe_ffn(cl, sl, H, I, x, np.array([[0, E]], np.int32), np.ones((1, k), np.float32))
    cl[5] = None
    sl[5] = None
    with pytest.raises(ValueError):
        oracle.moe_ffn(cl, sl, H, I, x, np.array([[5, 1]], np.int32), np.ones((1, k), np.float32))


# ---------------------------------------------------------------- routing

def test_route_equals_brute_force_scan():
    for T, E, k, zipf in [(1, 384, 6, False), (64, 384, 6, False), (512, 384, 6, True), (7, 8, 2, False)]:
        idx = synth.routing_zipf(T, E, k) if zipf else synth.routing_uniform(T, E, k)
        counts, offsets, perm, inv = oracle.route(idx, E)
        flat = idx.reshape(-1)
        ref_perm = [j for e in range(E) for j in range(T * k) if flat[j] == e]
        assert list(perm) == ref_perm
        assert list(counts) == [int((flat == e).sum()) for e in range(E)]
        assert offsets[0] == 0 and offsets[-1] == T * k
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(inv[perm], np.arange(T * k))
        assert sorted(perm) == list(range(T * k))


# --------------------------------------------------------------- RMSNorm/stack

def test_rmsnorm_matches_torch_and_closed_form():
    x = np.random.default_rng(4).standard_normal((3, 4096)) * 3.0
    got = oracle.rmsnorm_bf16(x, 1e-6)
    xt = torch.from_numpy(x)
    ref64 = xt / torch.sqrt((xt * xt).mean(dim=-1, keepdim=True) + 1e-6)
    ref = ref64.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    # fp64 -> fp32 -> bf16 may double-round; allow a 1-ulp difference on rare ties
    diff = np.abs(got.astype(np.int32) - ref.astype(np.int32))
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
    c = np.full((1, 64), 2.5)
    assert np.all(synth.bf16_bits_to_f32(oracle.rmsnorm_bf16(c, 0.0)) == 1.0)


def test_stack_is_composition_of_layers():
    E, k, H, I = TINY["E"], TINY["k"], TINY["H"], TINY["I"]
    L, T = 3, 2
    layers = []
    for l in range(L):
        ex = [synth.expert_canonical(H, I, e, layer=l) for e in range(E)]
        layers.append(([c for c, _ in ex], [s for _, s in ex], H, I))
    idx = np.stack([synth.routing_uniform(T, E, k, seed=l) for l in range(L)])
    w = np.stack([synth.routing_weights(T, k, seed=l) for l in range(L)])
    x0 = synth.activations_f32(T, H).astype(np.float64)
    got = oracle.moe_stack(layers, x0, idx, w)
    x = x0.copy()
    for l in range(L):
        u = oracle.rmsnorm_bf16(x, 1e-6)
        x = x + oracle.moe_ffn(layers[l][0], layers[l][1], H, I, u, idx[l], w[l])
    assert np.array_equal(got, x)


# ---- router ahead of the path: top-k of the router logits, softmax of the selected

def _rank_brute_force(row, k):
    """Expert ids ordered by (logit descending, id ascending), NaN last, by a
    plain sort of (key, id) pairs."""
    keys = [((1, 0.0) if np.isnan(v) else (0, -v), e) for e, v in enumerate(row)]
    return [e for _, e in sorted(keys)][:k]


def test_topk_selection_equals_a_sort_with_ties_and_nan():
    rng = np.random.default_rng(11)
    for E, k in ((40, 1), (40, 6), (40, 40), (384, 6)):
        l = rng.choice([-2.0, -0.5, 0.0, 0.5, 1.0, 3.0], size=(30, E))     # many ties
        l[3, 5] = np.nan
        l[4, :] = np.nan
        idx, w = oracle.topk_softmax(l, k)
        for t in range(l.shape[0]):
            assert list(idx[t]) == _rank_brute_force(l[t], k)


def test_topk_softmax_closed_form_and_normalization():
    rng = np.random.default_rng(12)
    l = rng.standard_normal((50, 16))
    idx, w = oracle.topk_softmax(l, 2)
    d = l[np.arange(50), idx[:, 1]] - l[np.arange(50), idx[:, 0]]
    assert np.allclose(w[:, 0], 1.0 / (1.0 + np.exp(d)), rtol=0, atol=1e-15)
    idx, w = oracle.topk_softmax(l, 6)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (np.diff(w, axis=1) <= 0).all()          # descending logits -> descending weights


def test_router_logits_one_hot_zero_and_matmul():
    E, H = 24, 256
    W = synth.router_weights_bf16(E, H)
    one = synth.f32_to_bf16_bits(np.float32([1.0]))[0]
    for j in (0, 77, 255):
        x = np.zeros((1, H), np.uint16)
        x[0, j] = one
        got = oracle.router_logits(x, W)[0]
        assert np.array_equal(got, synth.bf16_bits_to_f32(W[:, j]).astype(np.float64))
    z = oracle.router_logits(np.zeros((2, H), np.uint16), W)
    assert not z.any()
    idx, w = oracle.topk_softmax(z, 6)
    assert (idx == np.arange(6)).all() and np.allclose(w, 1.0 / 6, rtol=0, atol=1e-16)
    x = synth.activations_bf16(3, H, seed=4)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
    assert np.allclose(oracle.router_logits(x, W), ref, rtol=1e-13, atol=1e-13)
