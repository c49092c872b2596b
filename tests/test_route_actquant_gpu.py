"""GPU parity of the integer steps against the oracle, bit for bit: the
token -> expert grouping (counts, offsets, perm, inv) and the E4M3 / ue8m0-per-
128 activation quantizer.  Each case also runs several times and must give
identical bytes every time (the act_quant race on the pages was visible only as
run-to-run variation)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import oracle
import synth
from conftest import golden

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


def _handle(E, k, max_tokens, H=256, I=128):
    return moe.moe_ffn_create(moe.config(E, H, I, k, max_tokens), 0)


def _route_gpu(h, idx, E):
    T, k = idx.shape
    it = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((max(1, T * k),), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((max(1, T * k),), -7, dtype=torch.int32, device="cuda")
    moe.moe_ffn_route(h, it, T, counts, offsets, perm, inv)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (counts, offsets, perm[:T * k], inv[:T * k])]


@pytest.mark.parametrize("T,E,k,dist", [
    (1, 384, 6, "uniform"), (64, 384, 6, "uniform"), (512, 384, 6, "zipf"),
    (32, 128, 6, "uniform"), (7, 8, 2, "uniform"), (1000, 16, 4, "zipf"), (3, 5000, 3, "uniform"),
])
def test_route_bit_exact(T, E, k, dist):
    idx = synth.routing_zipf(T, E, k, seed=T) if dist == "zipf" else synth.routing_uniform(T, E, k, seed=T)
    h = _handle(E, k, T)
    try:
        ref = oracle.route(idx, E)
        for _ in range(5):
            got = _route_gpu(h, idx, E)
            for g, r, name in zip(got, ref, ("counts", "offsets", "perm", "inv")):
                assert np.array_equal(g, r), name
        assert moe.moe_ffn_status(h) == moe.MOE_OK
    finally:
        moe.moe_ffn_destroy(h)


def test_route_repeated_ids_and_bad_ids():
    E, k, T = 8, 3, 4
    idx = np.array([[1, 1, 2], [7, 0, 7], [3, 9, 3], [-1, 5, 5]], np.int32)
    h = _handle(E, k, T)
    try:
        counts, offsets, perm, inv = _route_gpu(h, idx, E)
        assert moe.moe_ffn_status(h) == moe.MOE_ERR_BAD_INDEX
        ok = idx.copy().reshape(-1)
        valid = (ok >= 0) & (ok < E)
        # oracle on the valid slots only, mapped back to slot ids
        slots = np.nonzero(valid)[0]
        ref_perm = [int(j) for e in range(E) for j in slots if ok[j] == e]
        assert list(perm[:len(ref_perm)]) == ref_perm
        assert np.all(perm[len(ref_perm):] == -1)
        assert np.all(inv[~valid] == -1)
        assert np.array_equal(inv[perm[:len(ref_perm)]], np.arange(len(ref_perm)))
        assert list(counts) == [int((ok == e).sum()) for e in range(E)]
        assert offsets[-1] == len(ref_perm)
    finally:
        moe.moe_ffn_destroy(h)


def _act_quant_gpu(h, x_bits):
    rows, n = x_bits.shape
    xt = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    codes = torch.empty((rows, n), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, (n + 127) // 128), dtype=torch.uint8, device="cuda")
    moe.moe_ffn_act_quant(h, xt, rows, n, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _act_quant_ref(x_bits):
    rows, n = x_bits.shape
    vals = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    cs, ss = [], []
    for r in range(rows):
        c, s = oracle.act_quant_e4m3(vals[r], 128)
        cs.append(c)
        ss.append(s)
    return np.stack(cs), np.stack(ss)


@pytest.mark.parametrize("rows", [int(r[0]) for r in golden("act_quant_rows.txt")])
def test_act_quant_bit_exact_at_page_row_counts(rows):
    h = _handle(8, 2, 1)
    try:
        x = synth.activations_bf16(rows, 4096, seed=rows)
        ref = _act_quant_ref(x)
        for _ in range(5):
            got = _act_quant_gpu(h, x)
            assert np.array_equal(got[1], ref[1]), "scales"
            assert np.array_equal(got[0], ref[0]), "codes"
    finally:
        moe.moe_ffn_destroy(h)


def test_act_quant_edge_values_and_ragged_tail():
    h = _handle(8, 2, 1)
    try:
        n = 2880                                     # 22 full blocks and a 64-wide tail
        rng = np.random.default_rng(5)
        v = (rng.standard_normal((6, n)) * 2.0 ** rng.integers(-30, 30, (6, 1))).astype(np.float32)
        v[1, :128] = 0.0                              # zero block -> scale byte 127
        v[2, 5] = -0.0
        v[2, 200:232] = 1e-40                         # subnormal values
        v[3, 300] = 448.0 * 2.0 ** 20                 # amax exactly on a scale boundary
        v[4, 1000] = 3.0e38                           # near the bf16 maximum
        v[5, :] = np.float32(2.0 ** -130)             # subnormal block maximum
        x = synth.f32_to_bf16_bits(v)
        ref = _act_quant_ref(x)
        got = _act_quant_gpu(h, x)
        assert np.array_equal(got[1], ref[1])
        assert np.array_equal(got[0], ref[0])
    finally:
        moe.moe_ffn_destroy(h)
