"""GPU parity of the E2M1 activation mode (x and h quantized to E2M1 with one
ue8m0 scale per 32) on both paths against the oracle's E2M1 mode, through the
C ABI.  x's codes are the same on both sides (bf16 in, exact scaling, one
rounding); h is fp32 on the GPU and fp64 in the oracle, so an element lying on
an E2M1 rounding midpoint may take the other code: the comparison allows
exactly those elements' effect (moe_setup.e2m1_flip_bound) on top of the usual
tolerance."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
from moe_setup import Layer, assert_close_e2m1, e2m1_flip_bound, inputs

pytestmark = pytest.mark.gpu

E2M1 = moe.MOE_ACT_E2M1_UE8M0_32
TINY = dict(E=8, H=256, I=128, k=2)
MID = dict(E=16, H=1024, I=448, k=6)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


def _check(L, cfg, T, seed, what):
    x, idx, w = inputs(T, cfg["E"], cfg["H"], cfg["k"], seed=seed)
    y = L.run(x, idx, w).cpu().numpy()
    ref = L.oracle(x, idx, w)
    bound, _ = e2m1_flip_bound(cfg["H"], cfg["I"], cfg["E"], x, idx, w)
    assert_close_e2m1(y, ref, bound, what)
    return y, ref


@pytest.mark.parametrize("path", ["slot", "group"])
@pytest.mark.parametrize("T", [1, 5, 17, 40])
def test_tiny_e2m1_matches_oracle(T, path):
    L = Layer(**TINY, max_tokens=64, act=E2M1, path=path)
    try:
        _check(L, TINY, T, 70 + T, f"tiny e2m1 {path} T={T}")
    finally:
        L.close()


@pytest.mark.parametrize("path,T", [("slot", 3), ("group", 3), ("group", 24)])
def test_mid_e2m1_ragged_k_tail_matches_oracle(path, T):
    """down K = 448: three full units and a 64-wide half unit."""
    L = Layer(**MID, max_tokens=32, act=E2M1, path=path)
    try:
        _check(L, MID, T, 80 + T, f"mid e2m1 {path} T={T}")
    finally:
        L.close()


def test_e2m1_paths_agree_and_differ_from_bf16():
    T = 12
    Ls = Layer(**MID, max_tokens=T, act=E2M1, path="slot")
    Lg = Layer(**MID, max_tokens=T, act=E2M1, path="group")
    Lb = Layer(**MID, max_tokens=T, path="slot")
    try:
        x, idx, w = inputs(T, MID["E"], MID["H"], MID["k"], seed=90)
        ys, yg = Ls.run(x, idx, w).cpu().numpy(), Lg.run(x, idx, w).cpu().numpy()
        ref = Ls.oracle(x, idx, w)
        bound, _ = e2m1_flip_bound(MID["H"], MID["I"], MID["E"], x, idx, w)
        assert_close_e2m1(ys, ref, bound, "slot-major")
        assert_close_e2m1(yg, ref, bound, "expert-major")
        # the quantization is real: the bf16 path's output is measurably different
        yb = Lb.run(x, idx, w).cpu().numpy()
        assert np.abs(yb - ys).max() > 1e-2 * np.sqrt(np.mean(yb ** 2))
        # deterministic
        assert np.array_equal(yg, Lg.run(x, idx, w).cpu().numpy())
    finally:
        Ls.close()
        Lg.close()
        Lb.close()


def test_e2m1_zero_input_and_bad_index():
    T = 6
    for path in ("slot", "group"):
        L = Layer(**TINY, max_tokens=T, act=E2M1, path=path)
        try:
            x, idx, w = inputs(T, TINY["E"], TINY["H"], TINY["k"], seed=91)
            assert torch.count_nonzero(L.run(np.zeros_like(x), idx, w)).item() == 0
            bad = idx.copy()
            bad[2, 1] = -3
            y = L.run(x, bad, w).cpu().numpy()
            assert moe.moe_ffn_status(L.h) == moe.MOE_ERR_BAD_INDEX
            ok, w0 = bad.copy(), w.copy()
            ok[2, 1], w0[2, 1] = 0, 0.0
            bound, _ = e2m1_flip_bound(TINY["H"], TINY["I"], TINY["E"], x, ok, w0)
            assert_close_e2m1(y, L.oracle(x, ok, w0), bound, f"bad slot dropped ({path})")
        finally:
            L.close()


@pytest.mark.parametrize("T", [1, 16])
def test_full_size_e2m1(T):
    """384 experts, H = 4096, I = 2880, top-6: batch 1 on the slot-major path,
    batch 16 on the expert-major path (the library's choice)."""
    L = Layer(E=384, H=4096, I=2880, k=6, max_tokens=T, act=E2M1, path="auto")
    try:
        x, idx, w = inputs(T, 384, 4096, 6, seed=92 + T)
        y = L.run(x, idx, w).cpu().numpy()
        ref = L.oracle(x, idx, w)
        bound, n = e2m1_flip_bound(4096, 2880, 384, x, idx, w)
        assert_close_e2m1(y, ref, bound, f"full-size e2m1 T={T} ({n} elements near a midpoint)")
    finally:
        L.close()
