"""Failure paths, driven without a GPU fault, trap or hang: a bounded device
wait that is made to run out (the slot-major kernel's first CTA keeps back its
partial sums, the others' waits give up after a shortened limit), and host
allocations that are made to fail.  Each call must return cleanly with its
error code, and the next normal call must work."""
import time

import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import synth
from moe_setup import Layer, assert_close, inputs

pytestmark = pytest.mark.gpu
TINY = dict(E=8, H=256, I=128, k=2)
MID = dict(E=16, H=1024, I=448, k=6)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield
    moe.moe_ffn_test_fail_allocs(0)


@pytest.mark.parametrize("shape,T", [(TINY, 1), (MID, 3)])
def test_timed_out_wait_reports_and_handle_recovers(shape, T):
    L = Layer(**shape, max_tokens=T)
    try:
        x, idx, w = inputs(T, shape["E"], shape["H"], shape["k"], seed=61)
        ref = L.oracle(x, idx, w)
        assert_close(L.run(x, idx, w).cpu().numpy(), ref, "before")
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK

        moe.moe_ffn_test_set_wait(L.h, 1_000_000, True)     # 1 ms, partial sums withheld
        t0 = time.perf_counter()
        L.run(x, idx, w)                                      # synchronizes
        took = time.perf_counter() - t0
        assert moe.moe_ffn_status(L.h) == moe.MOE_ERR_DEVICE_TIMEOUT
        assert took < 1.0, f"the timed-out call took {took:.3f} s"
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK          # read clears it

        moe.moe_ffn_test_set_wait(L.h, 0, False)
        y = L.run(x, idx, w).cpu().numpy()
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
        assert_close(y, ref, "after the timeout")
        assert np.array_equal(y, L.run(x, idx, w).cpu().numpy())
    finally:
        L.close()


def test_failed_workspace_allocation_returns_oom():
    cfg = moe.config(TINY["E"], TINY["H"], TINY["I"], TINY["k"], 4)
    moe.moe_ffn_test_fail_allocs(1)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_ffn_create(cfg, 0)
    assert e.value.code == moe.MOE_ERR_OOM
    moe.moe_ffn_test_fail_allocs(0)
    h = moe.moe_ffn_create(cfg, 0)                            # nothing left behind
    moe.moe_ffn_destroy(h)


def test_failed_staging_allocation_returns_oom_and_next_call_works():
    T = 1
    L = Layer(**TINY, max_tokens=T)
    try:
        x, idx, w = inputs(T, TINY["E"], TINY["H"], TINY["k"], seed=62)
        idx = np.ascontiguousarray(idx, np.int32)
        w = np.ascontiguousarray(w, np.float32)
        y = np.zeros((T, TINY["H"]), np.float32)
        args = (x.ctypes.data, idx.ctypes.data, w.ctypes.data, L.es.table, y.ctypes.data, T)
        moe.moe_ffn_test_fail_allocs(1)                       # the page-locked staging buffer
        with pytest.raises(moe.MoeError) as e:
            moe.moe_ffn_forward_host(L.h, *args)
        assert e.value.code == moe.MOE_ERR_OOM
        moe.moe_ffn_test_fail_allocs(0)
        moe.moe_ffn_forward_host(L.h, *args)
        assert_close(y, L.oracle(x, idx, w), "host call after a failed staging allocation")
    finally:
        L.close()


def test_failed_cache_allocation_returns_oom():
    cfg = moe.config(TINY["E"], TINY["H"], TINY["I"], TINY["k"], 1)
    blob = moe.moe_ffn_packed_expert_bytes(cfg)
    host = torch.empty(TINY["E"] * ((blob + 255) // 256 * 256), dtype=torch.uint8).pin_memory()
    ptrs = [host.data_ptr() + e * ((blob + 255) // 256 * 256) for e in range(TINY["E"])]
    for n in (1, 2, 3):                                       # device slots, device table, staging
        moe.moe_ffn_test_fail_allocs(n)
        with pytest.raises(moe.MoeError) as e:
            moe.moe_expert_cache_create(cfg, 0, ptrs, 4)
        assert e.value.code == moe.MOE_ERR_OOM
        moe.moe_ffn_test_fail_allocs(0)
    c = moe.moe_expert_cache_create(cfg, 0, ptrs, 4)
    moe.moe_expert_cache_destroy(c)
