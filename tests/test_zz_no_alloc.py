"""moe_ffn_forward_noalloc: the layer for callers that may not allocate device
memory on their call path (hosts that own every device allocation), with its
scratch in the library's fixed device array.  Its output must match
moe_ffn_forward's within the parity tolerance, on two calls in a row (the
array keeps the previous call's contents, so the second call checks that the
per-call clearing is right).  Collected last so that a failure here stops a
-x run only after every other test has run."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import synth
from moe_setup import assert_close, fill_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


@pytest.mark.parametrize("E,H,I,k,T", [(384, 4096, 2880, 6, 1), (16, 1024, 448, 6, 3)])
def test_noalloc_matches_forward_on_two_calls(E, H, I, k, T):
    cfg = moe.config(E, H, I, k, T, out_dtype=moe.MOE_OUT_F32)
    h = moe.moe_ffn_create(cfg, 0)
    try:
        es = fill_layer(h, cfg)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for call in range(2):
            x = torch.from_numpy(synth.activations_bf16(T, H, seed=40 + call).view(np.int16)).cuda()
            idx = torch.from_numpy(synth.routing_uniform(T, E, k, seed=40 + call)).cuda()
            w = torch.from_numpy(synth.routing_weights(T, k, seed=40 + call)).cuda()
            y_ref = torch.empty((T, H), dtype=torch.float32, device="cuda")
            y_na = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
            moe.moe_ffn_forward(h, x, idx, w, es.table, y_ref, T)
            moe.moe_ffn_forward_noalloc(cfg, 0, x, idx, w, es.table, y_na, T, status=status)
            torch.cuda.synchronize()
            assert_close(y_na.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64),
                         f"noalloc call {call}")
        assert int(status.item()) == 0
    finally:
        moe.moe_ffn_destroy(h)


def test_noalloc_alternating_shapes_match_forward():
    """Back-to-back calls of different shapes (T=3 at H=1024, then T=1 at
    H=4096, and back): every area of the shared array moves, except the
    launch-tagged partial sums, which sit at fixed offsets; each call must
    still equal moe_ffn_forward of its own shape."""
    shapes = [(16, 1024, 448, 6, 3), (384, 4096, 2880, 6, 1)]
    layers = []
    try:
        for E, H, I, k, T in shapes:
            cfg = moe.config(E, H, I, k, T, out_dtype=moe.MOE_OUT_F32)
            h = moe.moe_ffn_create(cfg, 0)
            layers.append((cfg, h, fill_layer(h, cfg)))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        for call, which in enumerate([0, 1, 0, 1, 0]):
            cfg, h, es = layers[which]
            E, H, I, k, T = shapes[which]
            x = torch.from_numpy(synth.activations_bf16(T, H, seed=70 + call).view(np.int16)).cuda()
            idx = torch.from_numpy(synth.routing_uniform(T, E, k, seed=70 + call)).cuda()
            w = torch.from_numpy(synth.routing_weights(T, k, seed=70 + call)).cuda()
            y_ref = torch.empty((T, H), dtype=torch.float32, device="cuda")
            y_na = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
            moe.moe_ffn_forward(h, x, idx, w, es.table, y_ref, T)
            moe.moe_ffn_forward_noalloc(cfg, 0, x, idx, w, es.table, y_na, T, status=status)
            torch.cuda.synchronize()
            assert_close(y_na.cpu().numpy(), y_ref.cpu().numpy().astype(np.float64), f"noalloc call {call}")
        assert int(status.item()) == 0
    finally:
        for _, h, _ in layers:
            moe.moe_ffn_destroy(h)


def test_noalloc_rejects_a_problem_larger_than_its_array():
    E, H, I, k = 384, 4096, 2880, 6
    cfg = moe.config(E, H, I, k, 64)
    T = 64                                   # about 15 MB of scratch: beyond the fixed array
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    ptrs = torch.zeros(E, dtype=torch.int64, device="cuda")
    table = moe.expert_table(ptrs)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_ffn_forward_noalloc(cfg, 0, x, idx, w, table, y, T)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED
