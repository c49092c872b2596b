"""moe_stack_forward_host (host x / routing, one graph that copies the inputs
in from a mapped staging buffer, runs the layers and copies x back) against
moe_stack_forward on device buffers, bit for bit: both paths (slot-major at
T = 1 and 4, expert-major at T = 8), several calls in a row with fresh inputs
(the staging buffer reused), and a deeper stack after a shallower one (the
staging buffers grown and the cached graphs replaced)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import synth
from moe_setup import Layer

pytestmark = pytest.mark.gpu


def _inputs(L, T, E, H, k, seed):
    x = synth.activations_f32(T, H, seed=seed)
    idx = np.stack([synth.routing_uniform(T, E, k, seed=seed + 1 + l) for l in range(L)]).astype(np.int32)
    w = np.stack([synth.routing_weights(T, k, seed=seed + 1 + l) for l in range(L)]).astype(np.float32)
    return x, idx, w


@pytest.mark.parametrize("T,path", [(1, "slot"), (4, "slot"), (8, "group")])
def test_stack_host_equals_device_stack(T, path):
    E, H, I, k = 16, 4096, 2880, 6
    lay = Layer(E=E, H=H, I=I, k=k, max_tokens=8, path=path)
    try:
        for L, seed in [(3, 10), (3, 20), (5, 30), (3, 40)]:
            x, idx, w = _inputs(L, T, E, H, k, seed)
            tables = [lay.es.table] * L
            xd = torch.from_numpy(x.copy()).cuda()
            moe.moe_stack_forward(lay.h, xd, tables, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), L, T)
            torch.cuda.synchronize()
            xh = torch.from_numpy(x.copy()).pin_memory() if seed % 20 == 0 else torch.from_numpy(x.copy())
            moe.moe_stack_forward_host(lay.h, xh, tables, torch.from_numpy(idx), torch.from_numpy(w), L, T)
            assert torch.equal(xd.cpu().view(torch.int32), xh.view(torch.int32)), f"L={L} seed={seed}"
            assert not np.array_equal(xh.numpy(), x)        # the layers did change x
        assert moe.moe_ffn_status(lay.h) == moe.MOE_OK
    finally:
        lay.close()
