"""Empty work through every entry point that takes a batch: T = 0 (and a
stack of L = 0 layers) returns MOE_OK, launches nothing that writes, and
leaves every output as it was."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import synth
from moe_setup import Layer

pytestmark = pytest.mark.gpu


def test_zero_tokens_and_zero_layers_leave_outputs_untouched():
    E, H, I, k = 8, 256, 128, 2
    L = Layer(E=E, H=H, I=I, k=k, max_tokens=4)
    try:
        sentinel = 12345.0
        x = torch.zeros((1, H), dtype=torch.int16, device="cuda")
        idx = torch.zeros((1, k), dtype=torch.int32, device="cuda")
        w = torch.ones((1, k), dtype=torch.float32, device="cuda")
        y = torch.full((1, H), sentinel, dtype=torch.float32, device="cuda")
        moe.moe_ffn_forward(L.h, x, idx, w, L.es.table, y, 0)
        xh = torch.zeros((1, H), dtype=torch.int16)
        yh = torch.full((1, H), sentinel, dtype=torch.float32)
        moe.moe_ffn_forward_host(L.h, xh, idx.cpu(), w.cpu(), L.es.table, yh, 0)
        xs = torch.full((1, H), sentinel, dtype=torch.float32, device="cuda")
        moe.moe_stack_forward(L.h, xs, [L.es.table], idx.view(1, 1, k), w.view(1, 1, k), 1, 0)
        moe.moe_stack_forward(L.h, xs, [], idx.view(1, 1, k), w.view(1, 1, k), 0, 1)
        xsh = torch.full((1, H), sentinel, dtype=torch.float32)
        moe.moe_stack_forward_host(L.h, xsh, [L.es.table], idx.cpu().view(1, 1, k), w.cpu().view(1, 1, k), 1, 0)
        moe.moe_stack_forward_host(L.h, xsh, [], idx.cpu().view(1, 1, k), w.cpu().view(1, 1, k), 0, 1)
        Wr = torch.from_numpy(synth.router_weights_bf16(E, H).view(np.int16)).cuda()
        ri = torch.full((1, k), -7, dtype=torch.int32, device="cuda")
        rw = torch.full((1, k), sentinel, dtype=torch.float32, device="cuda")
        moe.moe_router_topk(L.h, x, Wr, 0, ri, rw)
        torch.cuda.synchronize()
        assert torch.all(y == sentinel) and torch.all(yh == sentinel)
        assert torch.all(xs == sentinel) and torch.all(xsh == sentinel)
        assert torch.all(ri == -7) and torch.all(rw == sentinel)
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
    finally:
        L.close()
