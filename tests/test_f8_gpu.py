"""GPU parity of the expert-major path's kind::mxf8f6f4 form (E4M3
activations times E2M1 weights on the tensor core, one slot per MMA column,
groups of up to 224 slots) against the CPU oracle's E4M3 mode, through the C
ABI.  Shapes span the MMA's N range (16 to 224 columns, one and two scale
atoms), experts cut into several groups, a down projection with a 64-wide
last K unit, and the stack's fused RMSNorm.  Float outputs: max|err| <=
2e-3 * rms(ref), cosine >= 0.99999."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import oracle
import synth
from moe_setup import (Layer, assert_close, assert_close_e2m1, assert_close_e4m3, check_f8_h_and_down,
                       e2m1_flip_bound, e4m3_flip_candidates, host_experts, inputs)

pytestmark = pytest.mark.gpu

E4M3 = moe.MOE_ACT_E4M3_UE8M0_128
E2M1 = moe.MOE_ACT_E2M1_UE8M0_32
F8 = moe.MOE_MMA_MXF8F6F4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


@pytest.mark.parametrize("E,H,I,k,T", [
    (8, 256, 128, 2, 16),        # groups of about 4 slots: N = 16
    (8, 256, 448, 2, 40),        # down K = 448: three units and a half unit
    (4, 256, 192, 2, 300),       # about 150 slots an expert: N up to 160, two scale atoms
    (16, 1024, 448, 6, 64),      # 384 slots over 16 experts
])
def test_f8_layer_matches_oracle(E, H, I, k, T):
    L = Layer(E, H, I, k, max_tokens=T, act=E4M3, path="group", mma=F8)
    try:
        x, idx, w = inputs(T, E, H, k, seed=80 + T)
        y = L.run(x, idx, w).cpu().numpy()
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
        assert_close_e4m3(y, L.oracle(x, idx, w), (H, I, E, x, idx, w), f"f8 E={E} H={H} I={I} k={k} T={T}")
        # h itself, and the down step on the GPU's own quantized h
        flips, total = check_f8_h_and_down(L.h, H, I, E, x, idx, w, y, what=f"f8 T={T}")
        cand, _ = e4m3_flip_candidates(H, I, E, x, idx)
        print(f"E4M3 rounding decisions of h that differ from the oracle's: {flips} of {total} "
              f"({cand} within 1e-4 of a step midpoint or scale boundary)")
        assert flips <= cand
        # bit-identical on a repeat
        assert np.array_equal(L.run(x, idx, w).cpu().numpy(), y)
    finally:
        L.close()


def test_f8_experts_over_several_groups():
    """Two experts, both chosen by every one of 600 tokens: 600 slots each,
    cut into groups of 224, 224 and 152 (N = 224, 224, 160)."""
    E, H, I, k, T = 2, 256, 128, 2, 600
    L = Layer(E, H, I, k, max_tokens=T, act=E4M3, path="group", mma=F8)
    try:
        x = synth.activations_bf16(T, H, seed=3)
        idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
        idx[1::2] = idx[1::2, ::-1]
        w = synth.routing_weights(T, k, seed=3)
        y = L.run(x, idx, w).cpu().numpy()
        assert_close_e4m3(y, L.oracle(x, idx, w), (H, I, E, x, idx, w), "f8 600 slots per expert")
    finally:
        L.close()


def test_f8_and_pieces_agree():
    """The kind::mxf8f6f4 path and the kind::mxf4 pieces path compute the same
    function: each within the tolerance of the oracle."""
    E, H, I, k, T = 16, 1024, 448, 6, 24
    Lf = Layer(E, H, I, k, max_tokens=T, act=E4M3, path="group", mma=F8)
    Lp = Layer(E, H, I, k, max_tokens=T, act=E4M3, path="group", mma=moe.MOE_MMA_MXF4_PIECES)
    try:
        x, idx, w = inputs(T, E, H, k, seed=12)
        yf = Lf.run(x, idx, w).cpu().numpy()
        yp = Lp.run(x, idx, w).cpu().numpy()
        ref = Lf.oracle(x, idx, w)
        assert_close_e4m3(yf, ref, (H, I, E, x, idx, w), "f8")
        assert_close_e4m3(yp, ref, (H, I, E, x, idx, w), "pieces")
    finally:
        Lf.close()
        Lp.close()


def test_f8_zero_input_gives_zero():
    """Zero activations: every E4M3 code and h is zero, so is y."""
    E, H, I, k, T = 8, 256, 128, 2, 20
    L = Layer(E, H, I, k, max_tokens=T, act=E4M3, path="group", mma=F8)
    try:
        x, idx, w = inputs(T, E, H, k, seed=5)
        z = np.zeros_like(x)
        assert not np.any(L.run(z, idx, w).cpu().numpy())
    finally:
        L.close()


def test_f8_stack_fused_rmsnorm_matches_oracle():
    """Four layers on one residual stream at T = 48 (RMSNorm fused into the
    prep kernel), one cached graph, checked against the oracle's stack."""
    E, H, I, k, T, NL = 8, 256, 448, 2, 48, 4
    cfg = moe.config(E, H, I, k, T, act_mode=E4M3, gemm_min_tokens=1)
    h = moe.moe_ffn_create(cfg, 0)
    moe.moe_ffn_set_mma_kind(h, F8)
    from moe_setup import fill_layer
    sets = []
    try:
        sets = [fill_layer(h, cfg, layer=l) for l in range(NL)]
        idx = np.stack([synth.routing_uniform(T, E, k, seed=400 + l) for l in range(NL)])
        w = np.stack([synth.routing_weights(T, k, seed=400 + l) for l in range(NL)])
        x0 = synth.activations_f32(T, H, seed=21)
        x = torch.from_numpy(x0.copy()).cuda()
        moe.moe_stack_forward(h, x, [s.table for s in sets], torch.from_numpy(idx).cuda(),
                              torch.from_numpy(w).cuda(), NL, T)
        torch.cuda.synchronize()
        assert moe.moe_ffn_status(h) == moe.MOE_OK
        layers = []
        for l in range(NL):
            c, sc = host_experts(H, I, np.arange(E), layer=l, E=E)
            layers.append((c, sc, H, I))
        ref = oracle.moe_stack(layers, x0.astype(np.float64), idx, w, act_mode=oracle.ACT_E4M3_UE8M0_128,
                               nthreads=8)
        assert_close(x.cpu().numpy() - x0, ref - x0, "f8 stack")
    finally:
        del sets
        moe.moe_ffn_destroy(h)


@pytest.mark.parametrize("E,H,I,k,T", [
    (8, 256, 128, 2, 16),        # gate/up K = 256: two units; N = 16
    (8, 256, 448, 2, 40),        # down K = 448: a 64-wide last unit (one K = 64 MMA)
    (4, 256, 192, 2, 300),       # N up to 160: two scale atoms
    (16, 1024, 448, 6, 64),
])
def test_mxf4_direct_e2m1_matches_oracle(E, H, I, k, T):
    """The E2M1 activation mode on the same direct form, kind::mxf4: E2M1 weights
    as the blob holds them times the E2M1 rows of x and h (one per slot),
    against the oracle's E2M1 mode with its bound for h's E2M1 rounding flips."""
    L = Layer(E, H, I, k, max_tokens=T, act=E2M1, path="group", mma=F8)
    try:
        x, idx, w = inputs(T, E, H, k, seed=90 + T)
        y = L.run(x, idx, w).cpu().numpy()
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
        bound, n = e2m1_flip_bound(H, I, E, x, idx, w)
        assert_close_e2m1(y, L.oracle(x, idx, w), bound, f"mxf4 direct E={E} H={H} I={I} T={T} ({n} flips allowed)")
        assert np.array_equal(L.run(x, idx, w).cpu().numpy(), y)
    finally:
        L.close()


def test_mxf4_direct_and_pieces_agree_e2m1():
    """Both E2M1-mode forms (direct and one piece per value) against the oracle."""
    E, H, I, k, T = 16, 1024, 448, 6, 24
    Ld = Layer(E, H, I, k, max_tokens=T, act=E2M1, path="group", mma=F8)
    Lp = Layer(E, H, I, k, max_tokens=T, act=E2M1, path="group", mma=moe.MOE_MMA_MXF4_PIECES)
    try:
        x, idx, w = inputs(T, E, H, k, seed=13)
        bound, _ = e2m1_flip_bound(H, I, E, x, idx, w)
        ref = Ld.oracle(x, idx, w)
        assert_close_e2m1(Ld.run(x, idx, w).cpu().numpy(), ref, bound, "direct")
        assert_close_e2m1(Lp.run(x, idx, w).cpu().numpy(), ref, bound, "pieces")
    finally:
        Ld.close()
        Lp.close()


def test_mma_kind_change_replaces_the_cached_stack_graph():
    """The stack's cached graph holds the MMA kind it was captured with: after
    moe_ffn_set_mma_kind the same call (same pointers) runs the new kind, bit
    for bit what a fresh handle set to that kind computes, and switching back
    gives the first result again."""
    E, H, I, k, T, NL = 8, 256, 448, 2, 48, 3
    cfg = moe.config(E, H, I, k, T, act_mode=E4M3, gemm_min_tokens=1)
    from moe_setup import fill_layer
    h = moe.moe_ffn_create(cfg, 0)
    h2 = moe.moe_ffn_create(cfg, 0)
    try:
        sets = [fill_layer(h, cfg, layer=l) for l in range(NL)]
        idx = torch.from_numpy(np.stack([synth.routing_uniform(T, E, k, seed=500 + l) for l in range(NL)])).cuda()
        w = torch.from_numpy(np.stack([synth.routing_weights(T, k, seed=500 + l) for l in range(NL)])).cuda()
        x0 = torch.from_numpy(synth.activations_f32(T, H, seed=22)).cuda()
        x = torch.empty_like(x0)
        tables = [s.table for s in sets]

        def run(hh):
            x.copy_(x0)
            moe.moe_stack_forward(hh, x, tables, idx, w, NL, T)
            torch.cuda.synchronize()
            return x.clone()

        moe.moe_ffn_set_mma_kind(h, F8)
        y_f8 = run(h)
        moe.moe_ffn_set_mma_kind(h, moe.MOE_MMA_MXF4_PIECES)
        y_pc = run(h)
        moe.moe_ffn_set_mma_kind(h2, moe.MOE_MMA_MXF4_PIECES)
        y_pc_ref = run(h2)
        moe.moe_ffn_set_mma_kind(h, F8)
        y_f8_again = run(h)
        assert torch.equal(y_pc.view(torch.int32), y_pc_ref.view(torch.int32))
        assert torch.equal(y_f8.view(torch.int32), y_f8_again.view(torch.int32))
        assert not torch.equal(y_f8.view(torch.int32), y_pc.view(torch.int32))   # the two kinds differ in rounding
        assert moe.moe_ffn_status(h) == moe.MOE_OK
    finally:
        moe.moe_ffn_destroy(h)
        moe.moe_ffn_destroy(h2)
