"""GPU parity of the expert-major (grouped) path against the CPU oracle,
through the C ABI: route -> pieces in group order -> one persistent kernel for
both projections (MMA columns = up to 8 slots of one expert) -> combine.
Float outputs: max|err| <= 2e-3 * rms(ref), cosine >= 0.99999."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import oracle
import synth
from moe_setup import e4m3_flip_candidates, Layer, assert_close, bf16_to_f64, fill_layer, host_experts, inputs

pytestmark = pytest.mark.gpu

TINY = dict(E=8, H=256, I=128, k=2)
MID = dict(E=16, H=1024, I=448, k=6)      # down K = 448: 3 full units + a 64-wide half unit
E4M3 = moe.MOE_ACT_E4M3_UE8M0_128


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


@pytest.mark.parametrize("act", [moe.MOE_ACT_BF16, E4M3])
@pytest.mark.parametrize("T", [1, 2, 5, 17, 40])
def test_tiny_grouped_matches_oracle(T, act):
    """8 experts, top-2: at T = 40 every expert holds about 10 slots, i.e. one
    full group of 8 and a ragged one."""
    L = Layer(**TINY, max_tokens=64, act=act, path="group")
    try:
        x, idx, w = inputs(T, TINY["E"], TINY["H"], TINY["k"], seed=50 + T)
        assert_close(L.run(x, idx, w).cpu().numpy(), L.oracle(x, idx, w), f"tiny grouped T={T} act={act}")
    finally:
        L.close()


@pytest.mark.parametrize("act", [moe.MOE_ACT_BF16, E4M3])
@pytest.mark.parametrize("T", [3, 24])
def test_mid_grouped_ragged_k_tail_matches_oracle(T, act):
    L = Layer(**MID, max_tokens=32, act=act, path="group")
    try:
        x, idx, w = inputs(T, MID["E"], MID["H"], MID["k"], seed=60 + T)
        assert_close(L.run(x, idx, w).cpu().numpy(), L.oracle(x, idx, w), f"mid grouped T={T} act={act}")
    finally:
        L.close()


def test_one_hot_expert_many_groups():
    """Every token's first slot on expert 3 (41 slots: five groups of 8 and one
    of 1 for that expert), the others uniform: the (expert, tile, group) job
    order with several groups per expert."""
    T = 41
    L = Layer(**MID, max_tokens=T, path="group")
    try:
        x, idx, w = inputs(T, MID["E"], MID["H"], MID["k"], seed=7)
        for t in range(T):
            if 3 in idx[t]:
                j = int(np.nonzero(idx[t] == 3)[0][0])
                idx[t, j] = idx[t, 0]
            idx[t, 0] = 3
        assert (np.sort(idx, axis=1)[:, 1:] != np.sort(idx, axis=1)[:, :-1]).all()
        assert_close(L.run(x, idx, w).cpu().numpy(), L.oracle(x, idx, w), "hot expert")
    finally:
        L.close()


def test_grouped_and_slot_major_agree():
    T = 12
    Lg = Layer(**MID, max_tokens=T, path="group")
    Ls = Layer(**MID, max_tokens=T, path="slot")
    try:
        x, idx, w = inputs(T, MID["E"], MID["H"], MID["k"], seed=9)
        yg = Lg.run(x, idx, w).cpu().numpy()
        ys = Ls.run(x, idx, w).cpu().numpy()
        ref = Lg.oracle(x, idx, w)
        assert_close(yg, ref, "grouped")
        assert_close(ys, ref, "slot-major")
    finally:
        Lg.close()
        Ls.close()


def test_grouped_deterministic_and_bf16_out_is_rounded_f32():
    T = 20
    Lf = Layer(**MID, max_tokens=T, path="group")
    Lb = Layer(**MID, max_tokens=T, path="group", out=moe.MOE_OUT_BF16)
    try:
        x, idx, w = inputs(T, MID["E"], MID["H"], MID["k"], seed=11)
        ys = [Lf.run(x, idx, w).view(torch.int32).clone() for _ in range(5)]
        assert all(torch.equal(ys[0], y) for y in ys[1:])
        yb = Lb.run(x, idx, w)
        assert torch.equal(ys[0].view(torch.float32).to(torch.bfloat16).view(torch.int16), yb.view(torch.int16))
        ref = Lf.oracle(x, idx, w)
        yb64 = bf16_to_f64(yb).reshape(ref.shape)
        rms = np.sqrt(np.mean(ref ** 2))
        half_ulp = np.ldexp(1.0, np.floor(np.log2(np.abs(ref) + 1e-300)).astype(int) - 8)
        assert np.all(np.abs(yb64 - ref) <= 2e-3 * rms + half_ulp)
    finally:
        Lf.close()
        Lb.close()


def test_grouped_zero_input_and_bad_index():
    T = 6
    L = Layer(**TINY, max_tokens=T, path="group")
    try:
        x, idx, w = inputs(T, TINY["E"], TINY["H"], TINY["k"], seed=13)
        assert torch.count_nonzero(L.run(np.zeros_like(x), idx, w)).item() == 0
        bad = idx.copy()
        bad[1, 1] = TINY["E"] + 5
        bad[4, 0] = -1
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
        y = L.run(x, bad, w).cpu().numpy()
        assert moe.moe_ffn_status(L.h) == moe.MOE_ERR_BAD_INDEX
        ok, w0 = bad.copy(), w.copy()
        for t, j in ((1, 1), (4, 0)):
            ok[t, j] = 0
            w0[t, j] = 0.0
        assert_close(y, L.oracle(x, ok, w0), "bad slots dropped")
        # every slot invalid: y = 0
        y = L.run(x, np.full_like(idx, -7), w)
        assert torch.count_nonzero(y).item() == 0
        assert moe.moe_ffn_status(L.h) == moe.MOE_ERR_BAD_INDEX
    finally:
        L.close()


def test_grouped_stack_matches_oracle():
    E, H, I, k, Lnum, T = 8, 256, 128, 2, 4, 20
    cfg = moe.config(E, H, I, k, T, gemm_min_tokens=1)
    h = moe.moe_ffn_create(cfg, 0)
    try:
        sets = [fill_layer(h, cfg, layer=l) for l in range(Lnum)]
        idx = np.stack([synth.routing_uniform(T, E, k, seed=300 + l) for l in range(Lnum)])
        w = np.stack([synth.routing_weights(T, k, seed=300 + l) for l in range(Lnum)])
        x0 = synth.activations_f32(T, H, seed=17)
        x = torch.from_numpy(x0.copy()).cuda()
        it, wt = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
        moe.moe_stack_forward(h, x, [s.table for s in sets], it, wt, Lnum, T)
        torch.cuda.synchronize()
        layers = []
        for l in range(Lnum):
            c, s = host_experts(H, I, idx[l].reshape(-1), layer=l, E=E)
            layers.append((c, s, H, I))
        ref = oracle.moe_stack(layers, x0.astype(np.float64), idx, w)
        assert_close(x.cpu().numpy(), ref, "grouped stack")
        assert_close(x.cpu().numpy() - x0, ref - x0, "grouped stack delta")
    finally:
        moe.moe_ffn_destroy(h)


def test_full_size_batch64_e4m3_grouped_all_tokens():
    """384 experts, H=4096, I=2880, top-6, 64 tokens, uniform routing, E4M3:
    the batch-64 configuration on the path the library picks for it."""
    T = 64
    L = Layer(E=384, H=4096, I=2880, k=6, max_tokens=T, act=E4M3, path="auto")
    try:
        x, idx, w = inputs(T, 384, 4096, 6, seed=3)
        y = L.run(x, idx, w).cpu().numpy()
        assert_close(y, L.oracle(x, idx, w), "full-size grouped e4m3 T=64")
        assert np.array_equal(y, L.run(x, idx, w).cpu().numpy())
        # diagnostic: elements of h that may round to the other E4M3 neighbour
        # on the GPU (fp32 h) than in the oracle (fp64 h), on four tokens
        n, tot = e4m3_flip_candidates(4096, 2880, 384, x[:4], idx[:4])
        print(f"E4M3 h: {n} of {tot} elements within 1e-4 of a rounding midpoint or scale boundary")
    finally:
        L.close()


@pytest.mark.parametrize("path,T", [("slot", 1), ("slot", 5), ("group", 3), ("group", 20)])
@pytest.mark.parametrize("E,k", [(1, 1), (8, 8)])
@pytest.mark.parametrize("act", [moe.MOE_ACT_BF16, E4M3])
def test_degenerate_routing_shapes(E, k, path, T, act):
    """A single expert chosen by every token (E = k = 1: one group of all the
    slots on the expert-major path), and every expert chosen by every token
    (k = E = 8): both paths against the oracle."""
    L = Layer(E=E, H=256, I=128, k=k, max_tokens=24, act=act, path=path)
    try:
        x, idx, w = inputs(T, E, 256, k, seed=300 + 10 * E + T)
        assert sorted(idx[0].tolist()) == list(range(E)) if k == E else True
        assert_close(L.run(x, idx, w).cpu().numpy(), L.oracle(x, idx, w), f"E={E} k={k} {path} T={T} act={act}")
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
    finally:
        L.close()
