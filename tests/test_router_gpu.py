"""GPU parity of the router ahead of the path (logits = W x, top-k with ties to
the lower expert id, softmax of the selected logits) against the oracle,
through the C ABI."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import oracle
import synth
from moe_setup import Layer, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


def _handle(E, H, k, T):
    return moe.moe_ffn_create(moe.config(E, H, 128, k, T), 0)


def test_select_is_bit_exact_given_logits():
    E, k, T = 384, 6, 37
    rng = np.random.default_rng(21)
    l = rng.choice(np.float32([-1.5, -0.25, 0.0, 0.75, 2.0]), size=(T, E)).astype(np.float32)   # many ties
    l[:, 100] += rng.standard_normal(T).astype(np.float32)
    l[3, 7] = np.nan
    l[4, :] = np.nan
    h = _handle(E, 256, k, T)
    try:
        ld = torch.from_numpy(l).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        moe.moe_router_select(h, ld, T, idx, w)
        torch.cuda.synchronize()
        ridx, rw = oracle.topk_softmax(l.astype(np.float64), k)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        ok = ~np.isnan(rw).any(axis=1)
        assert np.abs(w.cpu().numpy()[ok] - rw[ok]).max() <= 2e-6
    finally:
        moe.moe_ffn_destroy(h)


@pytest.mark.parametrize("T", [1, 8, 9, 16, 37, 64, 300])
def test_router_full_size_matches_oracle(T):
    """T <= 8 on the CUDA cores, above on the tensor cores (tiles of 16..256
    tokens, split-K partials); 300 leaves a ragged second tile."""
    E, H, k = 384, 4096, 6
    W = synth.router_weights_bf16(E, H, layer=1)
    x = synth.activations_bf16(T, H, seed=30 + T)
    h = _handle(E, H, k, T)
    try:
        wd = torch.from_numpy(W.view(np.int16)).cuda()
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        moe.moe_router_topk(h, xd, wd, T, idx, w, logits=logits)
        torch.cuda.synchronize()
        got_l = logits.cpu().numpy().astype(np.float64)
        ref_l = oracle.router_logits(x, W)
        err = np.abs(got_l - ref_l).max()
        assert err <= 1e-5, f"router logits max|err| = {err:.3e}"
        gi, gw = idx.cpu().numpy(), w.cpu().numpy()
        # the selection is exactly the oracle's selection of the GPU's logits
        ci, cw = oracle.topk_softmax(got_l, k)
        assert np.array_equal(gi, ci)
        assert np.abs(gw - cw).max() <= 2e-6
        # and the oracle's own selection wherever its k-th / (k+1)-th margin is clear
        ri, rw = oracle.topk_softmax(ref_l, k)
        srt = -np.sort(-ref_l, axis=1)
        clear = (srt[:, k - 1] - srt[:, k]) > 10 * err + 1e-7
        assert clear.sum() >= T // 2
        assert np.array_equal(gi[clear], ri[clear])
        # the workspace path (no logits output) and a repeat give the same result
        idx2 = torch.empty_like(idx)
        w2 = torch.empty_like(w)
        moe.moe_router_topk(h, xd, wd, T, idx2, w2)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx2) and torch.equal(w.view(torch.int32), w2.view(torch.int32))
    finally:
        moe.moe_ffn_destroy(h)


def test_router_then_layer_matches_oracle():
    """Router on the device, its routing straight into the layer."""
    E, H, I, k, T = 8, 256, 128, 2, 5
    L = Layer(E=E, H=H, I=I, k=k, max_tokens=T)
    try:
        W = synth.router_weights_bf16(E, H, layer=2)
        x = synth.activations_bf16(T, H, seed=41)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        moe.moe_router_topk(L.h, xd, torch.from_numpy(W.view(np.int16)).cuda(), T, idx, w)
        y = torch.empty((T, H), dtype=torch.float32, device="cuda")
        moe.moe_ffn_forward(L.h, xd, idx, w, L.es.table, y, T)
        torch.cuda.synchronize()
        ri, rw = oracle.topk_softmax(oracle.router_logits(x, W), k)
        assert np.array_equal(idx.cpu().numpy(), ri)
        ref = L.oracle(x, ri, rw.astype(np.float32))
        assert_close(y.cpu().numpy(), ref, "router -> layer")
    finally:
        L.close()


@pytest.mark.parametrize("E", [64, 128, 200, 256])
def test_one_token_cluster_router_matches_oracle(E):
    """A single token with up to 256 experts: one thread-block cluster computes
    the logits (one warp per expert row) and its first CTA selects from them in
    shared memory; logits within 1e-5 of the oracle's, the selection exactly
    the oracle's selection of the GPU's logits, twelve calls in a row on one
    handle (fresh inputs each time) all equal to it."""
    H, k = 4096, 6
    W = synth.router_weights_bf16(E, H, layer=4)
    h = _handle(E, H, k, 1)
    try:
        wd = torch.from_numpy(W.view(np.int16)).cuda()
        for step in range(12):
            x = synth.activations_bf16(1, H, seed=90 + step)
            xd = torch.from_numpy(x.view(np.int16)).cuda()
            logits = torch.empty((1, E), dtype=torch.float32, device="cuda")
            idx = torch.full((1, k), -7, dtype=torch.int32, device="cuda")
            w = torch.empty((1, k), dtype=torch.float32, device="cuda")
            moe.moe_router_topk(h, xd, wd, 1, idx, w, logits=logits)
            torch.cuda.synchronize()
            got_l = logits.cpu().numpy().astype(np.float64)
            assert np.abs(got_l - oracle.router_logits(x, W)).max() <= 1e-5
            ci, cw = oracle.topk_softmax(got_l, k)
            assert np.array_equal(idx.cpu().numpy(), ci), f"step {step}"
            assert np.abs(w.cpu().numpy() - cw).max() <= 2e-6
        assert moe.moe_ffn_status(h) == moe.MOE_OK
    finally:
        moe.moe_ffn_destroy(h)


@pytest.mark.parametrize("E", [130, 384, 1000])
def test_single_launch_router_repeats_and_ragged_expert_rows(E):
    """At T <= 8 one launch computes the logits and, in the last CTA of each
    token tile, the selection (a per-tile counter cleared by that CTA): many
    calls in a row on one handle, T varying, E not a multiple of the CTA's
    warps (idle warps in the last CTA), each equal to the oracle's selection
    of the GPU's logits."""
    H, k = 512, 6
    W = synth.router_weights_bf16(E, H, layer=2)
    h = _handle(E, H, k, 8)
    try:
        wd = torch.from_numpy(W.view(np.int16)).cuda()
        for step, T in enumerate([1, 3, 8, 2, 1, 5, 8, 4]):
            x = synth.activations_bf16(T, H, seed=70 + step)
            xd = torch.from_numpy(x.view(np.int16)).cuda()
            logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
            idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
            w = torch.empty((T, k), dtype=torch.float32, device="cuda")
            moe.moe_router_topk(h, xd, wd, T, idx, w, logits=logits)
            torch.cuda.synchronize()
            got_l = logits.cpu().numpy().astype(np.float64)
            assert np.abs(got_l - oracle.router_logits(x, W)).max() <= 1e-5
            ci, cw = oracle.topk_softmax(got_l, k)
            assert np.array_equal(idx.cpu().numpy(), ci), f"step {step}, T {T}"
            assert np.abs(w.cpu().numpy() - cw).max() <= 2e-6
        assert moe.moe_ffn_status(h) == moe.MOE_OK
    finally:
        moe.moe_ffn_destroy(h)


@pytest.mark.parametrize("T", [1, 4, 20])
def test_router_feeds_layer_on_one_stream_without_waits(T):
    """Router then layer, step after step on one stream with no host wait, the
    routing buffers reused: the layer's first kernels read topk_idx before
    their griddepcontrol.wait, so the router must let them start only after
    it has written it.  Each step's y equals a later, synchronized forward of
    the same step's routing, bit for bit."""
    E, H, I, k = 16, 4096, 2880, 6
    L = Layer(E=E, H=H, I=I, k=k, max_tokens=T, path="auto")
    s = torch.cuda.Stream()
    try:
        Wd = torch.from_numpy(synth.router_weights_bf16(E, H, layer=3).view(np.int16)).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        steps = 6
        xs = [torch.from_numpy(synth.activations_bf16(T, H, seed=90 + i).view(np.int16)).cuda() for i in range(steps)]
        ys = [torch.empty((T, H), dtype=torch.float32, device="cuda") for _ in range(steps)]
        idx_s = [torch.empty_like(idx) for _ in range(steps)]
        w_s = [torch.empty_like(w) for _ in range(steps)]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for i in range(steps):
                moe.moe_router_topk(L.h, xs[i], Wd, T, idx, w, stream=s)
                moe.moe_ffn_forward(L.h, xs[i], idx, w, L.es.table, ys[i], T, s)
                idx_s[i].copy_(idx)
                w_s[i].copy_(w)
        s.synchronize()
        for i in range(steps):
            y_ref = torch.empty_like(ys[i])
            moe.moe_ffn_forward(L.h, xs[i], idx_s[i], w_s[i], L.es.table, y_ref, T)
            torch.cuda.synchronize()
            assert torch.equal(ys[i].view(torch.int32), y_ref.view(torch.int32)), f"step {i}"
        assert len({tuple(t.cpu().numpy().ravel()) for t in idx_s}) > 1       # the routing did change
        assert moe.moe_ffn_status(L.h) == moe.MOE_OK
    finally:
        L.close()



@pytest.mark.parametrize("T", [1, 4, 20])
def test_routing_wait_gives_identical_results(T):
    """moe_ffn_set_routing_wait(h, 1) (the routing read after the layer's
    dependency wait) changes no bit: a forward and a 3-layer stack with the
    setting on equal the same calls with it off (the cached stack graph is
    dropped and captured again at each change), and router -> layer chained on
    one stream without host waits (the router now letting the layer start at
    once, one launch at T <= 8, logits + selection above) stays equal to the
    synchronized forwards."""
    E, H, I, k, L = 16, 4096, 2880, 6, 3
    lay = Layer(E=E, H=H, I=I, k=k, max_tokens=T)
    try:
        x = synth.activations_bf16(T, H, seed=140 + T)
        idx = synth.routing_uniform(T, E, k, seed=140 + T)
        w = synth.routing_weights(T, k, seed=140 + T)
        y_off = lay.run(x, idx, w)
        moe.moe_ffn_set_routing_wait(lay.h, 1)
        y_on = lay.run(x, idx, w)
        assert torch.equal(y_off.view(torch.int32), y_on.view(torch.int32))
        # a stack of L layers (the handle's experts in every layer), on then off
        it = torch.from_numpy(np.stack([synth.routing_uniform(T, E, k, seed=150 + l) for l in range(L)])).cuda()
        wt = torch.from_numpy(np.stack([synth.routing_weights(T, k, seed=150 + l) for l in range(L)])).cuda()
        x0 = torch.from_numpy(synth.activations_f32(T, H, seed=160)).cuda()
        outs = []
        for on in (1, 0, 1):
            moe.moe_ffn_set_routing_wait(lay.h, on)
            xs = x0.clone()
            moe.moe_stack_forward(lay.h, xs, [lay.es.table] * L, it, wt, L, T)
            torch.cuda.synchronize()
            outs.append(xs)
        assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
        assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))
        # router -> layer chained with the setting on
        moe.moe_ffn_set_routing_wait(lay.h, 1)
        Wd = torch.from_numpy(synth.router_weights_bf16(E, H, layer=5).view(np.int16)).cuda()
        s = torch.cuda.Stream()
        ri = torch.empty((T, k), dtype=torch.int32, device="cuda")
        rw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        xs_ = [torch.from_numpy(synth.activations_bf16(T, H, seed=170 + i).view(np.int16)).cuda() for i in range(4)]
        ys = [torch.empty((T, H), dtype=torch.float32, device="cuda") for _ in range(4)]
        ri_s = [torch.empty_like(ri) for _ in range(4)]
        rw_s = [torch.empty_like(rw) for _ in range(4)]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for i in range(4):
                moe.moe_router_topk(lay.h, xs_[i], Wd, T, ri, rw, stream=s)
                moe.moe_ffn_forward(lay.h, xs_[i], ri, rw, lay.es.table, ys[i], T, s)
                ri_s[i].copy_(ri)
                rw_s[i].copy_(rw)
        s.synchronize()
        for i in range(4):
            yr = torch.empty((T, H), dtype=torch.float32, device="cuda")
            moe.moe_ffn_forward(lay.h, xs_[i], ri_s[i], rw_s[i], lay.es.table, yr, T)
            torch.cuda.synchronize()
            assert torch.equal(ys[i].view(torch.int32), yr.view(torch.int32)), f"step {i}"
        assert moe.moe_ffn_status(lay.h) == moe.MOE_OK
    finally:
        lay.close()
