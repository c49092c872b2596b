"""Host-resident experts (packed blobs in page-locked host memory) served
through the HBM expert cache: the layer's output equals, bit for bit, the
output with every expert resident in HBM, over steps that evict; the slot
choices follow least-recently-used exactly (a Python model); prefetched
experts turn into hits."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_gb300 as moe
import synth
from moe_setup import fill_layer

pytestmark = pytest.mark.gpu

MID = dict(E=16, H=1024, I=448, k=6)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.lib()
    yield


class LruModel:
    """Least recently used over `slots`, the request's own slots excluded,
    the lowest slot on ties; hits before misses within a request."""

    def __init__(self, E, slots):
        self.slot_of = [-1] * E
        self.expert_in = [-1] * slots
        self.last = [0] * slots
        self.clock = 0

    def request(self, ids):
        self.clock += 1
        ids = [int(e) for e in ids if e >= 0]
        in_req = [False] * len(self.last)
        for e in ids:
            if self.slot_of[e] >= 0:
                in_req[self.slot_of[e]] = True
        for e in ids:
            s = self.slot_of[e]
            if s >= 0:
                self.last[s] = self.clock
                continue
            cand = [t for t in range(len(self.last)) if not in_req[t]]
            v = min(cand, key=lambda t: (self.last[t], t))
            if self.expert_in[v] >= 0:
                self.slot_of[self.expert_in[v]] = -1
            self.expert_in[v], self.slot_of[e], self.last[v], in_req[v] = e, v, self.clock, True


def _setup(T, slots):
    cfg = moe.config(MID["E"], MID["H"], MID["I"], MID["k"], T, out_dtype=moe.MOE_OUT_F32)
    h = moe.moe_ffn_create(cfg, 0)
    es = fill_layer(h, cfg)
    host = torch.empty(es.E * es.stride, dtype=torch.uint8, pin_memory=True)
    host.copy_(es.blobs.cpu())
    ptrs = [host.data_ptr() + e * es.stride for e in range(es.E)]
    c = moe.moe_expert_cache_create(cfg, 0, ptrs, slots)
    return cfg, h, es, host, c


@pytest.mark.parametrize("T,slots", [(1, 8), (2, 12)])
def test_cache_matches_resident_experts_and_lru(T, slots):
    cfg, h, es, host, c = _setup(T, slots)
    model = LruModel(MID["E"], slots)
    s = torch.cuda.Stream()
    try:
        for step in range(12):
            x = torch.from_numpy(synth.activations_bf16(T, MID["H"], seed=step).view(np.int16)).cuda()
            idx_np = synth.routing_uniform(T, MID["E"], MID["k"], seed=200 + step)
            idx = torch.from_numpy(idx_np).cuda()
            w = torch.from_numpy(synth.routing_weights(T, MID["k"], seed=step)).cuda()
            y_ref = torch.empty((T, MID["H"]), dtype=torch.float32, device="cuda")
            y = torch.full((T, MID["H"]), float("nan"), dtype=torch.float32, device="cuda")
            with torch.cuda.stream(s):
                moe.moe_ffn_forward(h, x, idx, w, es.table, y_ref, T, s)
                tbl = moe.moe_expert_cache_fetch(c, idx_np, s)
                moe.moe_ffn_forward(h, x, idx, w, tbl, y, T, s)
            s.synchronize()
            assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32)), f"step {step}"
            model.request(idx_np.reshape(-1))
            assert [moe.moe_expert_cache_slot(c, e) for e in range(MID["E"])] == model.slot_of, f"step {step}"
        hits, misses, nbytes = moe.moe_expert_cache_stats(c)
        assert misses > slots and nbytes == misses * moe.moe_ffn_packed_expert_bytes(cfg)
        assert moe.moe_ffn_status(h) == moe.MOE_OK
    finally:
        moe.moe_expert_cache_destroy(c)
        moe.moe_ffn_destroy(h)


def test_prefetched_experts_are_hits_and_results_unchanged():
    T, slots = 1, 12
    cfg, h, es, host, c = _setup(T, slots)
    s = torch.cuda.Stream()
    try:
        routes = [synth.routing_uniform(T, MID["E"], MID["k"], seed=300 + i) for i in range(8)]
        for step, idx_np in enumerate(routes):
            x = torch.from_numpy(synth.activations_bf16(T, MID["H"], seed=step).view(np.int16)).cuda()
            idx = torch.from_numpy(idx_np).cuda()
            w = torch.from_numpy(synth.routing_weights(T, MID["k"], seed=step)).cuda()
            y_ref = torch.empty((T, MID["H"]), dtype=torch.float32, device="cuda")
            y = torch.empty_like(y_ref)
            with torch.cuda.stream(s):
                moe.moe_ffn_forward(h, x, idx, w, es.table, y_ref, T, s)
                h0, m0, _ = moe.moe_expert_cache_stats(c)
                tbl = moe.moe_expert_cache_fetch(c, idx_np, s)
                h1, m1, _ = moe.moe_expert_cache_stats(c)
                moe.moe_ffn_forward(h, x, idx, w, tbl, y, T, s)
                if step + 1 < len(routes):           # a perfect guess of the next step
                    moe.moe_expert_cache_prefetch(c, routes[step + 1], s)
            s.synchronize()
            assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32)), f"step {step}"
            if step > 0:
                assert (h1 - h0, m1 - m0) == (len(set(idx_np.reshape(-1).tolist())), 0)
    finally:
        moe.moe_expert_cache_destroy(c)
        moe.moe_ffn_destroy(h)


def test_request_larger_than_the_cache_is_rejected():
    cfg, h, es, host, c = _setup(1, 4)
    try:
        with pytest.raises(moe.MoeError) as e:
            moe.moe_expert_cache_fetch(c, np.arange(6, dtype=np.int32))
        assert e.value.code == moe.MOE_ERR_INVALID_ARG
        with pytest.raises(moe.MoeError):
            moe.moe_expert_cache_fetch(c, np.array([99], np.int32))
    finally:
        moe.moe_expert_cache_destroy(c)
        moe.moe_ffn_destroy(h)
