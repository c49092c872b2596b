"""Shared set-up for the GPU tests: synthetic expert sets, tolerance checks."""
import numpy as np
import torch

import fp4_block_scaled_gb300 as moe
import oracle
import synth
from fp4_block_scaled_gb300.experts import ExpertSet

# max|err| <= 2e-3 * rms(ref) and cosine >= 0.99999 (fp32 output vs fp64 oracle)
REL_MAX_ERR = 2e-3
MIN_COS = 0.99999


def fill_layer(handle, cfg, layer=0, seed=0, experts=None):
    """Device expert set of cfg.num_experts experts drawn from the synthetic
    recipe (codes uniform, scales in [119, 127]) and packed by the library."""
    H, I = cfg.hidden, cfg.inter
    es = ExpertSet(handle, cfg)
    nc, ns = synth.expert_sizes(H, I)
    tc = torch.empty(nc, dtype=torch.uint8, device="cuda")
    ts = torch.empty(ns, dtype=torch.uint8, device="cuda")
    for e in (range(cfg.num_experts) if experts is None else experts):
        synth.device_fill_expert(tc.data_ptr(), ts.data_ptr(), H, I, e, layer=layer, seed=seed)
        es.load(e, tc, ts)
    torch.cuda.synchronize()
    return es


def host_experts(H, I, ids, layer=0, seed=0, E=None):
    """Canonical blobs for the oracle: a list over E with None for unused ids."""
    E = E if E is not None else max(ids) + 1
    codes, scales = [None] * E, [None] * E
    for e in set(int(i) for i in ids):
        codes[e], scales[e] = synth.expert_canonical(H, I, e, layer=layer, seed=seed)
    return codes, scales


def errors(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.abs(y - ref).max()) if ref.size else 0.0
    cos = float((y * ref).sum() / (np.linalg.norm(y) * np.linalg.norm(ref))) if ref.size else 1.0
    return err / rms if rms > 0 else err, cos


def assert_close(y, ref, what=""):
    rel, cos = errors(y, ref)
    assert rel <= REL_MAX_ERR and cos >= MIN_COS, f"{what}: max|err|/rms={rel:.3e} cos={cos:.8f}"


def bf16_to_f64(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32).__lshift__(16).view(np.float32).astype(np.float64)


class Layer:
    """One layer's handle and device experts.  path: "slot" keeps every T on
    the slot-major path, "group" sends every T to the expert-major path,
    "auto" leaves the library default."""

    def __init__(self, E, H, I, k, max_tokens=8, out=moe.MOE_OUT_F32, seed=0, layer=0, act=moe.MOE_ACT_BF16,
                 path="slot"):
        self.E, self.H, self.I, self.k = E, H, I, k
        self.act = act
        gmin = {"slot": max_tokens + 1, "group": 1, "auto": 0}[path]
        self.cfg = moe.config(E, H, I, k, max_tokens, out_dtype=out, act_mode=act, gemm_min_tokens=gmin)
        self.h = moe.moe_ffn_create(self.cfg, 0)
        self.es = fill_layer(self.h, self.cfg, layer=layer, seed=seed)
        self.seed, self.layer = seed, layer
        self.out = out

    def run(self, x_bits, idx, w):
        T = x_bits.shape[0]
        x = torch.from_numpy(x_bits.view(np.int16)).cuda()
        it = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
        wt = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
        dt = torch.float32 if self.out == moe.MOE_OUT_F32 else torch.bfloat16
        y = torch.empty((T, self.H), dtype=dt, device="cuda")
        moe.moe_ffn_forward(self.h, x, it, wt, self.es.table, y, T)
        torch.cuda.synchronize()
        return y

    def oracle(self, x_bits, idx, w):
        codes, scales = host_experts(self.H, self.I, idx.reshape(-1), layer=self.layer,
                                     seed=self.seed, E=self.E)
        act = oracle.ACT_E4M3_UE8M0_128 if self.act == moe.MOE_ACT_E4M3_UE8M0_128 else oracle.ACT_BF16
        return oracle.moe_ffn(codes, scales, self.H, self.I, x_bits, idx, w, act_mode=act, nthreads=8)

    def close(self):
        moe.moe_ffn_destroy(self.h)


def inputs(T, E, H, k, seed=0):
    return (synth.activations_bf16(T, H, seed=seed), synth.routing_uniform(T, E, k, seed=seed),
            synth.routing_weights(T, k, seed=seed))
