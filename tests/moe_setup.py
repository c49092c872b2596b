"""Shared set-up for the GPU tests: synthetic expert sets, tolerance checks."""
import numpy as np
import torch

import fp4_block_scaled_gb300 as moe
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
