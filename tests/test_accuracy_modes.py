"""Accuracy of the quantized activation modes against the bf16 mode, on the
oracle (CPU): two tokens of the full-size layer (384 experts, H = 4096,
I = 2880, top-6) with the synthetic weights and activations.  E4M3 with a
ue8m0 scale per 128 and E2M1 with one per 32 (MXFP4) replace x and h by their
quantized values; the table of measured errors is in the design notes."""
import numpy as np

import oracle
import synth

E, H, I, K = 384, 4096, 2880, 6


def _modes(T=2, seed=5):
    x = synth.activations_bf16(T, H, seed=seed)
    idx = synth.routing_uniform(T, E, K, seed=seed)
    w = synth.routing_weights(T, K, seed=seed)
    codes, scales = [None] * E, [None] * E
    for e in set(int(i) for i in idx.reshape(-1)):
        codes[e], scales[e] = synth.expert_canonical(H, I, e)
    return {m: oracle.moe_ffn(codes, scales, H, I, x, idx, w, act_mode=m, nthreads=8)
            for m in (oracle.ACT_BF16, oracle.ACT_E4M3_UE8M0_128, oracle.ACT_E2M1_UE8M0_32)}


def _rel_rms(y, ref):
    return np.sqrt(((y - ref) ** 2).sum(axis=1) / (ref ** 2).sum(axis=1))


def test_quantized_modes_error_against_bf16():
    ys = _modes()
    ref = ys[oracle.ACT_BF16]
    e4 = _rel_rms(ys[oracle.ACT_E4M3_UE8M0_128], ref)
    e2 = _rel_rms(ys[oracle.ACT_E2M1_UE8M0_32], ref)
    print(f"relative rms error vs bf16: e4m3 {e4.round(4)}, e2m1 {e2.round(4)}")
    # E4M3 keeps 3 mantissa bits, E2M1 one: per element about 2^-4 and 2^-2
    # relative rounding, which the sums over K average but do not remove
    assert np.all(e4 < 0.08) and np.all(e2 < 0.35)
    assert np.all(e2 > 2 * e4)
