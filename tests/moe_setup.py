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
                 path="slot", mma=None):
        self.E, self.H, self.I, self.k = E, H, I, k
        self.act = act
        gmin = {"slot": max_tokens + 1, "group": 1, "auto": 0}[path]
        self.cfg = moe.config(E, H, I, k, max_tokens, out_dtype=out, act_mode=act, gemm_min_tokens=gmin)
        self.h = moe.moe_ffn_create(self.cfg, 0)
        if mma is not None:
            moe.moe_ffn_set_mma_kind(self.h, mma)
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
        act = {moe.MOE_ACT_E4M3_UE8M0_128: oracle.ACT_E4M3_UE8M0_128,
               moe.MOE_ACT_E2M1_UE8M0_32: oracle.ACT_E2M1_UE8M0_32}.get(self.act, oracle.ACT_BF16)
        return oracle.moe_ffn(codes, scales, self.H, self.I, x_bits, idx, w, act_mode=act, nthreads=8)

    def close(self):
        moe.moe_ffn_destroy(self.h)


def inputs(T, E, H, k, seed=0):
    return (synth.activations_bf16(T, H, seed=seed), synth.routing_uniform(T, E, k, seed=seed),
            synth.routing_weights(T, k, seed=seed))


# ----------------------------------------------------- E2M1 activation mode

E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def e2m1_flip_bound(H, I, E, x_bits, idx, w, layer=0, seed=0, delta=1e-4):
    """How far y[t] may move (per output row) because h, computed in fp32 on
    the GPU and in fp64 by the oracle, takes the other E2M1 code: every element
    of h within delta (in units of its block scale) of a rounding midpoint, and
    every element of a block whose maximum lies within a relative delta of a
    scale boundary, may move by up to the largest E2M1 step (2 units, at the
    larger candidate scale).  The fp32 h differs from the fp64 h by far less
    than delta.  Returns (bound [T][H], number of such elements)."""
    e2m1 = np.array([oracle.e2m1_value(c) for c in range(16)])
    T, k = idx.shape
    codes, scales = host_experts(H, I, idx.reshape(-1), layer=layer, seed=seed, E=E)
    gc, gs = I * H // 2, I * H // 32
    bound = np.zeros((T, H))
    n_amb = 0
    for t in range(T):
        xf = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xc, xs = oracle.act_quant_e2m1(xf, 32)
        xq = e2m1[xc] * np.ldexp(1.0, np.repeat(xs.astype(np.int64), 32)[:H] - 127)
        for j in range(k):
            e = int(idx[t, j])
            if e < 0 or e >= E:
                continue
            c, s = codes[e], scales[e]
            g = oracle.matvec(c[:gc], s[:gs], I, H, xq)
            u = oracle.matvec(c[gc:2 * gc], s[gs:2 * gs], I, H, xq)
            h = g / (1.0 + np.exp(-g)) * u
            dc = np.asarray(c[2 * gc:], np.uint8).reshape(H, I // 2)
            ds = np.asarray(s[2 * gs:], np.uint8).reshape(H, I // 32)
            for b0 in range(0, I, 32):
                blk = h[b0:b0 + 32]
                amax = float(np.abs(blk).max())
                kk = oracle.ue8m0_for_amax_e2m1(amax) - 127
                r = np.abs(blk) / 2.0 ** kk
                near = np.abs(r[:, None] - E2M1_MIDPOINTS[None, :]).min(axis=1) < delta
                edge = amax > 0 and (abs(amax / (6.0 * 2.0 ** (kk - 1)) - 1) < delta
                                     or abs(amax / (6.0 * 2.0 ** kk) - 1) < delta)
                amb = np.arange(32) if edge else np.nonzero(near)[0]
                for i in amb:
                    col_i = b0 + int(i)
                    byte = dc[:, col_i // 2]
                    nib = (byte >> 4) if col_i & 1 else (byte & 15)
                    col = e2m1[nib] * np.ldexp(1.0, ds[:, col_i // 32].astype(np.int64) - 127)
                    bound[t] += abs(float(w[t, j])) * np.abs(col) * 2.0 * 2.0 ** (kk + 1)
                    n_amb += 1
    return bound, n_amb


def e4m3_flip_candidates(H, I, E, x_bits, idx, layer=0, seed=0, delta=1e-4):
    """How many elements of h could round to the other E4M3 neighbour on the
    GPU (fp32 h) than in the oracle (fp64 h): elements of the oracle's h whose
    scaled value lies within delta (relative to the local grid step) of a
    midpoint between adjacent E4M3 values, plus whole 128-blocks (64 for the
    last) whose maximum lies within a relative delta of a scale boundary
    448 * 2^k.  Each such flip moves y by about 1e-3 rms.  Returns (count,
    elements of h examined)."""
    pos = np.unique([oracle.e4m3_value(c) for c in range(127)])
    mids = (pos[1:] + pos[:-1]) / 2.0
    steps = pos[1:] - pos[:-1]
    T, k = idx.shape
    codes, scales = host_experts(H, I, idx.reshape(-1), layer=layer, seed=seed, E=E)
    gc, gs = I * H // 2, I * H // 32
    n, total = 0, 0
    for t in range(T):
        xf = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xc, xsc = oracle.act_quant_e4m3(xf, 128)
        xq = np.array([oracle.e4m3_value(int(c)) for c in xc]) * np.ldexp(
            1.0, np.repeat(xsc.astype(np.int64), 128)[:H] - 127)
        for j in range(k):
            e = int(idx[t, j])
            c, sc = codes[e], scales[e]
            g = oracle.matvec(c[:gc], sc[:gs], I, H, xq)
            u = oracle.matvec(c[gc:2 * gc], sc[gs:2 * gs], I, H, xq)
            hv = g / (1.0 + np.exp(-g)) * u
            for b0 in range(0, I, 128):
                blk = hv[b0:b0 + 128]
                amax = float(np.abs(blk).max())
                kk = oracle.ue8m0_for_amax(amax) - 127
                total += blk.size
                if amax > 0 and (abs(amax / (448.0 * 2.0 ** kk) - 1) < delta
                                 or abs(amax / (448.0 * 2.0 ** (kk - 1)) - 1) < delta):
                    n += blk.size
                    continue
                r = np.abs(blk) / 2.0 ** kk
                pos_i = np.clip(np.searchsorted(mids, r), 1, len(mids) - 1)
                d = np.minimum(np.abs(r - mids[pos_i - 1]) / steps[pos_i - 1],
                               np.abs(r - mids[pos_i]) / steps[pos_i])
                n += int((d < delta).sum())
    return n, total


def e4m3_flip_bound(H, I, E, x_bits, idx, w, layer=0, seed=0, delta=1e-4):
    """How far y[t] may move (per output row) because an element of h,
    computed in fp32 on the GPU and in fp64 by the oracle, takes the other E4M3
    neighbour: each element of the oracle's h within delta (relative to the
    local grid step) of a midpoint moves by that step; every element of a
    128-block (64 for the last) whose maximum lies within a relative delta of a
    scale boundary 448 * 2^k by up to the largest E4M3 step at the larger
    candidate scale.  Each moves y by w times its down column.  Returns
    (bound [T][H], number of such elements)."""
    e2m1 = np.array([oracle.e2m1_value(c) for c in range(16)])
    pos = np.unique([oracle.e4m3_value(c) for c in range(127)])
    mids = (pos[1:] + pos[:-1]) / 2.0
    steps = pos[1:] - pos[:-1]
    T, k = idx.shape
    codes, scales = host_experts(H, I, idx.reshape(-1), layer=layer, seed=seed, E=E)
    gc, gs = I * H // 2, I * H // 32
    bound = np.zeros((T, H))
    n_amb = 0
    for t in range(T):
        xf = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xc, xsc = oracle.act_quant_e4m3(xf, 128)
        xq = np.array([oracle.e4m3_value(int(c)) for c in xc]) * np.ldexp(
            1.0, np.repeat(xsc.astype(np.int64), 128)[:H] - 127)
        for j in range(k):
            e = int(idx[t, j])
            if e < 0 or e >= E:
                continue
            c, sc = codes[e], scales[e]
            g = oracle.matvec(c[:gc], sc[:gs], I, H, xq)
            u = oracle.matvec(c[gc:2 * gc], sc[gs:2 * gs], I, H, xq)
            hv = g / (1.0 + np.exp(-g)) * u
            dc = np.asarray(c[2 * gc:], np.uint8).reshape(H, I // 2)
            ds = np.asarray(sc[2 * gs:], np.uint8).reshape(H, I // 32)
            for b0 in range(0, I, 128):
                blk = hv[b0:b0 + 128]
                amax = float(np.abs(blk).max())
                kk = oracle.ue8m0_for_amax(amax) - 127
                if amax > 0 and (abs(amax / (448.0 * 2.0 ** kk) - 1) < delta
                                 or abs(amax / (448.0 * 2.0 ** (kk - 1)) - 1) < delta):
                    amb = [(i, float(steps.max()) * 2.0 ** (kk + 1)) for i in range(blk.size)]
                else:
                    r = np.abs(blk) / 2.0 ** kk
                    pi = np.clip(np.searchsorted(mids, r), 1, len(mids) - 1)
                    d_lo = np.abs(r - mids[pi - 1]) / steps[pi - 1]
                    d_hi = np.abs(r - mids[pi]) / steps[pi]
                    st = np.where(d_lo < d_hi, steps[pi - 1], steps[pi])
                    amb = [(int(i), float(st[i]) * 2.0 ** kk) for i in np.nonzero(np.minimum(d_lo, d_hi) < delta)[0]]
                for i, step in amb:
                    ci = b0 + i
                    byte = dc[:, ci // 2]
                    nib = (byte >> 4) if ci & 1 else (byte & 15)
                    col = e2m1[nib] * np.ldexp(1.0, ds[:, ci // 32].astype(np.int64) - 127)
                    bound[t] += abs(float(w[t, j])) * np.abs(col) * step
                    n_amb += 1
    return bound, n_amb


def assert_close_e4m3(y, ref, layer_args, what=""):
    """The float tolerance, or -- when it fails -- the tolerance once each row's
    possible E4M3 flips of h are allowed for (e4m3_flip_bound over
    layer_args = (H, I, E, x_bits, idx, w[, layer, seed])); cosine >= 0.99999."""
    rel, cos = errors(y, ref)
    if rel <= REL_MAX_ERR and cos >= MIN_COS:
        return
    bound, n = e4m3_flip_bound(*layer_args)
    y = np.asarray(y, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = float((np.abs(y - ref) - bound).max()) / rms
    assert excess <= REL_MAX_ERR and cos >= MIN_COS, \
        f"{what}: max|err|/rms={rel:.3e}, beyond the bound of {n} possible h flips {excess:.3e}, cos={cos:.8f}"


def check_f8_h_and_down(handle, H, I, E, x_bits, idx, w, y, tokens=None, layer=0, seed=0, what=""):
    """For a call on the kind::mxf8f6f4 expert-major path: (1) the GPU's fp32
    h of each slot of the given tokens against the oracle's fp64 h (max |diff|
    <= 1e-5 max|h| per slot); (2) y against the oracle's down projection and
    combine of the GPU's own E4M3-quantized h (the oracle's quantizer on the
    GPU's h; max|err| <= 1e-5 rms, so every difference from the plain oracle
    is an E4M3 rounding decision of h).  Returns (flips, elements): the
    elements of h whose E4M3 code or block scale differs between the GPU's h
    and the oracle's."""
    import torch

    T, k = idx.shape
    tokens = range(T) if tokens is None else list(tokens)
    n = T * k
    hd, pd = moe.moe_ffn_test_copy_h(handle, n, I)
    torch.cuda.synchronize()
    hg, perm = hd.cpu().numpy().astype(np.float64), pd.cpu().numpy()
    pos_of = {int(perm[P]): P for P in range(n) if perm[P] >= 0}
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    codes, scales = host_experts(H, I, idx.reshape(-1), layer=layer, seed=seed, E=E)
    gc, gs = I * H // 2, I * H // 32

    def deq(c, sc, n_):
        return e4[c] * np.ldexp(1.0, np.repeat(sc.astype(np.int64), 128)[:n_] - 127)

    flips = total = 0
    for t in tokens:
        xf = (x_bits[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xq = deq(*oracle.act_quant_e4m3(xf, 128), H)
        y2 = np.zeros(H)
        for j in range(k):
            e = int(idx[t, j])
            P = pos_of[t * k + j]
            c, sc = codes[e], scales[e]
            g = oracle.matvec(c[:gc], sc[:gs], I, H, xq)
            u = oracle.matvec(c[gc:2 * gc], sc[gs:2 * gs], I, H, xq)
            h = g / (1.0 + np.exp(-g)) * u
            d = float(np.abs(hg[P] - h).max())
            assert d <= 1e-5 * float(np.abs(h).max()), f"{what}: h of token {t} slot {j}: max|diff| {d:.3e}"
            cg, sg = oracle.act_quant_e4m3(hg[P], 128)
            co, so = oracle.act_quant_e4m3(h, 128)
            flips += int(((cg != co) | (np.repeat(sg, 128)[:I] != np.repeat(so, 128)[:I])).sum())
            total += I
            y2 += float(w[t, j]) * oracle.matvec(c[2 * gc:], sc[2 * gs:], H, I, deq(cg, sg, I))
        rel, _ = errors(np.asarray(y[t:t + 1], np.float64), y2[None, :])
        assert rel <= 1e-5, f"{what}: token {t}: y vs down(GPU h): max|err|/rms={rel:.3e}"
    return flips, total


def assert_close_e2m1(y, ref, bound, what=""):
    """Within the usual tolerance once each row's possible code flips are
    allowed for; cosine >= 0.9999."""
    y = np.asarray(y, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    excess = np.abs(y - ref) - bound
    rel = float(excess.max()) / rms
    _, cos = errors(y, ref)
    assert rel <= REL_MAX_ERR and cos >= 0.9999, f"{what}: max(|err| - flip bound)/rms={rel:.3e} cos={cos:.8f}"
