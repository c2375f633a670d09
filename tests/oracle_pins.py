"""Pins of the CPU oracle to facts outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix.  They are chosen
so that a plausible mistake anywhere in the oracle (a dropped term, a wrong
sign, a swapped operand, a byte-order slip, an unstable sort) fails at least
one of them; ``test_oracle_mutants.py`` plants such mistakes and checks that.

Independent references used here: numpy's own float16 decoding, dense numpy /
torch fp64 matmuls over all experts (brute force), scipy's expit, Python's
stable ``sorted``, closed forms and the pages' printed byte sizes.
"""
from __future__ import annotations

import os

import numpy as np
import torch
from scipy.special import expit

from routed_mixture_experts_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers ----
def np_dequant(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Independent Q8_0 decode with numpy's float16 (fp64 result)."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 34)
    d = b[:, :2].copy().view("<f2").astype(np.float64)[:, 0]
    q = b[:, 2:].copy().view(np.int8).astype(np.float64)
    return (q * d[:, None]).reshape(rows, K)


def np_dequant_q4(blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Independent Q4_0 decode with numpy (fp64): nibbles split by array ops."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 18)
    d = b[:, :2].copy().view("<f2").astype(np.float64)[:, 0]
    p = b[:, 2:].astype(np.int64)
    n = np.concatenate([p % 16, p // 16], axis=1)
    return ((n - 8).astype(np.float64) * d[:, None]).reshape(rows, K)


def tiny_layer(seed: int, T: int, dm: int, f: int, E: int, k: int, zipf: bool = False, wfmt: str = "q8"):
    wl = synth.custom(f"tiny{seed}", wid=1000 + seed, T=T, d_model=dm, d_ff=f, E=E, k=k, zipf=zipf, wfmt=wfmt)
    w = synth.make_layer(wl, 0, "cpu")
    x = synth.make_x(wl, "cpu").double().numpy()
    return wl, x, {kk: (None if v is None else v.numpy()) for kk, v in w.items()}


def dense_bruteforce(x, Wr, bias, gate, up, down, dm, f, E, k, residual=False, deq=np_dequant):
    """All E experts for every token, full softmax, mask to top-k, renormalise, sum."""
    Wg = np.stack([deq(gate[e], f, dm) for e in range(E)])
    Wu = np.stack([deq(up[e], f, dm) for e in range(E)])
    Wd = np.stack([deq(down[e], dm, f) for e in range(E)])
    logits = x @ Wr.astype(np.float64).T
    if bias is not None:
        logits = logits + bias.astype(np.float64)[None, :]
    T = x.shape[0]
    # full softmax over all experts
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    # top-k by (logit desc, id asc)
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -logits), axis=-1)
    sel = order[:, :k]
    mask = np.zeros((T, E))
    np.put_along_axis(mask, sel, 1.0, axis=1)
    wmix = p * mask
    wmix /= wmix.sum(axis=1, keepdims=True)
    G = np.einsum("efd,td->tef", Wg, x)
    U = np.einsum("efd,td->tef", Wu, x)
    H = G * expit(G) * U
    Y = np.einsum("edf,tef->ted", Wd, H)
    out = np.einsum("te,ted->td", wmix, Y)
    if residual:
        out = out + x
    return out, sel.astype(np.int32), np.take_along_axis(wmix, sel, axis=1), logits


def rel_l2_max(a, b):
    num = np.linalg.norm(a - b, axis=-1)
    den = np.maximum(np.linalg.norm(b, axis=-1), 1e-300)
    return float((num / den).max())


# ------------------------------------------------------------------- pins ----
def pin_half_decode(orc):
    """fp16 decode equals numpy's float16 for every non-NaN bit pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for bv in list(range(0, 65536, 97)) + [0, 1, 0x3ff, 0x400, 0x3c00, 0x7bff, 0x7c00, 0x8000, 0x8001, 0xfbff, 0xfc00]:
        r = ref[bv]
        got = orc.half_to_double(bv)
        if np.isnan(r):
            assert np.isnan(got), bv
        else:
            assert got == r, (hex(bv), got, r)


def pin_q8_roundtrip(orc):
    """Dequantise then re-encode reproduces the bytes (blocks containing |q|=127),
    and every dequantised value is q*d of numpy's own decode."""
    g = torch.Generator().manual_seed(7)
    w = torch.randn(24, 96, generator=g) * 0.02
    w[3, :32] = 0.0                       # an all-zero block
    w[5, 32:64] *= 1e-3                   # small scales
    blocks = synth.quantize_q8_0(w).numpy()
    deq = orc.dequant_q8(blocks, 24, 96)
    assert np.array_equal(deq, np_dequant(blocks, 24, 96))
    again = synth.quantize_q8_0(torch.from_numpy(deq.astype(np.float32))).numpy()
    assert np.array_equal(again, blocks)
    assert np.all(deq[3, :32] == 0.0)
    # every dequantised weight is exact in fp32 (8-bit q times 11-bit d)
    assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)


def pin_page_sizes(orc):
    """The pages' printed expert-cache sizes follow from 34-byte Q8_0 blocks of
    32 weights and three expert matrices of 2048 x 768.  The three matrices
    come to 5,013,504 B (already a whole number of 4 KiB pages); the printed
    raw-cache sizes and bytes-per-miss match that plus one more 4 KiB page per
    page-aligned blob (the pages do not say what that page holds), and do not
    match the bare 5,013,504 B (1536 slots would print 7.17 GiB)."""
    bb, be = orc.q8_block_bytes(), orc.q8_block_elems()
    expert = 3 * (2048 * 768 // be) * bb
    assert expert == 5_013_504
    assert expert % 4096 == 0
    padded = expert + 4096
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "expert_cache_sizes.txt")) if ln.strip()
            and not ln.startswith("#")]
    for kind, *vals in rows:
        if kind == "raw_cache_gib":
            slots, gib = int(vals[0]), float(vals[1])
            assert round(slots * padded / 2 ** 30, 2) == gib, (slots, gib)
        elif kind == "miss_bytes":
            misses, gb = int(vals[0]), float(vals[1])
            per = gb * 1e9 / misses
            assert abs(per - padded) / padded < 3e-3, (misses, per)
        elif kind == "model_gb":
            total = 48 * 128 * expert
            assert round(total / 1e9) == int(vals[0])


def pin_dense_bruteforce(orc):
    """Sparse oracle == dense all-experts brute force (tiny shapes, several seeds)."""
    for seed, (T, dm, f, E, k, zipf, res) in enumerate([
        (4, 256, 128, 16, 2, False, False),    # the tiny workload's geometry
        (5, 64, 32, 8, 3, True, False),
        (3, 96, 64, 6, 6, False, True),         # k == E: full softmax mixture
        (7, 32, 64, 12, 1, True, True),
        (1, 64, 32, 4, 2, False, False),
    ]):
        wl, x, w = tiny_layer(seed, T, dm, f, E, k, zipf)
        out, idx, wt, logits = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k,
                                             residual=res)
        ro, ridx, rw, rl = dense_bruteforce(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k,
                                            residual=res)
        assert np.allclose(logits, rl, rtol=0, atol=1e-12)
        assert np.array_equal(idx, ridx), (seed, idx, ridx)
        assert np.allclose(wt, rw, rtol=1e-12, atol=1e-15)
        assert rel_l2_max(out, ro) < 1e-12, (seed, rel_l2_max(out, ro))


def pin_k_equals_E_closed_form(orc):
    """k = E: output is the full-softmax mixture of all experts (closed form)."""
    T, dm, f, E = 3, 64, 32, 5
    wl, x, w = tiny_layer(11, T, dm, f, E, E)
    out, idx, wt, logits = orc.moe_layer(x, w["Wr"], None, w["gate"], w["up"], w["down"], dm, f, E, E)
    lg = x @ w["Wr"].astype(np.float64).T
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ys = np.stack([[orc.expert_swiglu(w["gate"][e], w["up"][e], w["down"][e], dm, f, x[t]) for e in range(E)]
                   for t in range(T)])
    ref = np.einsum("te,ted->td", p, ys)
    assert rel_l2_max(out, ref) < 1e-12
    # every expert appears once per token, in descending-probability order
    for t in range(T):
        assert sorted(idx[t].tolist()) == list(range(E))
        assert np.all(np.diff(wt[t]) <= 0)


def pin_zero_input_ties(orc):
    """x = 0, bias = 0: all logits tie at 0 -> experts 0..k-1, w = 1/k, output 0."""
    T, dm, f, E, k = 3, 64, 32, 8, 3
    wl, x, w = tiny_layer(3, T, dm, f, E, k)
    x0 = np.zeros_like(x)
    out, idx, wt, logits = orc.moe_layer(x0, w["Wr"], None, w["gate"], w["up"], w["down"], dm, f, E, k)
    assert np.all(idx == np.arange(k)[None, :])
    assert np.all(wt == 1.0 / k)
    assert np.all(out == 0.0)


def pin_weights_simplex(orc):
    """Selected weights are positive, sum to 1 (1e-12) and descend; logits descend."""
    T, dm, f, E, k = 16, 64, 32, 16, 4
    wl, x, w = tiny_layer(5, T, dm, f, E, k, zipf=True)
    out, idx, wt, logits = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k)
    assert np.all(wt > 0)
    assert np.allclose(wt.sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(wt, axis=1) <= 0)
    sel_l = np.take_along_axis(logits, idx, axis=1)
    assert np.all(np.diff(sel_l, axis=1) <= 0)
    # the selected logits are the k largest
    kth = np.sort(logits, axis=1)[:, ::-1][:, k - 1]
    assert np.all(sel_l[:, -1] == kth)


def pin_permutation_equivariance(orc):
    """Permuting tokens permutes idx, w and out identically."""
    T, dm, f, E, k = 9, 64, 32, 8, 2
    wl, x, w = tiny_layer(9, T, dm, f, E, k, zipf=True)
    perm = np.random.default_rng(3).permutation(T)
    a = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k, residual=True)
    b = orc.moe_layer(x[perm], w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k, residual=True)
    assert np.array_equal(a[1][perm], b[1])
    assert np.array_equal(a[2][perm], b[2])
    assert np.array_equal(a[0][perm], b[0])


def pin_single_expert_swiglu(orc):
    """E = 1, k = 1 reduces to one SwiGLU FFN: torch fp64 matmuls + torch silu."""
    T, dm, f, E, k = 4, 96, 64, 1, 1
    wl, x, w = tiny_layer(13, T, dm, f, E, k)
    out, idx, wt, _ = orc.moe_layer(x, w["Wr"], None, w["gate"], w["up"], w["down"], dm, f, E, k)
    Wg = torch.from_numpy(np_dequant(w["gate"][0], f, dm))
    Wu = torch.from_numpy(np_dequant(w["up"][0], f, dm))
    Wd = torch.from_numpy(np_dequant(w["down"][0], dm, f))
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ Wg.T) * (xt @ Wu.T)) @ Wd.T
    assert np.all(idx == 0) and np.all(wt == 1.0)
    assert rel_l2_max(out, ref.numpy()) < 1e-13


def pin_bucket_bruteforce(orc):
    """Bucketing == Python's stable sort of pairs by expert; sum of counts = T*k."""
    rng = np.random.default_rng(5)
    for T, k, E in [(1, 8, 128), (17, 3, 8), (64, 8, 128), (5, 2, 16), (0, 2, 4)]:
        idx = np.array([rng.permutation(E)[:k] for _ in range(T)], dtype=np.int32).reshape(T, k)
        if T >= 8:
            idx[:4, 0] = 1          # a skewed expert
        off, pt, ps, pos = orc.bucket(idx, E)
        pairs = [(int(idx[t, s]), t, s) for t in range(T) for s in range(k)]
        order = sorted(range(len(pairs)), key=lambda p: pairs[p][0])     # stable: ties keep (t, s) order
        assert [pairs[p][1] for p in order] == pt.tolist()
        assert [pairs[p][2] for p in order] == ps.tolist()
        cnt = np.bincount(idx.reshape(-1), minlength=E) if T else np.zeros(E, np.int64)
        assert off[0] == 0 and off[-1] == T * k
        assert np.array_equal(np.diff(off), cnt)
        for p_ in range(T * k):
            assert pt[pos[p_]] == p_ // k and ps[pos[p_]] == p_ % k


def pin_residual_stack(orc):
    """With residual, out = x + MoE(x) exactly (same MoE term as without)."""
    T, dm, f, E, k = 3, 64, 32, 8, 2
    wl, x, w = tiny_layer(17, T, dm, f, E, k)
    a = orc.moe_layer(x, w["Wr"], None, w["gate"], w["up"], w["down"], dm, f, E, k, residual=False)[0]
    b = orc.moe_layer(x, w["Wr"], None, w["gate"], w["up"], w["down"], dm, f, E, k, residual=True)[0]
    assert np.array_equal(b, x + a)
    assert np.abs(a).max() > 0


def pin_q4_block_layout(orc):
    """Q4_0 reading, on hand-built blocks: the fp16 scale leads (little
    endian), byte j's low nibble is element j and its high nibble element
    j + 16, values are (n - 8) * d, blocks run along K and rows follow rows."""
    a = bytes([0x00, 0x3C]) + bytes(j | ((15 - j) << 4) for j in range(16))    # d = 1.0
    b = bytes([0x00, 0xB8]) + bytes([0x8F] * 16)                              # d = -0.5
    blocks = np.frombuffer(a + b + b + a, dtype=np.uint8)                     # 2 rows x 64
    got = orc.dequant(blocks, 2, 64, 1)
    blk_a = [float(j - 8) for j in range(16)] + [float(7 - j) for j in range(16)]
    blk_b = [-3.5] * 16 + [0.0] * 16
    assert got.tolist() == [blk_a + blk_b, blk_b + blk_a], got
    assert np.array_equal(got, np_dequant_q4(blocks, 2, 64))


def pin_q4_roundtrip(orc):
    """Q4_0: re-encoding the decoded weights gives the same bytes, every value
    lies within half a step of the fp32 weight it encodes (plus the fp16
    rounding of the scale), and the decode is exact in fp32."""
    g = torch.Generator().manual_seed(11)
    w = torch.randn(12, 128, generator=g) * 0.02
    w[2, 32:64] = 0.0
    blocks = synth.quantize_q4_0(w).numpy()
    assert blocks.shape == (12, 4 * 18)
    deq = orc.dequant(blocks, 12, 128, 1)
    again = synth.quantize_q4_0(torch.from_numpy(deq.astype(np.float32))).numpy()
    assert np.array_equal(again, blocks)
    amax = w.reshape(12, 4, 32).abs().amax(-1).double().numpy()
    step = np.repeat(amax / 7.0, 32, axis=1)
    assert np.all(np.abs(deq - w.double().numpy()) <= 0.5 * step * (1 + 2e-3) + 1e-12)
    assert np.all(deq[2, 32:64] == 0.0)
    assert np.array_equal(deq.astype(np.float32).astype(np.float64), deq)


def pin_dense_bruteforce_q4(orc):
    """Sparse oracle with Q4_0 experts == dense brute force over all experts
    decoded by numpy; the Q8_0 layer of the same seed differs from it."""
    for seed, (T, dm, f, E, k, zipf) in enumerate([(4, 64, 32, 8, 2, False), (6, 96, 64, 12, 3, True)]):
        wl, x, w = tiny_layer(40 + seed, T, dm, f, E, k, zipf, wfmt="q4")
        assert w["gate"].shape == (E, f * dm // 32 * 18)
        out, idx, wt, _ = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k, fmt=1)
        ro, ridx, rw, _ = dense_bruteforce(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k,
                                           deq=np_dequant_q4)
        assert np.array_equal(idx, ridx)
        assert np.allclose(wt, rw, rtol=1e-12, atol=1e-15)
        assert rel_l2_max(out, ro) < 1e-12, rel_l2_max(out, ro)


def _dense_with(x_router, x_expert, w, dm, f, E, sel):
    """Dense reference for a given selection: weights = softmax of the
    router logits over the selection (in its order), experts fed x_expert."""
    Wg = np.stack([np_dequant(w["gate"][e], f, dm) for e in range(E)])
    Wu = np.stack([np_dequant(w["up"][e], f, dm) for e in range(E)])
    Wd = np.stack([np_dequant(w["down"][e], dm, f) for e in range(E)])
    lg = x_router @ w["Wr"].astype(np.float64).T
    if w["bias"] is not None:
        lg = lg + w["bias"].astype(np.float64)[None, :]
    ls = np.take_along_axis(lg, sel, axis=1)
    p = np.exp(ls - ls.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    G = np.einsum("efd,td->tef", Wg, x_expert)
    U = np.einsum("efd,td->tef", Wu, x_expert)
    Y = np.einsum("edf,tef->ted", Wd, G * expit(G) * U)
    return np.einsum("ts,tsd->td", p, np.take_along_axis(Y, sel[:, :, None], axis=1)), p


def pin_bf16_expert_inputs(orc):
    """expert_input_bf16: the router reads x, the experts read
    bf16(fp32(x)) rounded to nearest even at each step -- torch's own
    conversions, on values placed at exact bf16 ties and on one where
    rounding via fp32 differs from rounding the double directly."""
    T, dm, f, E, k = 3, 64, 32, 8, 2
    wl, x, w = tiny_layer(21, T, dm, f, E, k, zipf=True)
    x = x.copy()
    x[0, :4] = [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -3 * (1 + 3 * 2.0 ** -8)]  # ties
    x[1, 0] = 1 + 2.0 ** -8 + 2.0 ** -30          # via fp32: a tie -> 1.0; directly: -> 1 + 2**-7
    xb = torch.from_numpy(x).float().bfloat16().double().numpy()
    assert xb[0, 0] == 1.0 and xb[0, 1] == 1 + 2.0 ** -6 and xb[1, 0] == 1.0
    out, idx, wt, _ = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k,
                                    expert_input_bf16=True)
    ref, rw = _dense_with(x, xb, w, dm, f, E, idx.astype(np.int64))
    _, ridx, _, _ = dense_bruteforce(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k)
    assert np.array_equal(idx, ridx)             # routing reads the unrounded x
    assert np.allclose(wt, rw, rtol=1e-12, atol=1e-15)
    assert rel_l2_max(out, ref) < 1e-12
    plain = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k)[0]
    assert rel_l2_max(out, plain) > 1e-6         # the rounding is applied


def pin_forced_selection(orc):
    """forced_idx: the given experts, in the given order, weighted by the
    softmax of their logits (dense reference over an arbitrary selection)."""
    T, dm, f, E, k = 4, 64, 32, 8, 3
    wl, x, w = tiny_layer(23, T, dm, f, E, k)
    rng = np.random.default_rng(23)
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    out, idx, wt, _ = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, f, E, k,
                                    forced_idx=sel)
    ref, rw = _dense_with(x, x, w, dm, f, E, sel.astype(np.int64))
    assert np.array_equal(idx, sel)
    assert np.allclose(wt, rw, rtol=1e-12, atol=1e-15)
    assert rel_l2_max(out, ref) < 1e-12


def np_route(x, Wr, bias, k):
    """Independent router reference in numpy: fp64 logits, top-k by (logit
    descending, id ascending), full softmax over every expert masked to the
    selection and renormalised."""
    logits = x @ Wr.astype(np.float64).T
    if bias is not None:
        logits = logits + bias.astype(np.float64)[None, :]
    T, E = logits.shape
    ids = np.broadcast_to(np.arange(E), (T, E))
    sel = np.lexsort((ids, -logits), axis=-1)[:, :k]
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ps = np.take_along_axis(p, sel, axis=1)
    return sel.astype(np.int32), ps / ps.sum(axis=1, keepdims=True), logits


def pin_route_standalone(orc):
    """The routing-only entry (every token's logits, selection and weights,
    written at its own stride) equals the numpy router reference and the
    routing the whole-layer entry reports, on several token counts, with and
    without the Zipf bias, k = E, and a zero token whose logits all tie."""
    for seed, (T, dm, E, k, zipf) in enumerate([
        (4, 256, 16, 2, False),     # the tiny workload's geometry
        (9, 64, 32, 4, True),
        (5, 32, 6, 6, False),       # k == E
        (37, 128, 128, 8, True),    # full expert count and top-8, many tokens
        (3, 64, 8, 3, False),
    ]):
        wl, x, w = tiny_layer(40 + seed, T, dm, 32, E, k, zipf)
        if T >= 3 and not zipf:
            x[1] = 0.0  # all logits exactly 0: the lowest ids, equal weights
        idx, wt, logits = orc.route(x, w["Wr"], w["bias"], k)
        ridx, rw, rl = np_route(x, w["Wr"], w["bias"], k)
        assert np.allclose(logits, rl, rtol=0, atol=1e-12), seed
        assert np.array_equal(idx, ridx), (seed, idx, ridx)
        assert np.allclose(wt, rw, rtol=1e-12, atol=1e-15), seed
        _, lidx, lw, ll = orc.moe_layer(x, w["Wr"], w["bias"], w["gate"], w["up"], w["down"], dm, 32, E, k)
        assert np.array_equal(idx, lidx) and np.array_equal(wt, lw) and np.array_equal(logits, ll), seed
        if T >= 3 and not zipf:
            assert np.array_equal(idx[1], np.arange(k)) and np.all(wt[1] == 1.0 / k)


ALL_PINS = [
    pin_half_decode,
    pin_q8_roundtrip,
    pin_page_sizes,
    pin_dense_bruteforce,
    pin_k_equals_E_closed_form,
    pin_zero_input_ties,
    pin_weights_simplex,
    pin_permutation_equivariance,
    pin_single_expert_swiglu,
    pin_bucket_bruteforce,
    pin_residual_stack,
    pin_q4_block_layout,
    pin_q4_roundtrip,
    pin_dense_bruteforce_q4,
    pin_bf16_expert_inputs,
    pin_forced_selection,
    pin_route_standalone,
]
