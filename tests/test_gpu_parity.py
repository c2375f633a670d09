"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Routing indices and bucket results bit-exact (near-tie tokens counted and
checked as valid selections), layer outputs within max relative L2 1e-5 on
the fp32-activation path.
"""
import zlib

import numpy as np
import pytest
import torch

from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import (TOL_F32, Case, check_bucket, check_routing, make_case, oracle_layer, rel_l2_max)

pytestmark = pytest.mark.gpu

# odd shapes: several row tiles plus ragged tails, small experts sets
SHAPES = [
    # name, T, d, f, E, k, zipf
    ("tiny", 4, 256, 128, 16, 2, False),
    ("odd_t3", 3, 256, 128, 16, 2, True),
    ("t63", 63, 512, 256, 32, 4, True),
    ("t65", 65, 512, 256, 32, 4, False),
    ("e8k8", 5, 256, 96, 8, 8, False),       # k == E, d_ff not a multiple of 64
    ("t2_k1", 2, 1024, 384, 64, 1, True),
    ("d4096", 9, 4096, 64, 24, 3, False),
    ("s256_t7", 7, 256, 256, 16, 4, True),    # streaming path, all tokens staged at once
    ("t12", 12, 1024, 512, 64, 6, True),      # lane-per-row path, per-chunk activations
    ("t2", 2, 2048, 768, 128, 8, False),      # full geometry, two tokens
    ("rows_t6", 6, 1024, 512, 32, 3, False),  # lane-per-row path, all tokens staged at once
    ("rows_t21", 21, 512, 768, 16, 4, True),  # lane-per-row path, ragged 8-pair chunks, 3 K stages per down warp
]


def _wl(name, T, d, f, E, k, zipf):
    return synth.custom(name, wid=zlib.crc32(name.encode()) % 10000 + 200,
                        T=T, d_model=d, d_ff=f, E=E, k=k, zipf=zipf)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def test_pack_q8_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(1)
    w = torch.randn(37, 96, generator=g, device="cuda") * 0.02
    blocks = synth.quantize_q8_0(w)
    qs, d = binding.pack_q8(blocks, 37, 96)
    b = blocks.cpu().numpy().reshape(37, 3, 34)
    # device layout: each int8 value q as the byte q + 128 (sign bit flipped)
    assert np.array_equal(qs.cpu().numpy().reshape(37, 3, 32).view(np.uint8), b[:, :, 2:] ^ 0x80)
    assert np.array_equal(d.cpu().numpy().view(np.uint8).reshape(37, 3, 2), b[:, :, :2])


def _route_and_check(case: Case):
    idx, wts = binding.route(case.x, case.layer)
    torch.cuda.synchronize()
    oi, ow, ol = __import__("oracle").get().route(case.host["x"], case.host["Wr"], case.host["bias"], case.wl.k)
    near = check_routing(idx.cpu().numpy(), wts.cpu().numpy(), oi, ow, ol, case.wl.k)
    return idx, wts, near


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
def test_route_bucket_small(shape):
    case = make_case(_wl(*shape))
    idx, wts, near = _route_and_check(case)
    off, pt, ps, pos = binding.bucket(idx, case.wl.E)
    torch.cuda.synchronize()
    check_bucket(idx.cpu().numpy(), case.wl.E, off.cpu().numpy(), pt.cpu().numpy(), ps.cpu().numpy(),
                 pos.cpu().numpy())


@pytest.mark.parametrize("name", ["decode_t1", "decode_t64_zipf", "prefill_t1024"])
def test_route_bucket_full(name):
    case = make_case(synth.WORKLOADS[name])
    idx, wts, near = _route_and_check(case)
    print(f"{name}: near-tie tokens {near} of {case.wl.T}")
    off, pt, ps, pos = binding.bucket(idx, case.wl.E)
    torch.cuda.synchronize()
    check_bucket(idx.cpu().numpy(), case.wl.E, off.cpu().numpy(), pt.cpu().numpy(), ps.cpu().numpy(),
                 pos.cpu().numpy())


def test_bucket_skew_and_empty():
    """All tokens on one expert, many empty experts, large T (several chunks)."""
    T, k, E = 2500, 8, 128
    rng = np.random.default_rng(0)
    idx = np.stack([np.concatenate([[7], rng.choice(np.setdiff1d(np.arange(40), [7]), k - 1, replace=False)])
                    for _ in range(T)]).astype(np.int32)
    di = torch.from_numpy(idx).cuda()
    off, pt, ps, pos = binding.bucket(di, E)
    torch.cuda.synchronize()
    check_bucket(idx, E, off.cpu().numpy(), pt.cpu().numpy(), ps.cpu().numpy(), pos.cpu().numpy())


def test_bucket_bad_ids_many_tiles():
    """Thousands of pairs (the many-CTA bucketing), odd k, invalid and repeated
    ids: a pair is dropped (pos -1) when its id is out of range or repeats an
    earlier slot of the same token; the rest are grouped by expert, stable in
    (token, slot) order."""
    T, k, E = 2100, 3, 64
    rng = np.random.default_rng(5)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    bad = rng.random((T, k))
    idx[bad < 0.01] = -1
    idx[(bad >= 0.01) & (bad < 0.02)] = E + 7
    idx[::97, 2] = idx[::97, 0]                 # repeats within a token
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    off, pt, ps, pos = binding.bucket(torch.from_numpy(idx).cuda(), E, status=status)
    torch.cuda.synchronize()
    assert status.item() & binding.MOE_STATUS_BAD_INDEX
    keep = np.zeros((T, k), dtype=bool)
    for t in range(T):
        seen = set()
        for s in range(k):
            e = int(idx[t, s])
            if 0 <= e < E and e not in seen:
                keep[t, s] = True
            if 0 <= e < E:
                seen.add(e)
    pairs = [(int(idx[t, s]), t, s) for t in range(T) for s in range(k) if keep[t, s]]
    pairs.sort()
    exp_off = np.searchsorted(np.array([p[0] for p in pairs]), np.arange(E + 1), side="left")
    exp_pos = -np.ones(T * k, dtype=np.int64)
    for r, (_, t, s) in enumerate(pairs):
        exp_pos[t * k + s] = r
    assert np.array_equal(off.cpu().numpy(), exp_off)
    assert np.array_equal(pos.cpu().numpy(), exp_pos)
    n = len(pairs)
    assert np.array_equal(pt.cpu().numpy()[:n], [p[1] for p in pairs])
    assert np.array_equal(ps.cpu().numpy()[:n], [p[2] for p in pairs])


@pytest.mark.parametrize("T,k,E", [(300, 8, 128), (100, 8, 128), (200, 12, 64), (50, 12, 64)])
def test_bucket_repeats_both_id_checks(T, k, E):
    """Invalid and repeated ids at k = 8 (ids in registers, 16-byte loads) and
    k = 12 (a bitmap over the experts), through the many-CTA kernel (T k >=
    2048 pairs) and the single-CTA one: the first occurrence of a valid id is
    kept, later repeats and out-of-range ids dropped (pos -1) and flagged."""
    rng = np.random.default_rng(T * 131 + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    r = rng.random((T, k))
    idx[r < 0.02] = -3
    idx[(r >= 0.02) & (r < 0.04)] = E
    for t in range(0, T, 7):                        # a repeat in every seventh token
        s_from, s_to = sorted(rng.choice(k, 2, replace=False))
        idx[t, s_to] = idx[t, s_from]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    off, pt, ps, pos = binding.bucket(torch.from_numpy(idx).cuda(), E, status=status)
    torch.cuda.synchronize()
    assert status.item() & binding.MOE_STATUS_BAD_INDEX
    pairs = []
    for t in range(T):
        seen = set()
        for s in range(k):
            e = int(idx[t, s])
            if 0 <= e < E and e not in seen:
                pairs.append((e, t, s))
            if 0 <= e < E:
                seen.add(e)
    pairs.sort()
    exp_pos = -np.ones(T * k, dtype=np.int64)
    for rank, (_, t, s) in enumerate(pairs):
        exp_pos[t * k + s] = rank
    assert np.array_equal(off.cpu().numpy(),
                          np.searchsorted(np.array([q[0] for q in pairs]), np.arange(E + 1), side="left"))
    assert np.array_equal(pos.cpu().numpy(), exp_pos)
    n = len(pairs)
    assert np.array_equal(pt.cpu().numpy()[:n], [q[1] for q in pairs])
    assert np.array_equal(ps.cpu().numpy()[:n], [q[2] for q in pairs])


def test_bucket_bad_ids_flag_status():
    idx = torch.tensor([[0, 1], [5, 5], [2, 99], [-1, 3]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    off, pt, ps, pos = binding.bucket(idx, 8, status=status)
    torch.cuda.synchronize()
    assert status.item() & binding.MOE_STATUS_BAD_INDEX
    off = off.cpu().numpy()
    assert off[0] == 0 and off[-1] == 5 and np.all(np.diff(off) >= 0)   # (0,0) (0,1) (1,0) (2,0) (3,1)
    p = pos.cpu().numpy()
    assert p[3] == -1 and p[5] == -1 and p[6] == -1


def _layer_check(case: Case, residual=False, flags=0, tokens=None):
    idx_out = torch.empty(case.wl.T, case.wl.k, dtype=torch.int32, device="cuda")
    wts_out = torch.empty(case.wl.T, case.wl.k, dtype=torch.float32, device="cuda")
    out = binding.layer_forward(case.x, case.layer, binding.MOE_ACT_F32, flags=flags, residual=residual,
                                idx_out=idx_out, wts_out=wts_out)
    torch.cuda.synchronize()
    gidx = idx_out.cpu().numpy()
    o_out, o_idx, o_w, o_l = oracle_layer(case, tokens=tokens, forced_idx=None if tokens is None else gidx[tokens])
    sel = slice(None) if tokens is None else tokens
    if tokens is None:
        near = check_routing(gidx, wts_out.cpu().numpy(), o_idx, o_w, o_l, case.wl.k)
        if near:
            o_out = oracle_layer(case, forced_idx=gidx)[0]
    g = out.cpu().numpy().astype(np.float64)[sel]
    xs = case.host["x"][sel]
    moe_gpu = g - xs if residual else g
    err = rel_l2_max(moe_gpu, o_out)
    assert err < TOL_F32, f"max rel L2 {err:.3e}"
    return out, err


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
@pytest.mark.parametrize("flags", [0, binding.MOE_FLAG_DETERMINISTIC], ids=["atomic", "det"])
def test_layer_f32_small(shape, flags):
    _layer_check(make_case(_wl(*shape)), flags=flags)


@pytest.mark.parametrize("name", ["tiny", "decode_t1", "decode_t64_zipf"])
def test_layer_f32_workloads(name):
    _, err = _layer_check(make_case(synth.WORKLOADS[name]))
    print(f"{name}: max rel L2 {err:.3e}")


def test_layer_f32_residual():
    _layer_check(make_case(_wl("t63", 63, 512, 256, 32, 4, True)), residual=True)
    _layer_check(make_case(_wl("t63", 63, 512, 256, 32, 4, True)), residual=True,
                 flags=binding.MOE_FLAG_DETERMINISTIC)


def test_layer_f32_full_t1024_sampled():
    """Full qwen3_moe geometry at T=1024 on the fp32 path: routing for all
    tokens, outputs on 48 sampled tokens recomputed by the oracle."""
    case = make_case(synth.WORKLOADS["prefill_t1024"])
    tokens = np.sort(np.random.default_rng(1).choice(case.wl.T, 48, replace=False))
    tokens[0], tokens[-1] = 0, case.wl.T - 1
    _layer_check(case, tokens=tokens)


def test_all_tokens_one_expert():
    """A dominant router bias sends every token to expert 3 first."""
    wl = _wl("hot", 40, 256, 128, 16, 4, False)
    case = make_case(wl)
    bias = torch.zeros(wl.E, device="cuda")
    bias[3] = 100.0
    case.layer = binding.Layer(wl.E, wl.k, wl.d_model, wl.d_ff, case.layer.gate, case.layer.up, case.layer.down,
                               case.layer.router_w, bias)
    case.host["bias"] = bias.cpu().numpy()
    out, _ = _layer_check(case)
    idx, _ = binding.route(case.x, case.layer)
    assert bool((idx[:, 0] == 3).all())


def test_zero_input_ties():
    """x = 0, no bias: all logits tie -> experts 0..k-1, w = 1/k, output 0."""
    wl = _wl("zero", 5, 256, 128, 16, 4, False)
    case = make_case(wl)
    x0 = torch.zeros_like(case.x)
    idx, wts = binding.route(x0, case.layer)
    out = binding.layer_forward(x0, case.layer)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), np.tile(np.arange(4, dtype=np.int32), (5, 1)))
    assert np.all(wts.cpu().numpy() == 0.25)
    assert np.all(out.cpu().numpy() == 0.0)


def test_t0_is_noop():
    wl = _wl("tiny", 4, 256, 128, 16, 2, False)
    case = make_case(wl)
    out = torch.full((0, 256), 7.0, device="cuda")
    binding.layer_forward(case.x[:0], case.layer, out=out)
    idx, wts = binding.route(case.x[:0], case.layer)
    assert idx.numel() == 0


def test_determinism():
    case = make_case(synth.WORKLOADS["decode_t64_zipf"])
    ref = None
    for _ in range(3):
        idx, wts = binding.route(case.x, case.layer)
        off, pt, ps, pos = binding.bucket(idx, case.wl.E)
        out = binding.layer_forward(case.x, case.layer, flags=binding.MOE_FLAG_DETERMINISTIC)
        torch.cuda.synchronize()
        cur = [t.cpu().numpy().copy() for t in (idx, wts, off, pt, ps, pos, out)]
        if ref is None:
            ref = cur
        else:
            for a, b in zip(ref, cur):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_graph_replay_changed_inputs():
    """Capture one layer call in a CUDA graph, change x in place, replay."""
    case = make_case(synth.WORKLOADS["decode_t1"])
    x = case.x.clone()
    out = torch.empty_like(x)
    ws = binding.workspace(1, case.layer, flags=binding.MOE_FLAG_DETERMINISTIC)
    binding.layer_forward(x, case.layer, out=out, ws=ws, flags=binding.MOE_FLAG_DETERMINISTIC)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            binding.layer_forward(x, case.layer, out=out, ws=ws, flags=binding.MOE_FLAG_DETERMINISTIC)
    for step in range(3):
        x.copy_(synth.make_x(case.wl, "cuda", step=10 + step))
        g.replay()
        torch.cuda.synchronize()
        direct = binding.layer_forward(x, case.layer, flags=binding.MOE_FLAG_DETERMINISTIC)
        torch.cuda.synchronize()
        assert torch.equal(out, direct)


def test_combine_entry_point():
    """moe_expert_ffn_q8 (ypairs) + moe_combine == the fused layer output."""
    case = make_case(_wl("t65", 65, 512, 256, 32, 4, False))
    idx, wts = binding.route(case.x, case.layer)
    off, pt, ps, pos = binding.bucket(idx, case.wl.E)
    yp = binding.expert_ffn_q8(case.x, case.layer, off, pt, ps, wts, fuse_combine=False)
    out = binding.combine(yp, wts, pos, case.wl.T, case.wl.k, case.wl.d_model, residual=case.x)
    fused = binding.expert_ffn_q8(case.x, case.layer, off, pt, ps, wts, fuse_combine=True, residual=True)
    torch.cuda.synchronize()
    o_out = oracle_layer(case, forced_idx=idx.cpu().numpy(), residual=True)[0]
    assert rel_l2_max(out.cpu().double().numpy() - case.host["x"], o_out - case.host["x"]) < TOL_F32
    assert rel_l2_max(fused.cpu().double().numpy() - case.host["x"], o_out - case.host["x"]) < TOL_F32


@pytest.mark.parametrize("act", [binding.MOE_ACT_F32, binding.MOE_ACT_BF16], ids=["f32", "bf16"])
def test_max_batch_t65536_sampled(act):
    """The largest batch the ABI takes (T = 65536, 524,288 pairs) at the full
    qwen3_moe geometry with the Zipf bias: routing of every token and the
    bucketing bit-exact (near-ties counted), outputs of sampled tokens within
    the path's tolerance of the oracle run with the GPU's selection."""
    bf16 = act == binding.MOE_ACT_BF16
    wl = synth.custom("max_t65536", wid=901, T=65536, d_model=2048, d_ff=768, E=128, k=8, zipf=True,
                      act="bf16" if bf16 else "f32")
    case = make_case(wl)
    idx, wts, near = _route_and_check(case)
    print(f"T=65536: near-tie tokens {near}")
    off, pt, ps, pos = binding.bucket(idx, wl.E)
    torch.cuda.synchronize()
    check_bucket(idx.cpu().numpy(), wl.E, off.cpu().numpy(), pt.cpu().numpy(), ps.cpu().numpy(), pos.cpu().numpy())
    idx_out = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.layer_forward(case.x, case.layer, act, idx_out=idx_out, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(idx_out, idx)
    tokens = np.sort(np.random.default_rng(65536).choice(wl.T, 32, replace=False))
    tokens[0], tokens[-1] = 0, wl.T - 1
    o_out = oracle_layer(case, tokens=tokens, forced_idx=idx.cpu().numpy()[tokens])[0]
    err = rel_l2_max(out.double().cpu().numpy()[tokens], o_out)
    print(f"T=65536 ({'bf16' if bf16 else 'f32'}): max rel L2 over 32 sampled tokens {err:.3e}")
    assert err < (1e-2 if bf16 else TOL_F32)
