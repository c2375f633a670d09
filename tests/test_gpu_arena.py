"""The expert arena on the GPU, through the C ABI.

* Admissions: the device's slot map, residency tables and counters equal the
  plain-Python LRU oracle's after every admission (integer work: bit-exact),
  and every occupied slot holds exactly its owner's weights.
* The layer through the arena equals the same layer with all experts
  resident, bit for bit with the fixed-order combine, on every kernel family
  that reads the slot map (streaming, lane-per-row Q8_0 and Q4_0,
  tcgen05), and matches the oracle.
* Too few slots: MOE_STATUS_ARENA_FULL, outputs stay finite.
* A captured CUDA graph of arena layers replays like the eager calls.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from oracle.arena import ArenaOracle
from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_F32, rel_l2_max

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def _wl(name, T, d, f, E, k, wfmt="q8", zipf=True):
    return synth.custom(name, wid=zlib.crc32(name.encode()) % 10000 + 700, T=T, d_model=d, d_ff=f, E=E, k=k,
                        zipf=zipf, wfmt=wfmt)


def _layers(wl, n):
    out = []
    for l in range(n):
        w = synth.make_layer(wl, l, "cuda")
        fmt = binding.MOE_WFMT_Q4_0 if wl.wfmt == "q4" else binding.MOE_WFMT_Q8_0
        out.append((w, binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"],
                                                 w["Wr"], w["bias"], wfmt=fmt)))
    return out


def _arena(wl, layers, S):
    ar = binding.Arena(layers[0][1], len(layers), S)
    for l, (_, lay) in enumerate(layers):
        ar.pack_layer(l, lay)
    torch.cuda.synchronize()
    return ar


def _check_slots(ar, layers, owner):
    """Every occupied slot holds its owner's six weight segments, byte for byte."""
    E = ar.E
    for s, key in enumerate(owner):
        if key < 0:
            continue
        l, e = divmod(int(key), E)
        lay = layers[l][1]
        for got, want in ((ar.gate, lay.gate), (ar.up, lay.up), (ar.down, lay.down)):
            for a, b in zip(got, want):
                n = a[s].numel()
                assert torch.equal(a[s].reshape(-1), b.reshape(-1)[e * n:(e + 1) * n]), (s, key)


def test_blob_layout():
    wl = _wl("arena_blob", 2, 512, 256, 8, 2)
    layers = _layers(wl, 1)
    ar = _arena(wl, layers, 4)
    lay = layers[0][1]
    payload = 3 * 256 * 512 + 3 * 256 * 512 // 16
    assert ar.blob_bytes == 4096 + ((payload + 4095) // 4096) * 4096
    b = ar.blob(0, 5).numpy()
    hdr = b[:32].view(np.uint32)
    assert hdr.tolist() == [0x424F454D, 1, 0, 0, 5, 512, 256, payload]
    assert not b[32:4096].any()
    seg = [lay.gate[0], lay.up[0], lay.down[0], lay.gate[1], lay.up[1], lay.down[1]]
    o = 4096
    for t in seg:
        want = t.view(torch.uint8).reshape(8, -1)[5].cpu().numpy()
        assert np.array_equal(b[o:o + want.size], want)
        o += want.size
    assert o == 4096 + payload


def test_qwen_blob_size():
    """Q8_0 at d_model 2048, d_ff 768: 5,017,600-byte blobs (the pages' bytes per miss)."""
    wl = synth.WORKLOADS["decode_t1"]
    lay = binding.Layer(wl.E, wl.k, wl.d_model, wl.d_ff, (torch.empty(16, dtype=torch.int8, device="cuda"),) * 2,
                        (torch.empty(16, dtype=torch.int8, device="cuda"),) * 2,
                        (torch.empty(16, dtype=torch.int8, device="cuda"),) * 2,
                        torch.empty(16, device="cuda"))
    assert int(binding.load().moe_arena_blob_bytes(lay.ref())) == 5_017_600


@pytest.mark.parametrize("S", [10, 48])
def test_admissions_match_oracle(S):
    L, E = 3, 16
    wl = _wl(f"arena_adm{S}", 2, 512, 256, E, 4)
    layers = _layers(wl, L)
    ar = _arena(wl, layers, S)
    orc = ArenaOracle(L, E, S)
    rng = np.random.default_rng(S)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for it in range(40):
        layer = int(rng.integers(L))
        active = np.sort(rng.choice(E, size=int(rng.integers(1, 9)), replace=False))
        counts = np.zeros(E, dtype=np.int32)
        counts[active] = rng.integers(1, 4, size=active.size)
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        off_d = torch.from_numpy(offsets).cuda()
        arena_layer = ar.layer(layers[layer][0]["Wr"], layers[layer][0]["bias"])
        smap = binding.arena_admit(ar, layer, off_d, int(offsets[-1]), arena_layer, status=status)
        want = orc.admit(layer, active.tolist())
        torch.cuda.synchronize()
        assert smap.cpu().numpy().tolist() == want, it
        slot_of, owner, stamp = ar.tables()
        assert slot_of.reshape(-1).tolist() == orc.slot_of
        assert owner.tolist() == orc.owner
        assert stamp.tolist() == orc.stamp
        st = ar.stats()
        assert (st["hits"], st["misses"], st["clock"], st["last_misses"], st["full_events"]) == \
            (orc.hits, orc.misses, orc.clock, orc.last_misses, orc.full_events)
        assert st["bytes_in"] == orc.misses * (ar.blob_bytes - 4096)
        if it % 8 == 7:
            _check_slots(ar, layers, owner)
    assert status.item() == 0
    assert orc.misses > 0 and (S >= L * E or orc.hits > 0)


CASES = [
    # name, T, d, f, E, k, wfmt, act
    ("arena_q8_t1", 1, 512, 256, 16, 4, "q8", binding.MOE_ACT_F32),      # streaming kernels
    ("arena_q8_t5", 5, 1024, 512, 16, 4, "q8", binding.MOE_ACT_F32),     # lane-per-row kernels
    ("arena_q4_t1", 1, 512, 256, 16, 4, "q4", binding.MOE_ACT_F32),      # lane-per-row, Q4_0
    ("arena_q4_t7", 7, 512, 768, 16, 4, "q4", binding.MOE_ACT_F32),
    ("arena_bf16_t32", 32, 512, 256, 16, 4, "q8", binding.MOE_ACT_BF16),  # tcgen05 (128 pairs)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_layer_through_arena_equals_resident(case):
    name, T, d, f, E, k, wfmt, act = case
    wl = _wl(name, T, d, f, E, k, wfmt)
    L = 2
    S = 12 if T * k <= 12 else E   # room for every expert one call routes to: no refusals
    layers = _layers(wl, L)
    ar = _arena(wl, layers, S)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flags = binding.MOE_FLAG_DETERMINISTIC
    for step in range(6):
        l = step % L
        w, lay = layers[l]
        x = synth.make_x(wl, "cuda", step=step)
        al = ar.layer(w["Wr"], w["bias"])
        got = binding.layer_forward_arena(x, al, ar, l, act, flags, status=status)
        want = binding.layer_forward(x, lay, act, flags)
        torch.cuda.synchronize()
        assert torch.equal(got, want), (name, step)
    assert status.item() == 0
    st = ar.stats()
    assert st["misses"] > 0 and st["clock"] == 6
    # the atomic combine through the arena against the oracle
    w, lay = layers[0]
    x = synth.make_x(wl, "cuda", step=9)
    got = binding.layer_forward_arena(x, ar.layer(w["Wr"], w["bias"]), ar, 0, binding.MOE_ACT_F32, 0)
    torch.cuda.synchronize()
    h = {kk: (None if v is None else v.cpu().numpy()) for kk, v in w.items()}
    o_out = oracle.get().moe_layer(x.double().cpu().numpy(), h["Wr"], h["bias"], h["gate"], h["up"], h["down"], d, f,
                                   E, k, fmt=1 if wfmt == "q4" else 0)[0]
    assert rel_l2_max(got.double().cpu().numpy(), o_out) < TOL_F32


def test_arena_full_flags_and_stays_finite():
    wl = _wl("arena_full", 4, 512, 256, 16, 4, zipf=False)
    layers = _layers(wl, 1)
    ar = _arena(wl, layers, 2)   # 4 tokens x top-4 route to more than 2 experts
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    w, _ = layers[0]
    out = binding.layer_forward_arena(synth.make_x(wl, "cuda"), ar.layer(w["Wr"], w["bias"]), ar, 0,
                                      status=status)
    torch.cuda.synchronize()
    assert status.item() & binding.MOE_STATUS_ARENA_FULL
    assert torch.isfinite(out).all()
    st = ar.stats()
    assert st["full_events"] == 1 and st["misses"] == 2


def test_arena_graph_replay():
    """Three arena layers captured in one CUDA graph; replays after a reset
    give the eager outputs and the same residency counters."""
    wl = _wl("arena_graph", 1, 512, 256, 16, 4)
    L = 3
    layers = _layers(wl, L)
    ar = _arena(wl, layers, 10)
    x0 = synth.make_x(wl, "cuda", step=3)
    bufs = [torch.empty_like(x0) for _ in range(L + 1)]
    ws = binding.workspace(1, layers[0][1], binding.MOE_ACT_F32, binding.MOE_FLAG_DETERMINISTIC, "cuda")
    als = [ar.layer(w["Wr"], w["bias"]) for w, _ in layers]
    s = torch.cuda.Stream()

    def chain():
        bufs[0].copy_(x0)
        for l in range(L):
            binding.layer_forward_arena(bufs[l], als[l], ar, l, binding.MOE_ACT_F32, binding.MOE_FLAG_DETERMINISTIC,
                                        residual=True, out=bufs[l + 1], ws=ws)

    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    eager, st_eager = bufs[L].clone(), ar.stats()
    ar.reset()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    ar.reset()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bufs[L], eager)
    assert ar.stats() == st_eager


@pytest.mark.parametrize("T", [1, 64])
def test_arena_full_geometry(T):
    """The qwen3_moe geometry (d_model 2048, d_ff 768, 128 experts, top-8,
    5,017,600-byte blobs), two layers alternating: the arena layer equals the
    resident layer bit for bit with the fixed-order combine."""
    wl = _wl(f"arena_full_t{T}", T, 2048, 768, 128, 8)
    L = 2
    S = 16 if T == 1 else 128
    layers = _layers(wl, L)
    ar = _arena(wl, layers, S)
    assert ar.blob_bytes == 5_017_600
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(4):
        l = step % L
        w, lay = layers[l]
        x = synth.make_x(wl, "cuda", step=step)
        got = binding.layer_forward_arena(x, ar.layer(w["Wr"], w["bias"]), ar, l, binding.MOE_ACT_F32,
                                          binding.MOE_FLAG_DETERMINISTIC, status=status)
        want = binding.layer_forward(x, lay, binding.MOE_ACT_F32, binding.MOE_FLAG_DETERMINISTIC)
        torch.cuda.synchronize()
        assert torch.equal(got, want), step
    assert status.item() == 0
    st = ar.stats()
    assert st["misses"] > 0 and st["bytes_in"] == st["misses"] * 5_013_504
