"""The single-launch decode path (one or two tokens, fp32 activations, Q8_0
or Q4_0 experts)
against the CPU oracle, through the C ABI: routing bit-exact (near-ties
counted), outputs within max relative L2 1e-5, at several geometries, with
and without the residual, tokens sharing experts, repeated calls on one
workspace, a workspace holding arbitrary bytes before the call (the launch
clears what it needs) and x in page-locked host memory."""
import zlib

import numpy as np
import pytest
import torch

from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_F32, check_routing, make_case, oracle_layer, rel_l2_max

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def _wl(name, T, d, f, E, k, zipf, wfmt="q8"):
    return synth.custom(name, wid=zlib.crc32(name.encode()) % 10000 + 500, T=T, d_model=d, d_ff=f, E=E, k=k,
                        zipf=zipf, wfmt=wfmt)


def _run(case, residual=False, flags=0, ws=None, x=None):
    wl = case.wl
    x = case.x if x is None else x
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    wts = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    off = torch.empty(wl.E + 1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(wl.T, wl.d_model, dtype=torch.float32, device="cuda")
    ws = binding.workspace(wl.T, case.layer, binding.MOE_ACT_F32, flags, "cuda") if ws is None else ws
    binding.layer_forward(x, case.layer, binding.MOE_ACT_F32, flags=flags, residual=residual, out=out, ws=ws,
                          idx_out=idx, wts_out=wts, offsets_out=off, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    return out, idx, wts, off


def _check(case, residual=False, flags=0, ws=None):
    out, idx, wts, off = _run(case, residual, flags, ws)
    gidx = idx.cpu().numpy()
    o_out, o_idx, o_w, o_l = oracle_layer(case, residual=residual)
    near = check_routing(gidx, wts.cpu().numpy(), o_idx, o_w, o_l, case.wl.k)
    if near:
        o_out = oracle_layer(case, residual=residual, forced_idx=gidx)[0]
    x = case.host["x"]
    g = out.cpu().double().numpy()
    err = rel_l2_max(g - x if residual else g, o_out - x if residual else o_out)
    assert err < TOL_F32, f"max rel L2 {err:.3e}"
    # offsets: the exclusive scan of the bucket sizes of the GPU's selection
    cnt = np.bincount(gidx.ravel(), minlength=case.wl.E)
    assert np.array_equal(off.cpu().numpy(), np.concatenate([[0], np.cumsum(cnt)]))
    return out, err


GEOMS = [
    # name, T, d_model, d_ff, E, k, zipf
    ("qwen_t1", 1, 2048, 768, 128, 8, False),
    ("qwen_t2", 2, 2048, 768, 128, 8, True),
    ("d512_f256", 1, 512, 256, 16, 2, False),
    ("d1024_f512_t2", 2, 1024, 512, 64, 4, True),
    ("d1536_f1024", 1, 1536, 1024, 32, 8, False),
    ("e256_k16_t2", 2, 2048, 256, 256, 16, True),
    ("e8_k8", 1, 1024, 768, 8, 8, False),         # k == E: every expert, full softmax
    ("k1_t2", 2, 2048, 768, 128, 1, False),
    # Q4_0 experts: a 16-byte chunk of a row holds a whole 32-value block;
    # CTA ranges start on 16-feature boundaries, i.e. mid-block
    ("q4_t1", 1, 2048, 768, 128, 8, False, "q4"),
    ("q4_t2", 2, 2048, 768, 128, 8, True, "q4"),
    ("q4_d1024_f512_t2", 2, 1024, 512, 64, 4, True, "q4"),
    ("q4_e256_k16_t2", 2, 2048, 256, 256, 16, True, "q4"),
    ("q4_k1", 1, 1024, 256, 16, 1, False, "q4"),
]


@pytest.mark.parametrize("shape", GEOMS, ids=lambda s: s[0])
@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
def test_decode_layer_geometries(shape, residual):
    _check(make_case(_wl(*shape)), residual=residual)


@pytest.mark.parametrize("shape", GEOMS, ids=lambda s: s[0])
def test_decode_geometries_separate_kernels(shape):
    """The same geometries through the separate router, bucketing and expert
    kernels (the deterministic combine takes that path)."""
    _check(make_case(_wl(*shape)), flags=binding.MOE_FLAG_DETERMINISTIC)


def test_decode_t2_tokens_share_experts():
    """Two identical tokens: every routed expert serves both (two pairs per bucket)."""
    case = make_case(_wl("twin", 2, 2048, 768, 128, 8, True))
    case.x[1].copy_(case.x[0])
    case.host["x"] = case.x.double().cpu().numpy()
    out, _ = _check(case)
    # same routing and values; only the order of the fp32 atomic adds differs
    o = out.double().cpu().numpy()
    assert rel_l2_max(o[:1], o[1:]) < 1e-6


@pytest.mark.parametrize("name", ["decode_t1", "stack48_t1", "decode_t1_q4"])
def test_decode_any_workspace_bytes(name):
    """Whatever the workspace held before (every byte random, the published
    logit words included), the call gives the same routing and, up to the
    order of the fp32 atomic adds, the same output."""
    case = make_case(synth.WORKLOADS[name])
    ws = binding.workspace(1, case.layer)
    ref, ridx = (t.clone() for t in _run(case, ws=ws, residual=case.wl.residual)[:2])
    g = torch.Generator(device="cuda").manual_seed(3)
    for i in range(4):
        ws.copy_(torch.randint(0, 256, ws.shape, generator=g, device="cuda", dtype=torch.int32).to(ws.dtype))
        out, idx = _run(case, ws=ws, residual=case.wl.residual)[:2]
        assert torch.equal(idx, ridx)
        assert rel_l2_max(out.double().cpu().numpy(), ref.double().cpu().numpy()) < 1e-6


def test_decode_many_calls_one_workspace():
    """Many back-to-back calls on one stream and one workspace: every output
    matches its own single call."""
    case = make_case(synth.WORKLOADS["decode_t1"])
    ws = binding.workspace(1, case.layer)
    xs = [synth.make_x(case.wl, "cuda", step=100 + i) for i in range(37)]
    outs = [binding.layer_forward(x, case.layer, ws=ws) for x in xs]
    torch.cuda.synchronize()
    for x, o in zip(xs[::9], outs[::9]):
        ref = binding.layer_forward(x, case.layer)
        torch.cuda.synchronize()
        assert rel_l2_max(o.double().cpu().numpy(), ref.double().cpu().numpy()) < 1e-6


def test_decode_host_x():
    """x read straight from page-locked host memory (GB300: coherent over NVLink-C2C)."""
    case = make_case(synth.WORKLOADS["decode_t1"])
    xh = case.x.cpu().pin_memory()
    ref = _run(case)[0]
    out = _run(case, x=xh)[0]
    assert rel_l2_max(out.double().cpu().numpy(), ref.double().cpu().numpy()) < 1e-6


def test_decode_graph_replays_see_new_inputs():
    """One layer call captured in a CUDA graph and replayed with x changed in
    place each time: every replay routes and computes the new token (no
    routing result of an earlier launch is taken for this one's)."""
    case = make_case(synth.WORKLOADS["decode_t1"])
    x = case.x.clone()
    out = torch.empty_like(x)
    idx = torch.empty(1, case.wl.k, dtype=torch.int32, device="cuda")
    ws = binding.workspace(1, case.layer)
    binding.layer_forward(x, case.layer, out=out, ws=ws, idx_out=idx)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            binding.layer_forward(x, case.layer, out=out, ws=ws, idx_out=idx)
    for step in range(6):
        x.copy_(synth.make_x(case.wl, "cuda", step=20 + step))
        g.replay()
        torch.cuda.synchronize()
        ridx = torch.empty_like(idx)
        ref = binding.layer_forward(x, case.layer, idx_out=ridx)
        torch.cuda.synchronize()
        assert torch.equal(idx, ridx), step
        assert rel_l2_max(out.double().cpu().numpy(), ref.double().cpu().numpy()) < 1e-6, step


def test_decode_inputs_written_by_the_previous_kernel():
    """The decode kernel may start while the previous kernel in the stream
    still runs (programmatic dependent launch): x, the router weights and the
    bias written by the kernels right before the call must all be the values
    it uses.  Each step, captured once in a graph, first overwrites them in
    place (a copy kernel), then runs the layer."""
    case = make_case(synth.WORKLOADS["stack48_t1"])  # Zipf bias: all three inputs matter
    layer = case.layer
    x = case.x.clone()
    out = torch.empty_like(x)
    idx = torch.empty(1, case.wl.k, dtype=torch.int32, device="cuda")
    ws = binding.workspace(1, layer)
    srcs = []
    for step in range(4):
        wr, b = synth.make_router(case.wl, 10 + step, "cuda")
        srcs.append((synth.make_x(case.wl, "cuda", step=40 + step), wr, b))
    nx, nwr, nb = (torch.empty_like(t) for t in srcs[0])
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.layer_forward(x, layer, out=out, ws=ws, idx_out=idx)  # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            x.copy_(nx)
            layer.router_w.copy_(nwr)
            layer.router_bias.copy_(nb)
            binding.layer_forward(x, layer, out=out, ws=ws, idx_out=idx)
    for sx, swr, sb in srcs:
        nx.copy_(sx)
        nwr.copy_(swr)
        nb.copy_(sb)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref_layer = binding.Layer(case.wl.E, case.wl.k, case.wl.d_model, case.wl.d_ff, layer.gate, layer.up,
                                  layer.down, swr, sb)
        ridx = torch.empty_like(idx)
        ref = binding.layer_forward(sx, ref_layer, idx_out=ridx)
        torch.cuda.synchronize()
        assert torch.equal(idx, ridx)
        assert rel_l2_max(out.double().cpu().numpy(), ref.double().cpu().numpy()) < 1e-6
