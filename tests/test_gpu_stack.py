"""The 48-layer MoE stack (x_{l+1} = x_l + MoE_l(x_l), every layer with its
own seeded router and Zipf bias, all layers resident), through the C ABI.

Layer by layer: each layer's MoE part (x_{l+1} - x_l) is checked against the
oracle evaluated on the GPU's own x_l, so errors are measured per layer and
do not compound.  The captured 48-layer CUDA graph must reproduce the same
chain run eagerly (bit for bit with the deterministic combine).
"""
import numpy as np
import pytest
import torch

import oracle
from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_BF16, TOL_F32, check_routing, rel_l2_max

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def _layer(wl, l):
    w = synth.make_layer(wl, l, "cuda")
    lay = binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"], w["Wr"],
                                    w["bias"])
    return w, lay


def _stack_layerwise(name, nlayers, tokens=None, tol=TOL_F32):
    wl = synth.WORKLOADS[name]
    bf16 = wl.act == "bf16"
    act = binding.MOE_ACT_BF16 if bf16 else binding.MOE_ACT_F32
    orc = oracle.get()
    x = synth.make_x(wl, "cuda", step=0)
    errs = []
    for l in range(nlayers):
        w, lay = _layer(wl, l)
        idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
        wts = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
        out = binding.layer_forward(x, lay, act, 0, True, idx_out=idx, wts_out=wts)
        torch.cuda.synchronize()
        h = {k: (None if v is None else v.cpu().numpy()) for k, v in w.items()}
        sel = np.arange(wl.T) if tokens is None else np.asarray(tokens)
        xh = x.double().cpu().numpy()[sel]
        gidx, gw = idx.cpu().numpy()[sel], wts.cpu().numpy()[sel]
        args = (h["Wr"], h["bias"], h["gate"], h["up"], h["down"], wl.d_model, wl.d_ff, wl.E, wl.k)
        o_out, o_idx, o_w, o_l = orc.moe_layer(xh, *args, expert_input_bf16=bf16)
        if check_routing(gidx, gw, o_idx, o_w, o_l, wl.k):
            o_out = orc.moe_layer(xh, *args, expert_input_bf16=bf16, forced_idx=gidx)[0]
        moe_gpu = out.double().cpu().numpy()[sel] - xh
        err = rel_l2_max(moe_gpu, o_out)
        errs.append(err)
        assert err < tol, f"layer {l}: max rel L2 {err:.3e}"
        assert torch.isfinite(out).all()
        x = out
        del w, lay
    return errs


def test_stack_t1_layerwise():
    errs = _stack_layerwise("stack48_t1", 6)
    print("stack48_t1 per-layer max rel L2:", ["%.2e" % e for e in errs])


def test_stack_t64_layerwise():
    errs = _stack_layerwise("stack48_t64", 4)
    print("stack48_t64 per-layer max rel L2:", ["%.2e" % e for e in errs])


def test_stack_t1024_bf16_layerwise_sampled():
    tokens = np.random.default_rng(7).choice(1024, size=48, replace=False)
    errs = _stack_layerwise("stack48_t1024", 2, tokens=tokens, tol=TOL_BF16)
    print("stack48_t1024 per-layer max rel L2 (48 sampled tokens):", ["%.2e" % e for e in errs])


@pytest.mark.parametrize("flags", [binding.MOE_FLAG_DETERMINISTIC, 0], ids=["det", "atomic"])
def test_stack48_graph_matches_eager(flags):
    """All 48 layers resident (30.8 GB), chained through two buffers; one CUDA
    graph of the whole stack == the eager chain (bit-exact when the combine
    is deterministic; with fp32 atomics the summation order differs, and the
    rounding differences pass through 48 residual layers: 1e-4)."""
    wl = synth.WORKLOADS["stack48_t1"]
    layers = []
    for l in range(wl.layers):
        w, lay = _layer(wl, l)
        layers.append(lay)
        del w
    x0 = synth.make_x(wl, "cuda", step=0)
    bufs = [torch.empty_like(x0), torch.empty_like(x0)]
    ws = binding.workspace(wl.T, layers[0], binding.MOE_ACT_F32, flags, "cuda")
    torch.cuda.synchronize()  # weights, x0 and buffers were made on the default stream
    s = torch.cuda.Stream()

    def chain():
        bufs[0].copy_(x0)
        for l, lay in enumerate(layers):
            binding.layer_forward(bufs[l % 2], lay, binding.MOE_ACT_F32, flags, True, out=bufs[(l + 1) % 2], ws=ws)

    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    eager = bufs[wl.layers % 2].clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    bufs[0].zero_()
    bufs[1].zero_()
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    replay = bufs[wl.layers % 2]
    assert torch.isfinite(replay).all()
    if flags & binding.MOE_FLAG_DETERMINISTIC:
        assert torch.equal(replay, eager)
    else:
        err = rel_l2_max(replay.double().cpu().numpy(), eager.double().cpu().numpy())
        assert err < 1e-4, f"graph vs eager max rel L2 {err:.3e}"
