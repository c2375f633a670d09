"""Q4_0 experts (fp16 scale, 16 bytes of 4-bit values per 32-wide block)
through the C ABI against the oracle decoding the same blocks.

Q4_0 with fp32 activations runs on the lane-per-row kernels for every
batch size (bf16 activations at 128+ pairs take the tensor-core path, tested
in test_gpu_tc.py), so the cases
span one and two tokens (which Q8_0 sends elsewhere), the staged-all-tokens
and per-chunk variants of the gate/up kernel, and one to three K stages per
warp in the down kernel (d_ff 256 to 768).
Routing does not depend on the weight format; it is checked again here
because each case draws its own router.
"""
import zlib

import numpy as np
import pytest
import torch

from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_F32, check_routing, make_case, oracle_layer, rel_l2_max

pytestmark = pytest.mark.gpu

SHAPES = [
    # name, T, d, f, E, k, zipf
    ("q4_t1", 1, 512, 256, 16, 4, False),       # one K stage per down warp
    ("q4_t2", 2, 1024, 512, 32, 4, True),       # two K stages per down warp
    ("q4_t3", 3, 512, 768, 16, 2, False),       # three K stages per down warp
    ("q4_t7", 7, 1024, 256, 24, 3, True),       # all tokens staged
    ("q4_d256", 5, 256, 256, 16, 4, False),     # one K stage per gate/up warp
    ("q4_t21", 21, 512, 768, 16, 4, True),      # per-chunk activations, ragged 8-pair chunks
    ("q4_t64", 64, 1024, 512, 32, 8, False),
    ("q4_t2_full", 2, 2048, 768, 128, 8, False),
]


def _wl(name, T, d, f, E, k, zipf):
    return synth.custom(name, wid=zlib.crc32(name.encode()) % 10000 + 500,
                        T=T, d_model=d, d_ff=f, E=E, k=k, zipf=zipf, wfmt="q4")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def test_pack_q4_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(3)
    w = torch.randn(37, 96, generator=g, device="cuda") * 0.02
    blocks = synth.quantize_q4_0(w)
    qs, d = binding.pack_q4(blocks, 37, 96)
    b = blocks.cpu().numpy().reshape(37, 3, 18)
    assert np.array_equal(qs.cpu().numpy().reshape(37, 3, 16), b[:, :, 2:])
    assert np.array_equal(d.cpu().numpy().view(np.uint8).reshape(37, 3, 2), b[:, :, :2])


def _check(case, act=binding.MOE_ACT_F32, flags=0, residual=False):
    wl = case.wl
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    wts = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    out = binding.layer_forward(case.x, case.layer, act, flags=flags, residual=residual, idx_out=idx, wts_out=wts)
    torch.cuda.synchronize()
    gidx = idx.cpu().numpy()
    o_out, o_idx, o_w, o_l = oracle_layer(case, residual=residual)
    if check_routing(gidx, wts.cpu().numpy(), o_idx, o_w, o_l, wl.k):
        o_out = oracle_layer(case, forced_idx=gidx, residual=residual)[0]
    err = rel_l2_max(out.cpu().numpy().astype(np.float64), o_out)
    assert err < TOL_F32, f"max rel L2 {err:.3e}"
    return err


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s[0])
@pytest.mark.parametrize("flags", [0, binding.MOE_FLAG_DETERMINISTIC], ids=["atomic", "det"])
def test_layer_q4_small(shape, flags):
    _check(make_case(_wl(*shape)), flags=flags)


@pytest.mark.parametrize("name", ["decode_t1_q4", "decode_t64_zipf_q4"])
def test_layer_q4_workloads(name):
    err = _check(make_case(synth.WORKLOADS[name]))
    print(f"{name}: max rel L2 {err:.3e}")


def test_layer_q4_residual():
    _check(make_case(_wl("q4_res", 9, 512, 256, 16, 4, True)), residual=True)


def test_layer_q4_bf16_act_small_batch_runs_fp32():
    """MOE_ACT_BF16 with Q4_0 weights and fewer than 128 pairs (one MMA
    tile) runs the fp32 kernels: fp32 accuracy against the oracle fed the
    fp32 inputs.  (128 pairs or more take the tensor-core path, tested with
    the other tensor-core cases.)"""
    _check(make_case(_wl("q4_bf16", 15, 1024, 512, 32, 8, False)), act=binding.MOE_ACT_BF16)


def test_q4_differs_from_q8():
    """The same seeded weights in Q8_0 and Q4_0 give different outputs (the
    format field is honoured), each matching its own oracle."""
    wl4 = _wl("q4_vs_q8", 5, 512, 256, 16, 4, False)
    wl8 = synth.custom("q4_vs_q8", wid=wl4.wid, T=5, d_model=512, d_ff=256, E=16, k=4)
    c4, c8 = make_case(wl4), make_case(wl8)
    _check(c4)
    _check(c8)
    o4 = binding.layer_forward(c4.x, c4.layer)
    o8 = binding.layer_forward(c8.x, c8.layer)
    torch.cuda.synchronize()
    assert torch.equal(c4.x, c8.x)
    rel = (o4 - o8).norm() / o8.norm()
    assert 1e-3 < rel.item() < 0.5


def test_q4_unsupported_geometry():
    """d_ff 128 is not a multiple of 256 (the down kernel splits K = d_ff into
    four 64-wide slices): Q4_0 is refused before any launch."""
    wl = _wl("q4_bad", 3, 256, 128, 8, 2, False)
    case = make_case(wl)
    with pytest.raises(binding.MoeError) as ei:
        binding.layer_forward(case.x, case.layer)
    assert ei.value.rc == binding.MOE_ERR_UNSUPPORTED


def test_layer_q4_prefill_t1024_sampled():
    """Q4_0 at the full geometry and a prefill batch (lane-per-row kernels,
    per-chunk activations, 128 experts): 48 sampled tokens against the oracle."""
    wl = _wl("q4_t1024", 1024, 2048, 768, 128, 8, False)
    case = make_case(wl)
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    out = binding.layer_forward(case.x, case.layer, idx_out=idx)
    torch.cuda.synchronize()
    tokens = np.sort(np.random.default_rng(1024).choice(wl.T, 48, replace=False))
    o_out = oracle_layer(case, tokens=tokens, forced_idx=idx.cpu().numpy()[tokens])[0]
    err = rel_l2_max(out.double().cpu().numpy()[tokens], o_out)
    assert err < TOL_F32, f"max rel L2 {err:.3e}"
