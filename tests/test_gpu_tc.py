"""GPU parity of the tensor-core (tcgen05, bf16 operands) expert path against
the CPU oracle: routing bit-exact, layer outputs within max relative L2 1e-2."""
import zlib

import numpy as np
import pytest
import torch

from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_BF16, check_routing, make_case, oracle_layer, rel_l2_max

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


def _run(case, flags=0, residual=False):
    wl = case.wl
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    wts = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.layer_forward(case.x, case.layer, binding.MOE_ACT_BF16, flags=flags, residual=residual,
                                idx_out=idx, wts_out=wts, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    return out.cpu().double().numpy(), idx.cpu().numpy(), wts.cpu().numpy()


def _check(case, tokens=None, flags=0, residual=False):
    g, gidx, gw = _run(case, flags, residual)
    sel = slice(None) if tokens is None else tokens
    o_out, o_idx, o_w, o_l = oracle_layer(case, tokens=tokens, forced_idx=gidx[sel], residual=residual)
    if tokens is None:
        check_routing(gidx, gw, *oracle_layer(case)[1:], case.wl.k)
    x = case.host["x"][sel]
    moe_g = g[sel] - x if residual else g[sel]
    moe_o = o_out - x if residual else o_out
    err = rel_l2_max(moe_g, moe_o)
    # diagnostic: against the oracle fed the same bf16-rounded expert inputs
    o_bf = oracle_layer(case, tokens=tokens, forced_idx=gidx[sel], bf16=True)[0]
    err_bf = rel_l2_max(g[sel] - (x if residual else 0), o_bf)
    print(f"{case.wl.name}: max rel L2 {err:.3e} (vs bf16-input oracle {err_bf:.3e})")
    assert err < TOL_BF16, f"max rel L2 {err:.3e}"
    return err


def _wl(name, T, d, f, E, k, zipf=False, wfmt="q8"):
    return synth.custom(name, wid=zlib.crc32(name.encode()) % 10000 + 300,
                        T=T, d_model=d, d_ff=f, E=E, k=k, zipf=zipf, act="bf16", wfmt=wfmt)


@pytest.mark.parametrize("shape", [
    ("tc_small", 64, 256, 256, 16, 8, False),
    ("tc_zipf", 100, 512, 768, 32, 4, True),
    ("tc_k2", 96, 768, 256, 8, 2, False),
], ids=lambda s: s[0])
def test_tc_layer_small(shape):
    _check(make_case(_wl(*shape)))


def test_tc_layer_small_deterministic_residual():
    case = make_case(_wl("tc_det", 64, 256, 256, 16, 8, True))
    _check(case, flags=binding.MOE_FLAG_DETERMINISTIC, residual=True)


def test_tc_many_tokens_one_expert():
    """A dominant bias sends all 300 tokens to expert 2: its bucket spans three 128-pair tiles."""
    wl = _wl("tc_hot", 300, 256, 256, 16, 4)
    case = make_case(wl)
    bias = torch.zeros(wl.E, device="cuda")
    bias[2] = 100.0
    case.layer = binding.Layer(wl.E, wl.k, wl.d_model, wl.d_ff, case.layer.gate, case.layer.up, case.layer.down,
                               case.layer.router_w, bias)
    case.host["bias"] = bias.cpu().numpy()
    _check(case)


@pytest.mark.parametrize("shape", [
    ("tc_q4_small", 64, 256, 256, 16, 8, False),     # one 256-K raw stage per row tile
    ("tc_q4_zipf", 100, 512, 768, 32, 4, True),      # three raw stages of the down projection
    ("tc_q4_ragged", 37, 1024, 512, 64, 8, False),   # 296 pairs, ragged buckets
], ids=lambda s: s[0])
def test_tc_layer_q4(shape):
    """Q4_0 experts on the tensor-core path (nibbles dequantised into the
    MMA's A operand): the same bf16 tolerance against the oracle decoding the
    same Q4_0 blocks."""
    _check(make_case(_wl(*shape, wfmt="q4")))


def test_tc_layer_q4_deterministic_residual():
    case = make_case(_wl("tc_q4_det", 64, 512, 256, 16, 8, True, wfmt="q4"))
    _check(case, flags=binding.MOE_FLAG_DETERMINISTIC, residual=True)


@pytest.mark.parametrize("name", ["prefill_t1024", "prefill_t768", "prefill_t2048", "prefill_t1024_q4"])
def test_tc_prefill_full_sampled(name):
    """qwen3_moe geometry: routing for all tokens, outputs on sampled tokens."""
    case = make_case(synth.WORKLOADS[name])
    g, gidx, gw = _run(case)
    oi, ow, ol = __import__("oracle").get().route(case.host["x"], case.host["Wr"], case.host["bias"], case.wl.k)
    near = check_routing(gidx, gw, oi, ow, ol, case.wl.k)
    print(f"{name}: near-tie tokens {near}")
    tokens = np.sort(np.random.default_rng(2).choice(case.wl.T, 40, replace=False))
    tokens[0], tokens[-1] = 0, case.wl.T - 1
    o_out = oracle_layer(case, tokens=tokens, forced_idx=gidx[tokens])[0]
    err = rel_l2_max(g[tokens], o_out)
    print(f"{name}: max rel L2 {err:.3e} on {len(tokens)} sampled tokens")
    assert err < TOL_BF16


def test_tc_repeatable_with_deterministic_flag():
    case = make_case(_wl("tc_rep", 128, 256, 256, 16, 8, True))
    a = _run(case, flags=binding.MOE_FLAG_DETERMINISTIC)[0]
    b = _run(case, flags=binding.MOE_FLAG_DETERMINISTIC)[0]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [
    ("tc_reuse_multi", 512, 1024, 256, 8, 2, True),    # ~128 pairs per expert: several chunks each; 2 bands
    ("tc_reuse_t2048", 2048, 2048, 768, 128, 8, False),  # the full geometry in one call
], ids=lambda s: s[0])
def test_reuse_order_traversal(shape):
    """The band traversal of the down projection (MOE_FLAG_REUSE_ORDER) runs
    the same tiles in another order: bit-identical with the fixed-order
    combine, within fp32 reassociation of the atomic combine otherwise, and
    within the bf16 tolerance of the oracle."""
    case = make_case(_wl(*shape))
    det = binding.MOE_FLAG_DETERMINISTIC
    a, ia, _ = _run(case, det)
    b, ib, _ = _run(case, det | binding.MOE_FLAG_REUSE_ORDER)
    assert np.array_equal(ia, ib)
    assert np.array_equal(a, b)
    c, _, _ = _run(case, 0)
    d, _, _ = _run(case, binding.MOE_FLAG_REUSE_ORDER)
    assert rel_l2_max(d, c) < 1e-5
    tokens = np.sort(np.random.default_rng(4).choice(case.wl.T, 24, replace=False))
    _check(case, tokens=tokens, flags=binding.MOE_FLAG_REUSE_ORDER)
