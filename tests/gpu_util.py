"""Helpers shared by the GPU parity tests: building a seeded layer on the
device, copying what the oracle needs to the host, and the parity checks
(routing bit-exact up to counted near-ties, outputs by max relative L2)."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from routed_mixture_experts_router_gb300 import binding, synth

NEAR_TIE = 1e-5      # top-(k+1) adjacent logit gap that counts as a near-tie
TOL_F32 = 1e-5       # max relative L2 of the layer output, fp32-activation path
TOL_BF16 = 1e-2      # max relative L2 of the layer output, bf16 tensor-core path


@dataclass
class Case:
    wl: synth.Workload
    layer: binding.Layer
    blocks: dict          # device AoS blocks + router (the synth output)
    x: torch.Tensor       # device fp32 [T][d]
    host: dict            # numpy copies for the oracle


def wfmt_of(wl: synth.Workload) -> int:
    return binding.MOE_WFMT_Q4_0 if wl.wfmt == "q4" else binding.MOE_WFMT_Q8_0


def make_case(wl: synth.Workload, layer_id: int = 0, step: int = 0, T: int | None = None) -> Case:
    w = synth.make_layer(wl, layer_id, "cuda")
    x = synth.make_x(wl, "cuda", step, T)
    lay = binding.Layer.from_blocks(wl.E, wl.k, wl.d_model, wl.d_ff, w["gate"], w["up"], w["down"], w["Wr"],
                                    w["bias"], wfmt=wfmt_of(wl))
    torch.cuda.synchronize()
    host = {
        "x": x.double().cpu().numpy(),
        "Wr": w["Wr"].cpu().numpy(),
        "bias": None if w["bias"] is None else w["bias"].cpu().numpy(),
        "gate": w["gate"].cpu().numpy(),
        "up": w["up"].cpu().numpy(),
        "down": w["down"].cpu().numpy(),
    }
    return Case(wl, lay, w, x, host)


def oracle_layer(case: Case, tokens=None, forced_idx=None, residual=False, bf16=False, x=None):
    h = case.host
    xv = h["x"] if x is None else x
    if tokens is not None:
        xv = xv[tokens]
    wl = case.wl
    return oracle.get().moe_layer(xv, h["Wr"], h["bias"], h["gate"], h["up"], h["down"], wl.d_model, wl.d_ff, wl.E,
                                  wl.k, residual=residual, expert_input_bf16=bf16, forced_idx=forced_idx,
                                  fmt=wfmt_of(wl))


def near_tie_mask(logits: np.ndarray, k: int) -> np.ndarray:
    s = -np.sort(-logits, axis=1)[:, :k + 1]
    if s.shape[1] < 2:
        return np.zeros(logits.shape[0], dtype=bool)
    return ((s[:, :-1] - s[:, 1:]) < NEAR_TIE).any(axis=1)


def check_routing(gpu_idx: np.ndarray, gpu_w: np.ndarray, orc_idx: np.ndarray, orc_w: np.ndarray,
                  logits: np.ndarray, k: int) -> int:
    """Indices bit-exact except near-tie tokens, which must hold a valid top-k
    under the oracle's logits within the near-tie slack.  Returns the number
    of near-tie tokens."""
    near = near_tie_mask(logits, k)
    ok = ~near
    bad = np.nonzero((gpu_idx[ok] != orc_idx[ok]).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} non-tie tokens routed differently, e.g. token {np.nonzero(ok)[0][bad[0]]}"
    np.testing.assert_allclose(gpu_w[ok], orc_w[ok], rtol=0, atol=5e-6)
    E = logits.shape[1]
    for t in np.nonzero(near)[0]:
        sel = gpu_idx[t]
        assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < E
        lsel = logits[t, sel]
        rest = np.delete(logits[t], sel)
        if rest.size:
            assert lsel.min() >= rest.max() - NEAR_TIE
        assert np.all(np.diff(lsel) <= NEAR_TIE)
    # weights are a probability vector in every row
    np.testing.assert_allclose(gpu_w.sum(axis=1), 1.0, rtol=0, atol=1e-6)
    return int(near.sum())


def rel_l2_max(a: np.ndarray, b: np.ndarray) -> float:
    num = np.linalg.norm(a - b, axis=-1)
    den = np.maximum(np.linalg.norm(b, axis=-1), 1e-30)
    return float((num / den).max()) if num.size else 0.0


def check_bucket(idx: np.ndarray, E: int, off, ptok, pslot, pos):
    """Bucketing of the GPU's own idx, bit-exact against the oracle's."""
    o_off, o_pt, o_ps, o_pos = oracle.get().bucket(idx, E)
    assert np.array_equal(off, o_off)
    assert np.array_equal(ptok, o_pt)
    assert np.array_equal(pslot, o_ps)
    assert np.array_equal(pos, o_pos)
