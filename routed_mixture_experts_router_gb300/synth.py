"""Seeded synthetic inputs for the routed MoE layer.

This module holds no arithmetic of the layer itself: it draws hidden states,
router weights, router biases and expert weights, and encodes the expert
weights into Q8_0 bytes.  Both the CUDA path and the CPU oracle consume what
it produces; neither imports the other.

Distributions (the workloads of the qwen3_moe geometry, d_model 2048,
d_ff 768, 128 experts, top-8, 48 layers -- amalgafy.com/evidence,
"Historical baseline environment"):

* hidden states x ~ N(0, 1), fp32;
* router weights Wr ~ N(0, std = 1/sqrt(d_model)), fp32;
* expert weights ~ N(0, std = 0.02), encoded as Q8_0;
* optional router bias with a Zipf(s = 1.1) rank profile scaled to 2.0:
  a seeded permutation gives expert e the rank r_e in 1..E and
  bias_e = 2.0 * r_e ** -1.1.

Q8_0 encoding (input preparation only; the layer never quantises weights):
per 32-weight block along K, amax = max |w|, d32 = amax / 127 (fp32),
q = clamp(round_half_away(w / d32), -127, 127), stored scale d = fp16(d32)
(round to nearest even); an all-zero block stores d = 0 and q = 0.  A block
is 34 bytes: the fp16 scale (little endian) followed by the 32 int8 values.
This is the block the pages' "native Q8_0 weights" use: 34 B per 32 weights,
which reproduces their printed expert-cache sizes (amalgafy.com/evidence,
"Cache tradeoff" table).

Seeds: every tensor gets its own generator, seeded from
(workload id, layer, tensor id), so any tensor can be regenerated alone.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

Q8_BLOCK = 32
Q8_BLOCK_BYTES = 34
Q4_BLOCK_BYTES = 18

# tensor ids for the seed scheme
_T_X, _T_WR, _T_BIAS, _T_GATE, _T_UP, _T_DOWN = range(6)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: geometry, routing skew and expert-input dtype."""
    name: str
    wid: int          # workload id used in the seed scheme
    T: int            # tokens per layer call
    d_model: int
    d_ff: int
    E: int
    k: int
    zipf: bool = False
    act: str = "f32"  # "f32": fp32 expert inputs; "bf16": tensor-core path
    layers: int = 1
    residual: bool = False
    wfmt: str = "q8"  # expert weight blocks: "q8" (Q8_0, 34 B) or "q4" (Q4_0, 18 B)
    arena_slots: int = 0  # > 0: experts served from an arena of this many HBM slots
    microbatch: int = 0   # > 0: the T tokens run as T / microbatch layer calls of this many tokens


WORKLOADS = {
    # tiny layer: T=4, d 256, d_ff 128, 16 experts, top-2
    "tiny": Workload("tiny", 1, 4, 256, 128, 16, 2),
    # qwen3_moe geometry, decode T=1, uniform routing
    "decode_t1": Workload("decode_t1", 2, 1, 2048, 768, 128, 8),
    # batched decode T=64 with Zipf-skewed router bias
    "decode_t64_zipf": Workload("decode_t64_zipf", 3, 64, 2048, 768, 128, 8, zipf=True),
    # prefill T=1024 (also 768, and 2048 as two 1024-token microbatches), bf16 expert inputs
    "prefill_t1024": Workload("prefill_t1024", 4, 1024, 2048, 768, 128, 8, act="bf16"),
    "prefill_t768": Workload("prefill_t768", 4, 768, 2048, 768, 128, 8, act="bf16"),
    "prefill_t2048": Workload("prefill_t2048", 4, 2048, 2048, 768, 128, 8, act="bf16"),
    # the same 2048 tokens as two 1024-token microbatches (two layer calls)
    "prefill_t2048_mb1024": Workload("prefill_t2048_mb1024", 4, 2048, 2048, 768, 128, 8, act="bf16",
                                     microbatch=1024),
    # 48-layer stack, residual between layers, Zipf routing; T in {1, 64, 1024}
    "stack48_t1": Workload("stack48_t1", 5, 1, 2048, 768, 128, 8, zipf=True, layers=48, residual=True),
    "stack48_t64": Workload("stack48_t64", 5, 64, 2048, 768, 128, 8, zipf=True, layers=48, residual=True),
    "stack48_t1024": Workload("stack48_t1024", 5, 1024, 2048, 768, 128, 8, zipf=True, act="bf16", layers=48,
                              residual=True),
    # the stack48_t1 weights served from a 1,536-slot expert arena (25% of the
    # 6,144 experts resident, the pages' main cache configuration), a new
    # token every step
    "arena48_t1": Workload("arena48_t1", 5, 1, 2048, 768, 128, 8, zipf=True, layers=48, residual=True,
                           arena_slots=1536),
    # Q4_0 experts (the 4-bit format of the pages' next stage), decode
    "decode_t1_q4": Workload("decode_t1_q4", 6, 1, 2048, 768, 128, 8, wfmt="q4"),
    "decode_t64_zipf_q4": Workload("decode_t64_zipf_q4", 7, 64, 2048, 768, 128, 8, zipf=True, wfmt="q4"),
    "prefill_t1024_q4": Workload("prefill_t1024_q4", 8, 1024, 2048, 768, 128, 8, act="bf16", wfmt="q4"),
}


def seed_for(wid: int, layer: int, tensor: int, extra: int = 0) -> int:
    """Deterministic 63-bit seed from (workload id, layer, tensor id, extra)."""
    h = 0x9E3779B97F4A7C15
    for v in (wid, layer, tensor, extra):
        h ^= (v + 0x632BE59BD9B4E019 + ((h << 6) & 0xFFFFFFFFFFFFFFFF) + (h >> 2)) & 0xFFFFFFFFFFFFFFFF
        h = (h * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    return h & 0x7FFFFFFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def quantize_q8_0(w: torch.Tensor) -> torch.Tensor:
    """Encode fp32 weights [..., K] (K % 32 == 0) into Q8_0 bytes [..., K/32*34] (uint8)."""
    assert w.dtype == torch.float32 and w.shape[-1] % Q8_BLOCK == 0
    lead = w.shape[:-1]
    K = w.shape[-1]
    blk = w.reshape(*lead, K // Q8_BLOCK, Q8_BLOCK)
    amax = blk.abs().amax(dim=-1, keepdim=True)
    d32 = amax / 127.0
    safe = torch.where(d32 > 0, d32, torch.ones_like(d32))
    v = blk / safe
    q = torch.sign(v) * torch.floor(v.abs() + 0.5)        # round half away from zero
    q = torch.clamp(q, -127, 127)
    q = torch.where(d32 > 0, q, torch.zeros_like(q)).to(torch.int8)
    d16 = d32.to(torch.float16)
    by = torch.cat([d16.contiguous().view(torch.uint8), q.contiguous().view(torch.uint8)], dim=-1)
    return by.reshape(*lead, (K // Q8_BLOCK) * Q8_BLOCK_BYTES).contiguous()


def quantize_q4_0(w: torch.Tensor) -> torch.Tensor:
    """Encode fp32 weights [..., K] (K % 32 == 0) into Q4_0 bytes [..., K/32*18] (uint8).

    Per 32-block: d32 = max|w| / 7, q = clamp(round_half_away(w / d32), -8, 7),
    stored as n = q + 8 in 4 bits: byte j holds element j (low nibble) and
    element j + 16 (high nibble); the fp16 scale leads the block.
    """
    assert w.dtype == torch.float32 and w.shape[-1] % Q8_BLOCK == 0
    lead = w.shape[:-1]
    K = w.shape[-1]
    blk = w.reshape(*lead, K // Q8_BLOCK, Q8_BLOCK)
    amax = blk.abs().amax(dim=-1, keepdim=True)
    d32 = amax / 7.0
    safe = torch.where(d32 > 0, d32, torch.ones_like(d32))
    v = blk / safe
    q = torch.sign(v) * torch.floor(v.abs() + 0.5)
    q = torch.clamp(q, -8, 7)
    q = torch.where(d32 > 0, q, torch.zeros_like(q))
    n = (q + 8).to(torch.uint8)
    packed = n[..., :16] | (n[..., 16:] << 4)
    d16 = d32.to(torch.float16)
    by = torch.cat([d16.contiguous().view(torch.uint8), packed.contiguous()], dim=-1)
    return by.reshape(*lead, (K // Q8_BLOCK) * Q4_BLOCK_BYTES).contiguous()


def q4_matrix_bytes(rows: int, K: int) -> int:
    return rows * (K // Q8_BLOCK) * Q4_BLOCK_BYTES


def q8_matrix_bytes(rows: int, K: int) -> int:
    return rows * (K // Q8_BLOCK) * Q8_BLOCK_BYTES


def zipf_bias(E: int, gen: torch.Generator, device) -> torch.Tensor:
    """bias_e = 2.0 * rank_e ** -1.1 with a seeded permutation of ranks 1..E."""
    perm = torch.randperm(E, generator=gen, device=device)
    rank = (perm + 1).to(torch.float64)
    return (2.0 * rank.pow(-1.1)).to(torch.float32)


def make_x(wl: Workload, device, step: int = 0, T: int | None = None) -> torch.Tensor:
    """Hidden states x [T][d_model] fp32 ~ N(0,1) for one step of a workload."""
    T = wl.T if T is None else T
    g = _gen(device, seed_for(wl.wid, 0, _T_X, step))
    return torch.randn(T, wl.d_model, generator=g, device=device, dtype=torch.float32)


def make_router(wl: Workload, layer: int, device):
    """(Wr [E][d_model] fp32, bias [E] fp32 or None)."""
    g = _gen(device, seed_for(wl.wid, layer, _T_WR))
    Wr = torch.randn(wl.E, wl.d_model, generator=g, device=device, dtype=torch.float32)
    Wr.mul_(1.0 / (wl.d_model ** 0.5))
    bias = None
    if wl.zipf:
        bias = zipf_bias(wl.E, _gen(device, seed_for(wl.wid, layer, _T_BIAS)), device)
    return Wr, bias


def make_expert_q8(wl: Workload, layer: int, which: str, device, chunk: int = 16) -> torch.Tensor:
    """Quantised bytes of one expert matrix family for all E experts, in the
    workload's block format (Q8_0, or Q4_0 when wl.wfmt == "q4").

    which = "gate" | "up": E x [d_ff][d_model]; "down": E x [d_model][d_ff].
    Returns uint8 [E][rows * K/32 * block bytes].  Generated `chunk` experts at
    a time to bound temporary memory.
    """
    tid = {"gate": _T_GATE, "up": _T_UP, "down": _T_DOWN}[which]
    rows, K = (wl.d_ff, wl.d_model) if which != "down" else (wl.d_model, wl.d_ff)
    q4 = wl.wfmt == "q4"
    g = _gen(device, seed_for(wl.wid, layer, tid))
    nbytes = q4_matrix_bytes(rows, K) if q4 else q8_matrix_bytes(rows, K)
    out = torch.empty(wl.E, nbytes, dtype=torch.uint8, device=device)
    for e0 in range(0, wl.E, chunk):
        n = min(chunk, wl.E - e0)
        w = torch.randn(n, rows, K, generator=g, device=device, dtype=torch.float32).mul_(0.02)
        out[e0:e0 + n] = (quantize_q4_0(w) if q4 else quantize_q8_0(w)).reshape(n, -1)
        del w
    return out


def make_layer(wl: Workload, layer: int, device) -> dict:
    """All weights of one layer: Wr, bias, and quantised gate/up/down bytes (AoS blocks)."""
    Wr, bias = make_router(wl, layer, device)
    return {
        "Wr": Wr,
        "bias": bias,
        "gate": make_expert_q8(wl, layer, "gate", device),
        "up": make_expert_q8(wl, layer, "up", device),
        "down": make_expert_q8(wl, layer, "down", device),
    }


def custom(name: str = "custom", wid: int = 99, **kw) -> Workload:
    """A workload with explicit geometry (tests of odd shapes)."""
    return Workload(name, wid, **kw)
