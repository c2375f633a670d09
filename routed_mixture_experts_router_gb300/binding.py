"""Thin ctypes binding of libmoe_gb300.so (C ABI declared in include/moe.h).

Argument marshalling only: every function passes torch tensors' device
pointers and the current CUDA stream to the C entry point of the same name,
and raises ``MoeError`` on a non-zero return code.  No computation happens in
Python, and there is no fallback: if the library is missing or fails to load,
the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_WORKSPACE = 4
MOE_STATUS_BAD_INDEX = 1
MOE_STATUS_TIMEOUT = 2
MOE_STATUS_ARENA_FULL = 4
MOE_ACT_F32 = 0
MOE_ACT_BF16 = 1
MOE_FLAG_DETERMINISTIC = 1
MOE_FLAG_REUSE_ORDER = 2
MOE_WFMT_Q8_0 = 0
MOE_WFMT_Q4_0 = 1

_ERR = {1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA", 4: "MOE_ERR_WORKSPACE"}

ENTRY_POINTS = ("moe_workspace_size", "moe_pack_q8", "moe_pack_q4", "moe_arena_blob_bytes", "moe_arena_state_bytes",
                "moe_arena_init", "moe_arena_pack_blob", "moe_arena_admit", "moe_layer_forward_arena", "moe_route", "moe_bucket", "moe_expert_ffn_q8", "moe_combine",
                "moe_layer_forward", "moe_layer_forward_static", "moe_version")
MOE_STATIC_SCRATCH_BYTES = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"{fn} returned {rc} ({_ERR.get(rc, 'unknown')})")
        self.rc = rc


class Q8Mat(ctypes.Structure):
    _fields_ = [("qs", ctypes.c_void_p), ("d", ctypes.c_void_p)]


class LayerW(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("k", ctypes.c_int), ("d_model", ctypes.c_int), ("d_ff", ctypes.c_int),
                ("gate", Q8Mat), ("up", Q8Mat), ("down", Q8Mat), ("router_w", ctypes.c_void_p),
                ("router_bias", ctypes.c_void_p), ("wfmt", ctypes.c_int), ("n_slots", ctypes.c_int),
                ("expert_slot", ctypes.c_void_p)]


class ArenaStats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_ulonglong), ("misses", ctypes.c_ulonglong), ("bytes_in", ctypes.c_ulonglong),
                ("clock", ctypes.c_uint), ("layers", ctypes.c_int), ("experts", ctypes.c_int), ("slots", ctypes.c_int),
                ("last_misses", ctypes.c_int), ("full_events", ctypes.c_int), ("reserved", ctypes.c_int * 2)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe_gb300.so not found at {path}; build it with "
                           "`python -m routed_mixture_experts_router_gb300.build`")
    L = ctypes.CDLL(path)
    P, I, LL, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
    LWP = ctypes.POINTER(LayerW)
    L.moe_workspace_size.restype = SZ
    L.moe_workspace_size.argtypes = [I, LWP, I, I]
    L.moe_pack_q8.restype = I
    L.moe_pack_q8.argtypes = [P, LL, I, P, P, P]
    L.moe_pack_q4.restype = I
    L.moe_pack_q4.argtypes = [P, LL, I, P, P, P]
    L.moe_arena_blob_bytes.restype = SZ
    L.moe_arena_blob_bytes.argtypes = [LWP]
    L.moe_arena_state_bytes.restype = SZ
    L.moe_arena_state_bytes.argtypes = [I, I, I]
    L.moe_arena_init.restype = I
    L.moe_arena_init.argtypes = [P, I, I, I, P]
    L.moe_arena_pack_blob.restype = I
    L.moe_arena_pack_blob.argtypes = [LWP, I, I, P, P]
    L.moe_arena_admit.restype = I
    L.moe_arena_admit.argtypes = [P, I, P, I, P, LWP, P, P, P]
    L.moe_layer_forward_arena.restype = I
    L.moe_layer_forward_arena.argtypes = [P, I, LWP, I, I, I, P, P, I, P, P, SZ, P, P]
    L.moe_route.restype = I
    L.moe_route.argtypes = [P, I, LWP, P, P, P]
    L.moe_bucket.restype = I
    L.moe_bucket.argtypes = [P, I, I, I, P, P, P, P, P, P]
    L.moe_expert_ffn_q8.restype = I
    L.moe_expert_ffn_q8.argtypes = [P, I, LWP, P, P, P, P, I, I, P, I, P, SZ, P, P]
    L.moe_combine.restype = I
    L.moe_combine.argtypes = [P, P, P, I, I, I, P, P, P]
    L.moe_layer_forward.restype = I
    L.moe_layer_forward.argtypes = [P, I, LWP, I, I, I, P, P, P, P, P, SZ, P, P]
    L.moe_layer_forward_static.restype = I
    L.moe_layer_forward_static.argtypes = [P, I, LWP, I, I, I, P, P, P]
    L.moe_version.restype = ctypes.c_char_p
    L.moe_version.argtypes = []
    _lib = L
    return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoeError(fn, rc)


class Layer:
    """Device-resident weights of one MoE layer in the library's layout.

    Holds the packed expert tensors (Q8_0: qs [E][rows][K], bytes q + 128; Q4_0: qs
    uint8 [E][rows][K/2]; d fp16-bits [E][rows][K/32]) and the fp32 router,
    plus the C struct pointing at them.  wfmt: MOE_WFMT_Q8_0 or MOE_WFMT_Q4_0.
    """

    def __init__(self, E, k, d_model, d_ff, gate, up, down, router_w, router_bias=None, wfmt=None, n_slots=0,
                 expert_slot=None):
        wfmt = MOE_WFMT_Q8_0 if wfmt is None else wfmt
        self.E, self.k, self.d_model, self.d_ff, self.wfmt = E, k, d_model, d_ff, wfmt
        self.n_slots, self.expert_slot = n_slots, expert_slot
        self.gate, self.up, self.down = gate, up, down          # (qs, d) tuples
        self.router_w = router_w.contiguous()
        self.router_bias = None if router_bias is None else router_bias.contiguous()
        self.c = LayerW(E, k, d_model, d_ff, Q8Mat(gate[0].data_ptr(), gate[1].data_ptr()),
                        Q8Mat(up[0].data_ptr(), up[1].data_ptr()), Q8Mat(down[0].data_ptr(), down[1].data_ptr()),
                        self.router_w.data_ptr(), 0 if self.router_bias is None else self.router_bias.data_ptr(),
                        wfmt, n_slots, 0 if expert_slot is None else expert_slot.data_ptr())

    @classmethod
    def from_blocks(cls, E, k, d_model, d_ff, gate_blocks, up_blocks, down_blocks, router_w, router_bias=None,
                    wfmt=None):
        """Pack 34-byte Q8_0 blocks (moe_pack_q8) or, for wfmt MOE_WFMT_Q4_0,
        18-byte Q4_0 blocks (moe_pack_q4); device uint8 tensors."""
        wfmt = MOE_WFMT_Q8_0 if wfmt is None else wfmt
        pack = pack_q4 if wfmt == MOE_WFMT_Q4_0 else pack_q8
        gate = pack(gate_blocks, E * d_ff, d_model)
        up = pack(up_blocks, E * d_ff, d_model)
        down = pack(down_blocks, E * d_model, d_ff)
        return cls(E, k, d_model, d_ff, gate, up, down, router_w, router_bias, wfmt)

    def ref(self):
        return ctypes.byref(self.c)


def version() -> str:
    return load().moe_version().decode()


def pack_q8(blocks: torch.Tensor, rows: int, K: int):
    """moe_pack_q8: 34-byte blocks -> (qs [rows][K] holding q + 128 as bytes, d int16-bits [rows][K/32])."""
    L = load()
    qs = torch.empty(rows, K, dtype=torch.int8, device=blocks.device)
    d = torch.empty(rows, K // 32, dtype=torch.int16, device=blocks.device)
    _check("moe_pack_q8", L.moe_pack_q8(_ptr(blocks), rows, K, _ptr(qs), _ptr(d), _stream()))
    return qs, d


def pack_q4(blocks: torch.Tensor, rows: int, K: int):
    """moe_pack_q4: 18-byte blocks -> (qs uint8 [rows][K/2], d int16-bits [rows][K/32])."""
    L = load()
    qs = torch.empty(rows, K // 2, dtype=torch.uint8, device=blocks.device)
    d = torch.empty(rows, K // 32, dtype=torch.int16, device=blocks.device)
    _check("moe_pack_q4", L.moe_pack_q4(_ptr(blocks), rows, K, _ptr(qs), _ptr(d), _stream()))
    return qs, d


def workspace_size(T: int, layer: Layer, act: int = MOE_ACT_F32, flags: int = 0) -> int:
    return int(load().moe_workspace_size(T, layer.ref(), act, flags))


def workspace(T: int, layer: Layer, act: int = MOE_ACT_F32, flags: int = 0, device="cuda") -> torch.Tensor:
    n = workspace_size(T, layer, act, flags)
    if n == 0 and T > 0:
        raise MoeError("moe_workspace_size", MOE_ERR_INVALID_ARG)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def route(x: torch.Tensor, layer: Layer):
    T = x.shape[0]
    idx = torch.empty(T, layer.k, dtype=torch.int32, device=x.device)
    wts = torch.empty(T, layer.k, dtype=torch.float32, device=x.device)
    _check("moe_route", load().moe_route(_ptr(x), T, layer.ref(), _ptr(idx), _ptr(wts), _stream()))
    return idx, wts


def bucket(idx: torch.Tensor, E: int, status: torch.Tensor | None = None):
    T, k = idx.shape
    dev = idx.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    pair_tok = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    pair_slot = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    pos = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    _check("moe_bucket", load().moe_bucket(_ptr(idx), T, k, E, _ptr(offsets), _ptr(pair_tok), _ptr(pair_slot),
                                           _ptr(pos), _ptr(status), _stream()))
    return offsets, pair_tok[:T * k], pair_slot[:T * k], pos[:T * k]


def expert_ffn_q8(x, layer: Layer, offsets, pair_tok, pair_slot, wts, act=MOE_ACT_F32, fuse_combine=True,
                  residual=False, ws=None, status=None, out=None):
    T = x.shape[0]
    if out is None:
        rows = T if fuse_combine else T * layer.k
        out = torch.empty(rows, layer.d_model, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(T, layer, act, 0, x.device)
    _check("moe_expert_ffn_q8", load().moe_expert_ffn_q8(
        _ptr(x), T, layer.ref(), _ptr(offsets), _ptr(pair_tok), _ptr(pair_slot), _ptr(wts), act,
        int(bool(fuse_combine)), _ptr(out), int(bool(residual)), _ptr(ws), ws.numel(), _ptr(status), _stream()))
    return out


def combine(ypairs, wts, pos, T: int, k: int, d_model: int, residual=None, out=None):
    if out is None:
        out = torch.empty(T, d_model, dtype=torch.float32, device=ypairs.device)
    _check("moe_combine", load().moe_combine(_ptr(ypairs), _ptr(wts), _ptr(pos), T, k, d_model, _ptr(residual),
                                             _ptr(out), _stream()))
    return out


def layer_forward(x, layer: Layer, act=MOE_ACT_F32, flags=0, residual=False, out=None, ws=None, status=None,
                  idx_out=None, wts_out=None, offsets_out=None):
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, layer.d_model, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(T, layer, act, flags, x.device)
    _check("moe_layer_forward", load().moe_layer_forward(
        _ptr(x), T, layer.ref(), act, flags, int(bool(residual)), _ptr(out), _ptr(idx_out), _ptr(wts_out),
        _ptr(offsets_out), _ptr(ws), ws.numel(), _ptr(status), _stream()))
    return out


def layer_forward_static(x, layer: Layer, act=MOE_ACT_F32, flags=0, residual=False, out=None, status=None):
    """moe_layer_forward_static: the layer forward with the library's fixed
    scratch region instead of a caller workspace (for callers that cannot
    allocate device memory where they run the layer)."""
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, layer.d_model, dtype=torch.float32, device=x.device)
    _check("moe_layer_forward_static", load().moe_layer_forward_static(
        _ptr(x), T, layer.ref(), act, flags, int(bool(residual)), _ptr(out), _ptr(status), _stream()))
    return out


# ------------------------------------------------------------- expert arena --
class Arena:
    """An expert arena: `slots` HBM slots for the experts of `layers` layers of
    one geometry and format, the residency state (moe_arena_state_bytes) and
    every expert's blob in page-locked host memory (blob l*E + e).

    template: any Layer of that geometry/format (only its shape is used).
    """

    def __init__(self, template: Layer, layers: int, slots: int, device="cuda"):
        L = load()
        self.E, self.k, self.d_model, self.d_ff, self.wfmt = (template.E, template.k, template.d_model,
                                                              template.d_ff, template.wfmt)
        self.layers, self.slots = layers, slots
        f, dm = self.d_ff, self.d_model
        q4 = self.wfmt == MOE_WFMT_Q4_0
        u8 = torch.uint8 if q4 else torch.int8

        def mat(rows, K):
            return (torch.empty(slots, rows, K // 2 if q4 else K, dtype=u8, device=device),
                    torch.empty(slots, rows, K // 32, dtype=torch.int16, device=device))
        self.gate, self.up, self.down = mat(f, dm), mat(f, dm), mat(dm, f)
        self.blob_bytes = int(L.moe_arena_blob_bytes(template.ref()))
        if self.blob_bytes == 0:
            raise MoeError("moe_arena_blob_bytes", MOE_ERR_INVALID_ARG)
        n = int(L.moe_arena_state_bytes(layers, self.E, slots))
        if n == 0:
            raise MoeError("moe_arena_state_bytes", MOE_ERR_INVALID_ARG)
        self.state = torch.empty(n, dtype=torch.uint8, device=device)
        self.host_blobs = torch.empty(layers * self.E * self.blob_bytes, dtype=torch.uint8, pin_memory=True)
        self.reset()

    def reset(self):
        _check("moe_arena_init", load().moe_arena_init(_ptr(self.state), self.layers, self.E, self.slots, _stream()))

    def blob(self, layer: int, e: int) -> torch.Tensor:
        i = layer * self.E + e
        return self.host_blobs[i * self.blob_bytes:(i + 1) * self.blob_bytes]

    def pack_layer(self, layer: int, weights: Layer):
        """Write every expert blob of layer `layer` from resident weights (expert order)."""
        L = load()
        for e in range(self.E):
            _check("moe_arena_pack_blob", L.moe_arena_pack_blob(weights.ref(), layer, e,
                                                                ctypes.c_void_p(self.blob(layer, e).data_ptr()),
                                                                _stream()))

    def layer(self, router_w, router_bias=None, slot_map=None) -> Layer:
        """A Layer over the arena slots with this router (slot_map: the FFN's expert -> slot map, or None)."""
        return Layer(self.E, self.k, self.d_model, self.d_ff, self.gate, self.up, self.down, router_w, router_bias,
                     self.wfmt, n_slots=self.slots, expert_slot=slot_map)

    def stats(self) -> dict:
        raw = self.state[:ctypes.sizeof(ArenaStats)].cpu().numpy().tobytes()
        st = ArenaStats.from_buffer_copy(raw)
        return {k: getattr(st, k) for k, _ in ArenaStats._fields_ if k != "reserved"}

    def tables(self):
        """(slot_of [L][E], owner [S], stamp [S]) as host arrays (layout of include/moe.h's arena state)."""
        def a256(v):
            return (v + 255) & ~255
        o = a256(ctypes.sizeof(ArenaStats))
        n_so = self.layers * self.E
        slot_of = self.state[o:o + 4 * n_so].view(torch.int32).cpu().numpy().reshape(self.layers, self.E)
        o = a256(o + 4 * n_so)
        owner = self.state[o:o + 4 * self.slots].view(torch.int32).cpu().numpy()
        o = a256(o + 4 * self.slots)
        stamp = self.state[o:o + 4 * self.slots].view(torch.int32).cpu().numpy().view("uint32")
        return slot_of, owner, stamp


def arena_admit(arena: Arena, layer: int, offsets: torch.Tensor, P: int, arena_layer: Layer, slot_map=None,
                status=None):
    """moe_arena_admit: returns the expert -> slot map (int32 [E])."""
    if slot_map is None:
        slot_map = torch.empty(arena.E, dtype=torch.int32, device=offsets.device)
    _check("moe_arena_admit", load().moe_arena_admit(
        _ptr(arena.state), layer, _ptr(offsets), P, ctypes.c_void_p(arena.host_blobs.data_ptr()),
        arena_layer.ref(), _ptr(slot_map), _ptr(status), _stream()))
    return slot_map


def layer_forward_arena(x, arena_layer: Layer, arena: Arena, layer: int, act=MOE_ACT_F32, flags=0, residual=False,
                        out=None, ws=None, status=None):
    T = x.shape[0]
    if out is None:
        out = torch.empty(T, arena_layer.d_model, dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(T, arena_layer, act, flags, x.device)
    _check("moe_layer_forward_arena", load().moe_layer_forward_arena(
        _ptr(x), T, arena_layer.ref(), act, flags, int(bool(residual)), _ptr(out), _ptr(arena.state), layer,
        ctypes.c_void_p(arena.host_blobs.data_ptr()), _ptr(ws), ws.numel(), _ptr(status), _stream()))
    return out
