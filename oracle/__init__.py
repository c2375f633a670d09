"""Plain fp64 CPU oracle of the routed MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product (the CUDA library and its Python
binding) never imports, links or executes anything here, and this package
never imports the product: the two share only the seeded input generators.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, no CUDA headers),
compiled with gcc into ``oracle/_build/liboracle.so`` and called via ctypes.
Every function takes and returns numpy arrays.  Weights are Q8_0 in the pages'
own 34-byte block format (fp16 scale, then 32 int8 values along K) or Q4_0
(18-byte blocks: fp16 scale, 16 bytes of 4-bit values), as raw uint8 arrays;
the oracle decodes them itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

_lock = threading.Lock()


def build(source: str = SOURCE, out: str = LIB_PATH, openmp: bool = True) -> str:
    """Compile the oracle with gcc (plain C, -O2, OpenMP over tokens)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", out + ".tmp", source, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build(out: str, source: str) -> bool:
    return (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(source)


_P = ctypes.c_void_p
_I = ctypes.c_int


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str = LIB_PATH, source: str = SOURCE):
        with _lock:
            if lib_path == LIB_PATH and _needs_build(lib_path, source):
                build(source, lib_path)
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_dequant_q8.restype = None
        lib.oracle_dequant_q8.argtypes = [_P, _I, _I, _P]
        lib.oracle_expert_swiglu.restype = _I
        lib.oracle_expert_swiglu.argtypes = [_P, _P, _P, _I, _I, _P, _P]
        lib.oracle_route.restype = _I
        lib.oracle_route.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
        lib.oracle_moe_layer.restype = _I
        lib.oracle_moe_layer.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _P]
        lib.oracle_moe_layer_fmt.restype = _I
        lib.oracle_moe_layer_fmt.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P,
                                             _P, _P]
        lib.oracle_dequant.restype = None
        lib.oracle_dequant.argtypes = [_P, _I, _I, _I, _P]
        lib.oracle_bucket.restype = _I
        lib.oracle_bucket.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P]
        lib.oracle_q8_block_bytes.restype = _I
        lib.oracle_q8_block_elems.restype = _I
        lib.oracle_num_threads.restype = _I
        self.lib = lib

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _c(a, dtype):
        return np.ascontiguousarray(a, dtype=dtype)

    @staticmethod
    def _p(a):
        return None if a is None else a.ctypes.data_as(_P)

    # -- API -----------------------------------------------------------------
    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def q8_block_bytes(self) -> int:
        return int(self.lib.oracle_q8_block_bytes())

    def q8_block_elems(self) -> int:
        return int(self.lib.oracle_q8_block_elems())

    def half_to_double(self, bits: int) -> float:
        return float(self.lib.oracle_half_to_double(ctypes.c_uint16(bits)))

    def dequant_q8(self, blocks: np.ndarray, rows: int, K: int) -> np.ndarray:
        b = self._c(blocks, np.uint8)
        assert b.size == rows * (K // 32) * 34
        out = np.empty((rows, K), dtype=np.float64)
        self.lib.oracle_dequant_q8(self._p(b), rows, K, self._p(out))
        return out

    def dequant(self, blocks: np.ndarray, rows: int, K: int, fmt: int) -> np.ndarray:
        """fmt 0: Q8_0 (34-byte blocks); 1: Q4_0 (18-byte blocks)."""
        b = self._c(blocks, np.uint8)
        assert b.size == rows * (K // 32) * (18 if fmt == 1 else 34)
        out = np.empty((rows, K), dtype=np.float64)
        self.lib.oracle_dequant(self._p(b), rows, K, fmt, self._p(out))
        return out

    def expert_swiglu(self, gate, up, down, dm: int, f: int, x: np.ndarray) -> np.ndarray:
        g, u, d = (self._c(a, np.uint8) for a in (gate, up, down))
        xv = self._c(x, np.float64)
        y = np.empty(dm, dtype=np.float64)
        if self.lib.oracle_expert_swiglu(self._p(g), self._p(u), self._p(d), dm, f, self._p(xv), self._p(y)):
            raise MemoryError("oracle_expert_swiglu: scratch allocation failed")
        return y

    def route(self, x, Wr, bias, k: int):
        xv = self._c(x, np.float64)
        T, dm = xv.shape
        wr = self._c(Wr, np.float32)
        E = wr.shape[0]
        b = None if bias is None else self._c(bias, np.float32)
        idx = np.empty((T, k), dtype=np.int32)
        w = np.empty((T, k), dtype=np.float64)
        logits = np.empty((T, E), dtype=np.float64)
        rc = self.lib.oracle_route(T, dm, E, k, self._p(xv), self._p(wr), self._p(b), self._p(idx), self._p(w),
                                   self._p(logits))
        if rc != 0:
            raise ValueError(f"oracle_route rc={rc}")
        return idx, w, logits

    def moe_layer(self, x, Wr, bias, gate, up, down, dm: int, f: int, E: int, k: int, residual: bool = False,
                  expert_input_bf16: bool = False, forced_idx=None, fmt: int = 0):
        """Returns (out [T][dm] f64, idx [T][k] i32, w [T][k] f64, logits [T][E] f64).
        fmt: expert block format, 0 = Q8_0, 1 = Q4_0."""
        xv = self._c(x, np.float64).reshape(-1, dm)
        T = xv.shape[0]
        wr = self._c(Wr, np.float32)
        b = None if bias is None else self._c(bias, np.float32)
        g, u, d = (self._c(a, np.uint8) for a in (gate, up, down))
        fi = None if forced_idx is None else self._c(forced_idx, np.int32)
        out = np.empty((T, dm), dtype=np.float64)
        idx = np.empty((T, k), dtype=np.int32)
        w = np.empty((T, k), dtype=np.float64)
        logits = np.empty((T, E), dtype=np.float64)
        rc = self.lib.oracle_moe_layer_fmt(T, dm, f, E, k, self._p(xv), self._p(wr), self._p(b), self._p(g),
                                           self._p(u), self._p(d), int(fmt), int(residual), int(expert_input_bf16),
                                           self._p(fi), self._p(out), self._p(idx), self._p(w), self._p(logits))
        if rc != 0:
            raise ValueError(f"oracle_moe_layer rc={rc}")
        return out, idx, w, logits

    def bucket(self, idx, E: int):
        iv = self._c(idx, np.int32)
        T, k = iv.shape
        P = T * k
        off = np.empty(E + 1, dtype=np.int32)
        pt = np.empty(P, dtype=np.int32)
        ps = np.empty(P, dtype=np.int32)
        pos = np.empty(P, dtype=np.int32)
        rc = self.lib.oracle_bucket(self._p(iv), T, k, E, self._p(off), self._p(pt), self._p(ps), self._p(pos))
        if rc != 0:
            raise ValueError(f"oracle_bucket rc={rc}")
        return off, pt, ps, pos


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this package's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
