"""CPU oracle for the OSCAR-style 2-bit rotated KV cache (TEST INFRASTRUCTURE ONLY).

Only tests/, the package's smoke check and the benchmark's CPU-baseline leg may import
this package.  It shares no code with the CUDA library; the one thing both sides take is
the seeded input generator module, which holds none of the method's arithmetic.

Layers:
  oscar_oracle.c   plain C: bf16 rounding, the fp32 rotation chain, the INT2 quantizer
                   and packer, the append state machine, fp64 decode attention.
  calibration.py   numpy: covariances, eigenbases, Hadamard, bit reversal, clip.
  model.py         a whole cache (layers x requests x kv-heads) built from those calls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oscar_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboscar_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, no fast-math, fp contraction off)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
               "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            so = build()
            L = ctypes.CDLL(so)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int, ctypes.c_long, ctypes.c_float
            L.oo_f32_to_bf16.argtypes = [f32]
            L.oo_f32_to_bf16.restype = ctypes.c_uint16
            L.oo_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oo_bf16_to_f32.restype = f32
            L.oo_code_bitpos.argtypes = [i32]
            L.oo_code_bitpos.restype = i32
            L.oo_pack_row.argtypes = [P, i32, P]
            L.oo_unpack_row.argtypes = [P, i32, P]
            L.oo_rotate.argtypes = [P, P, i64, i32, P]
            L.oo_quantize_token.argtypes = [P, i32, i32, f32, P, P]
            L.oo_dequant_token.argtypes = [P, P, i32, i32, P]
            L.oo_append.argtypes = [i32, i32, i32, i32, f32, P, P, P, P, P, P, P, i64, P, i64]
            L.oo_append.restype = i32
            L.oo_decode.argtypes = [i32, i32, i32, i32, i32, i32, i32] + [P] * 12
            L.oo_decode_folded.argtypes = [i32, i32, i32, i32, i32, i32, i32] + [P] * 10
            L.oo_bf16_decode.argtypes = [i32, i32, i64, P, P, P, P]
            L.oo_max_threads.restype = i32
            L.oo_set_threads.argtypes = [i32]
            _lib = L
        return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    raise TypeError("expected bf16 bit patterns as uint16")


def set_threads(n: int) -> None:
    lib().oo_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oo_max_threads())


def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, np.uint16)
    L = lib()
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = L.oo_f32_to_bf16(float(flat_in[i]))
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def code_bitpos(c: int) -> int:
    return int(lib().oo_code_bitpos(int(c)))


def pack_row(codes) -> np.ndarray:
    codes = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    d = codes.size
    row = np.zeros(d // 4, np.uint8)
    lib().oo_pack_row(_p(codes), d, _p(row))
    return row


def unpack_row(row, d: int = 128) -> np.ndarray:
    row = np.ascontiguousarray(np.asarray(row, dtype=np.uint8))
    codes = np.zeros(d, np.uint8)
    lib().oo_unpack_row(_p(row), d, _p(codes))
    return codes


def rotate(R: np.ndarray, x) -> np.ndarray:
    """bf16 r = R^T x per token, the fixed fp32 fma chain.  x: uint16 [..., d]."""
    R = np.ascontiguousarray(R, dtype=np.float32)
    x = _u16(x)
    d = R.shape[0]
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    lib().oo_rotate(_p(R), _p(flat), flat.shape[0], d, _p(out))
    return out.reshape(x.shape)


def quantize_token(r, g: int, clip: float):
    """(32-byte code row, sz[ng*2] bf16 bits) of one rotated bf16 token."""
    r = _u16(r)
    d = r.size
    row = np.zeros(d // 4, np.uint8)
    sz = np.zeros((d // g) * 2, np.uint16)
    lib().oo_quantize_token(_p(r), d, g, float(clip), _p(row), _p(sz))
    return row, sz


def dequant_token(row, sz, g: int, d: int = 128) -> np.ndarray:
    row = np.ascontiguousarray(np.asarray(row, dtype=np.uint8))
    sz = _u16(sz)
    out = np.zeros(d, np.float32)
    lib().oo_dequant_token(_p(row), _p(sz), d, g, _p(out))
    return out


class Stream:
    """One request x layer x kv-head x {K or V} token stream of the mixed-precision cache."""

    def __init__(self, d: int, g: int, n_sink: int, window: int, capacity: int, R: np.ndarray, clip: float):
        self.d, self.g, self.S, self.W = d, g, n_sink, window
        self.R = np.ascontiguousarray(R, dtype=np.float32)
        self.clip = float(clip)
        self.L = np.zeros(1, np.int32)
        self.H = np.full(1, n_sink, np.int32)
        self.sink = np.zeros((max(n_sink, 1), d), np.uint16)
        self.ring = np.zeros((max(window, 1), d), np.uint16)
        self.rows = np.zeros((capacity, d // 4), np.uint8)
        self.sz = np.zeros((capacity, (d // g) * 2), np.uint16)
        self.capacity = capacity

    @property
    def length(self) -> int:
        return int(self.L[0])

    @property
    def history_end(self) -> int:
        return int(self.H[0])

    def append(self, x) -> None:
        x = _u16(x).reshape(-1, self.d)
        rc = lib().oo_append(self.d, self.g, self.S, self.W, self.clip, _p(self.R), _p(self.L), _p(self.H),
                             _p(self.sink), _p(self.ring), _p(self.rows), _p(self.sz), self.capacity, _p(x),
                             x.shape[0])
        if rc != 0:
            raise ValueError("oracle stream capacity exceeded")

    def share_from(self, src: "Stream", n_tokens: int) -> None:
        """Take src's first n_tokens (all history or sink) as this empty stream's own."""
        assert self.length == 0 and n_tokens <= src.history_end
        self.sink[:] = src.sink
        self.rows[:n_tokens] = src.rows[:n_tokens]
        self.sz[:n_tokens] = src.sz[:n_tokens]
        self.L[0] = n_tokens
        self.H[0] = max(n_tokens, self.S)

    def route(self, p: int) -> str:
        if p < min(self.length, self.S):
            return "sink"
        if p < self.history_end:
            return "int2"
        return "ring"


def decode(q, K: Stream, V: Stream, R_K: np.ndarray, R_V: np.ndarray) -> np.ndarray:
    """fp64 attention output [G, d] for the G query heads of one kv-head."""
    q = _u16(q)
    G, d = q.shape
    out = np.zeros((G, d), np.float64)
    R_K = np.ascontiguousarray(R_K, dtype=np.float32)
    R_V = np.ascontiguousarray(R_V, dtype=np.float32)
    assert K.length == V.length and K.history_end == V.history_end
    lib().oo_decode(d, G, K.g, K.S, K.W, K.length, K.history_end, _p(K.sink), _p(V.sink), _p(K.ring),
                    _p(V.ring), _p(K.rows), _p(K.sz), _p(V.rows), _p(V.sz), _p(q), _p(R_K), _p(R_V), _p(out))
    return out


def decode_folded(qt, K: Stream, V: Stream) -> np.ndarray:
    """decode() with the rotations folded into the model's projections: qt are the rotated
    queries (bf16 bits [G, d]); the result is the output in the rotated basis (fp64 [G, d]),
    before the inverse value rotation."""
    qt = _u16(qt)
    G, d = qt.shape
    out = np.zeros((G, d), np.float64)
    assert K.length == V.length and K.history_end == V.history_end
    lib().oo_decode_folded(d, G, K.g, K.S, K.W, K.length, K.history_end, _p(K.sink), _p(V.sink), _p(K.ring),
                           _p(V.ring), _p(K.rows), _p(K.sz), _p(V.rows), _p(V.sz), _p(qt), _p(out))
    return out


def bf16_decode(q, K, V) -> np.ndarray:
    """fp64 softmax(q K^T / sqrt(d)) V over plain bf16 K, V [L, d]; q [G, d]."""
    q, K, V = _u16(q), _u16(K), _u16(V)
    G, d = q.shape
    out = np.zeros((G, d), np.float64)
    lib().oo_bf16_decode(d, G, K.shape[0], _p(K), _p(V), _p(q), _p(out))
    return out
