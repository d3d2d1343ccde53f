"""CPU oracle for the FP8 (e4m3) 3D convolution with a BF16 NCDHW output, and its BF16-input twin.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. It imports nothing from the
CUDA package and the CUDA package imports nothing from it.

The arithmetic lives in ``conv3d_fp8_oracle.c`` (plain C, fp64, OpenMP over output channels);
this module only builds that file with gcc and marshals numpy arrays through ctypes.
What it computes, and the passages it follows, are stated in the C file's header.
``alias.py`` holds the padded-row alias predictor (a counting function, no convolution);
``quantize.py`` the per-tensor e4m3 quantiser (numpy).

Every function here is pinned by ``tests/test_oracle_pins.py`` against values fixed by the
e4m3/bfloat16 formats, closed forms, special cases that reduce to library routines, brute force
on tiny inputs, and the figures printed on the subject page.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv3d_fp8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_conv3d_fp8.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP if the compiler has it). Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r2 = subprocess.run(base, capture_output=True, text=True)
        if r2.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr + "\n" + r2.stderr)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_ubyte)
            dp = ctypes.POINTER(ctypes.c_double)
            u16p = ctypes.POINTER(ctypes.c_ushort)
            i64p = ctypes.POINTER(ctypes.c_longlong)
            ci = ctypes.c_int
            lib.o_e4m3_decode.restype = ctypes.c_double
            lib.o_e4m3_decode.argtypes = [ctypes.c_ubyte]
            lib.o_bf16_rne.restype = ctypes.c_ushort
            lib.o_bf16_rne.argtypes = [ctypes.c_double]
            lib.o_out_dim.restype = ci
            lib.o_out_dim.argtypes = [ci, ci, ci, ci]
            lib.o_max_threads.restype = ci
            lib.o_max_threads.argtypes = []
            shape = [ci] * 15
            lib.o_conv3d_fp8.restype = ci
            lib.o_conv3d_fp8.argtypes = ([u8p, u8p, ctypes.c_float, ctypes.c_float] + shape
                                         + [dp, dp, u16p])
            lib.o_conv3d_fp8_points.restype = ci
            lib.o_conv3d_fp8_points.argtypes = ([u8p, u8p, ctypes.c_float, ctypes.c_float] + shape
                                                + [i64p, ctypes.c_longlong, dp, dp, u16p])
            lib.o_bf16_decode.restype = ctypes.c_double
            lib.o_bf16_decode.argtypes = [ctypes.c_ushort]
            lib.o_conv3d_bf16.restype = ci
            lib.o_conv3d_bf16.argtypes = [u16p, u16p] + shape + [dp, u16p]
            lib.o_conv3d_bf16_points.restype = ci
            lib.o_conv3d_bf16_points.argtypes = ([u16p, u16p] + shape
                                                 + [i64p, ctypes.c_longlong, dp, u16p])
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _triple(v) -> tuple[int, int, int]:
    if isinstance(v, int):
        return (v, v, v)
    t = tuple(int(i) for i in v)
    assert len(t) == 3
    return t


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use (1 when built without OpenMP)."""
    return int(_load().o_max_threads())


def e4m3_decode(b) -> np.ndarray:
    """Exact fp64 value of each e4m3 byte (NaN for 0x7F / 0xFF)."""
    lib = _load()
    b = np.asarray(b, dtype=np.uint8)
    out = np.array([lib.o_e4m3_decode(int(v)) for v in b.ravel()], dtype=np.float64)
    return out.reshape(b.shape)


def bf16_rne(v) -> np.ndarray:
    """bfloat16 bit pattern of each double, rounded to nearest even in one step."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    out = np.array([lib.o_bf16_rne(float(a)) for a in v.ravel()], dtype=np.uint16)
    return out.reshape(v.shape)


def bf16_decode(bits) -> np.ndarray:
    """Exact fp64 value of each bfloat16 bit pattern, decoded from the format definition."""
    lib = _load()
    bits = np.asarray(bits, dtype=np.uint16)
    out = np.array([lib.o_bf16_decode(int(v)) for v in bits.ravel()], dtype=np.float64)
    return out.reshape(bits.shape)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Value of bfloat16 bit patterns (shift into the top half of an fp32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def out_dims(D: int, H: int, W: int, T: int, R: int, S: int, stride, pad) -> tuple[int, int, int]:
    lib = _load()
    sd, sh, sw = _triple(stride)
    pd, ph, pw = _triple(pad)
    return (lib.o_out_dim(D, T, sd, pd), lib.o_out_dim(H, R, sh, ph), lib.o_out_dim(W, S, sw, pw))


def _shape_args(x: np.ndarray, w: np.ndarray, stride, pad):
    assert x.ndim == 5 and w.ndim == 5 and x.shape[1] == w.shape[1]
    N, C, D, H, W = (int(v) for v in x.shape)
    K, _, T, R, S = (int(v) for v in w.shape)
    sd, sh, sw = _triple(stride)
    pd, ph, pw = _triple(pad)
    return (N, C, D, H, W, K, T, R, S, sd, sh, sw, pd, ph, pw)


def _check(rc: int):
    if rc == -1:
        raise ValueError("oracle: invalid shape, stride or padding")
    if rc == -2:
        raise ValueError("oracle: NaN (or, for bfloat16, infinite) value in an input")
    if rc == -3:
        raise IndexError("oracle: output index out of range")
    if rc != 0:
        raise RuntimeError(f"oracle: error {rc}")


def conv3d_fp8(x: np.ndarray, w: np.ndarray, sx: float, sw: float, stride=1, pad=1,
               want_sum: bool = False):
    """Full convolution. x: uint8 [N,C,D,H,W] e4m3 bytes; w: uint8 [K,C,T,R,S].

    Returns (y64, ybf16) -- or (ysum, y64, ybf16) with ``want_sum`` -- each [N,K,Do,Ho,Wo].
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint8)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    args = _shape_args(x, w, stride, pad)
    N, _, D, H, W_, K, T, R, S, sd, sh, sww, pd, ph, pw = args
    Do, Ho, Wo = out_dims(D, H, W_, T, R, S, (sd, sh, sww), (pd, ph, pw))
    if min(Do, Ho, Wo) <= 0:
        raise ValueError("oracle: empty output")
    shape = (N, K, Do, Ho, Wo)
    ysum = np.empty(shape, np.float64) if want_sum else None
    y64 = np.empty(shape, np.float64)
    yb = np.empty(shape, np.uint16)
    rc = lib.o_conv3d_fp8(_ptr(x, ctypes.c_ubyte), _ptr(w, ctypes.c_ubyte), float(sx), float(sw),
                          *args, _ptr(ysum, ctypes.c_double), _ptr(y64, ctypes.c_double),
                          _ptr(yb, ctypes.c_ushort))
    _check(rc)
    return (ysum, y64, yb) if want_sum else (y64, yb)


def conv3d_fp8_points(x: np.ndarray, w: np.ndarray, sx: float, sw: float, idx, stride=1, pad=1,
                      want_sum: bool = False):
    """Selected outputs. ``idx``: flat NCDHW indices into the [N,K,Do,Ho,Wo] output.

    Returns (y64, ybf16) -- or (ysum, y64, ybf16) -- one entry per index.
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint8)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    args = _shape_args(x, w, stride, pad)
    n = idx.size
    ysum = np.empty(n, np.float64) if want_sum else None
    y64 = np.empty(n, np.float64)
    yb = np.empty(n, np.uint16)
    rc = lib.o_conv3d_fp8_points(_ptr(x, ctypes.c_ubyte), _ptr(w, ctypes.c_ubyte), float(sx),
                                 float(sw), *args, _ptr(idx, ctypes.c_longlong), n,
                                 _ptr(ysum, ctypes.c_double), _ptr(y64, ctypes.c_double),
                                 _ptr(yb, ctypes.c_ushort))
    _check(rc)
    return (ysum, y64, yb) if want_sum else (y64, yb)


def _u16(a) -> np.ndarray:
    """bfloat16 bit patterns as a contiguous uint16 array (accepts uint16/int16 arrays)."""
    a = np.asarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


def conv3d_bf16(x, w, stride=1, pad=1):
    """Full convolution of the BF16-input twin. x: uint16 [N,C,D,H,W] bfloat16 bit patterns;
    w: uint16 [K,C,T,R,S]. No scales. Returns (y64, ybf16), each [N,K,Do,Ho,Wo]."""
    lib = _load()
    x, w = _u16(x), _u16(w)
    args = _shape_args(x, w, stride, pad)
    N, _, D, H, W_, K, T, R, S, sd, sh, sww, pd, ph, pw = args
    Do, Ho, Wo = out_dims(D, H, W_, T, R, S, (sd, sh, sww), (pd, ph, pw))
    if min(Do, Ho, Wo) <= 0:
        raise ValueError("oracle: empty output")
    shape = (N, K, Do, Ho, Wo)
    y64 = np.empty(shape, np.float64)
    yb = np.empty(shape, np.uint16)
    rc = lib.o_conv3d_bf16(_ptr(x, ctypes.c_ushort), _ptr(w, ctypes.c_ushort), *args,
                           _ptr(y64, ctypes.c_double), _ptr(yb, ctypes.c_ushort))
    _check(rc)
    return y64, yb


def conv3d_bf16_points(x, w, idx, stride=1, pad=1):
    """Selected outputs of the BF16-input twin (flat NCDHW indices). Returns (y64, ybf16)."""
    lib = _load()
    x, w = _u16(x), _u16(w)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    args = _shape_args(x, w, stride, pad)
    n = idx.size
    y64 = np.empty(n, np.float64)
    yb = np.empty(n, np.uint16)
    rc = lib.o_conv3d_bf16_points(_ptr(x, ctypes.c_ushort), _ptr(w, ctypes.c_ushort), *args,
                                  _ptr(idx, ctypes.c_longlong), n, _ptr(y64, ctypes.c_double),
                                  _ptr(yb, ctypes.c_ushort))
    _check(rc)
    return y64, yb
