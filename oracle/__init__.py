"""CPU oracle for GDN ReplaySSM verify / accept / flush.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only users.  The product path never
imports this package, and this package imports nothing from the product.

The arithmetic lives in ``gdn_oracle.c`` (plain sequential C, fp64); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Each function below follows the same passages as its C counterpart; see the
header comment of ``gdn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, f) for f in ("gdn_oracle.c", "gdn_layer_ops_oracle.c")]
_LIB = os.path.join(_HERE, "_build", "libgdnoracle.so")

BAD_ACCEPT, NO_ROOM, BAD_LEN, BAD_SLOT = 1, 2, 4, 8


class _ConvDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("D", ctypes.c_int), ("W", ctypes.c_int), ("T", ctypes.c_int),
                ("cap", ctypes.c_int), ("n_slot", ctypes.c_int), ("act", ctypes.c_int)]


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
                ("T", ctypes.c_int), ("cap", ctypes.c_int), ("threshold", ctypes.c_int),
                ("n_slot", ctypes.c_int), ("scale", ctypes.c_double), ("fp32_mode", ctypes.c_int),
                ("n_threads", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into one shared library with gcc (no -march flags)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(s)
                                                 for s in _SRCS):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, *_SRCS,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.orc_recur.argtypes = [ctypes.POINTER(_Dims), P, ctypes.c_int,
                                  P, ctypes.c_long, P, ctypes.c_long, P, P, ctypes.c_long,
                                  P, ctypes.c_long, P, ctypes.c_long]
        lib.orc_verify.argtypes = [ctypes.POINTER(_Dims)] + [P] * 14
        lib.orc_accept.argtypes = [ctypes.POINTER(_Dims), P, P, P, P]
        lib.orc_flush.argtypes = [ctypes.POINTER(_Dims)] + [P] * 7 + [ctypes.c_int, P]
        lib.orc_nr_verify.argtypes = [ctypes.POINTER(_Dims)] + [P] * 10
        lib.orc_nr_accept.argtypes = [ctypes.POINTER(_Dims)] + [P] * 5
        for f in (lib.orc_recur, lib.orc_verify, lib.orc_accept, lib.orc_flush, lib.orc_nr_verify,
                  lib.orc_nr_accept):
            f.restype = ctypes.c_int
        CD = ctypes.POINTER(_ConvDims)
        lib.orc_conv_verify.argtypes = [CD] + [P] * 8
        lib.orc_conv_accept.argtypes = [CD] + [P] * 4
        lib.orc_e4m3_decode.argtypes = [ctypes.c_int]
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
        lib.orc_e4m3_encode.restype = ctypes.c_int
        lib.orc_gated_rmsnorm_fp8.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_double,
                                              ctypes.c_double, P, P]
        for f in (lib.orc_conv_verify, lib.orc_conv_accept, lib.orc_gated_rmsnorm_fp8):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


@dataclass
class Dims:
    B: int
    H: int
    dk: int
    dv: int
    T: int
    cap: int
    threshold: int
    n_slot: int
    scale: float
    fp32_mode: bool = False
    n_threads: int = 1

    def c(self) -> _Dims:
        return _Dims(self.B, self.H, self.dk, self.dv, self.T, self.cap, self.threshold,
                     self.n_slot, float(self.scale), int(self.fp32_mode), int(self.n_threads))


def _f64(a, shape=None):
    a = np.asarray(a)
    if a.dtype != np.float64 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("oracle arrays must be C-contiguous float64")
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"shape {a.shape} != {tuple(shape)}")
    return a


def _i32(a, shape=None):
    a = np.asarray(a)
    if a.dtype != np.int32 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("oracle index arrays must be C-contiguous int32")
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"shape {a.shape} != {tuple(shape)}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def recur(d: Dims, S: np.ndarray, k, v, g, beta, q=None):
    """Straight sequential gated delta rule over n tokens; S [dv, dk] updated in place.

    k [n, dk], v [n, dv], g/beta [n]; with q [n, dk] returns outputs [n, dv].
    """
    S = _f64(S, (d.dv, d.dk))          # updated in place: must already be contiguous
    c = lambda a: np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731  (read-only inputs)
    k, v, g, beta = c(k), c(v), c(g), c(beta)
    n = k.shape[0]
    assert k.shape == (n, d.dk) and v.shape == (n, d.dv) and g.shape == (n,) and beta.shape == (n,)
    o = None
    if q is not None:
        q = _f64(np.ascontiguousarray(q, dtype=np.float64), (n, d.dk))
        o = np.zeros((n, d.dv))
    _load().orc_recur(ctypes.byref(d.c()), _p(S), n, _p(k), d.dk, _p(v), d.dv, _p(g), _p(beta), 1,
                      _p(q), d.dk, _p(o), d.dv)
    return o


def verify(d: Dims, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len,
           q, k, v, g, beta, out, status):
    """Outputs of the draft block from checkpoint + committed buffer; stages the
    draft into buf[len:len+T].  Never writes ``state`` or ``buf_len``."""
    H, cap = d.H, d.cap
    args = [_f64(state, (d.n_slot, H, d.dv, d.dk)),
            None if state_idx is None else _i32(state_idx, (d.B,)),
            _f64(buf_k, (d.n_slot, H, cap, d.dk)), _f64(buf_v, (d.n_slot, H, cap, d.dv)),
            _f64(buf_g, (d.n_slot, H, cap)), _f64(buf_beta, (d.n_slot, H, cap)),
            _i32(buf_len, (d.n_slot,)),
            _f64(q, (d.B, d.T, H, d.dk)), _f64(k, (d.B, d.T, H, d.dk)), _f64(v, (d.B, d.T, H, d.dv)),
            _f64(g, (d.B, d.T, H)), _f64(beta, (d.B, d.T, H)), _f64(out, (d.B, d.T, H, d.dv)),
            _i32(status, (1,))]
    return _load().orc_verify(ctypes.byref(d.c()), *[_p(a) for a in args])


def accept(d: Dims, buf_len, state_idx, accepted, status):
    """Commit the first accepted[b] draft tokens: len += p (0 <= p <= T)."""
    args = [_i32(buf_len, (d.n_slot,)), None if state_idx is None else _i32(state_idx, (d.B,)),
            _i32(accepted, (d.B,)), _i32(status, (1,))]
    return _load().orc_accept(ctypes.byref(d.c()), *[_p(a) for a in args])


def flush(d: Dims, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len, force, status):
    """Fold the buffer into the checkpoint for every b with len >= threshold
    (or len > 0 when forced); the state is rounded to fp32 and len reset to 0."""
    H, cap = d.H, d.cap
    args = [_f64(state, (d.n_slot, H, d.dv, d.dk)),
            None if state_idx is None else _i32(state_idx, (d.B,)),
            _f64(buf_k, (d.n_slot, H, cap, d.dk)), _f64(buf_v, (d.n_slot, H, cap, d.dv)),
            _f64(buf_g, (d.n_slot, H, cap)), _f64(buf_beta, (d.n_slot, H, cap)),
            _i32(buf_len, (d.n_slot,))]
    return _load().orc_flush(ctypes.byref(d.c()), *[_p(a) for a in args], int(force),
                             _p(_i32(status, (1,))))


class Layer:
    """One layer's checkpoint, buffer and lengths held by the oracle (fp64)."""

    def __init__(self, d: Dims, init: dict):
        self.d = d
        f = lambda t: np.ascontiguousarray(t.double().numpy())  # noqa: E731  exact widening
        self.state = f(init["state"])
        self.state_idx = np.ascontiguousarray(init["state_idx"].numpy().astype(np.int32))
        self.buf_k, self.buf_v = f(init["buf_k"]), f(init["buf_v"])
        self.buf_g, self.buf_beta = f(init["buf_g"]), f(init["buf_beta"])
        self.buf_len = np.ascontiguousarray(init["buf_len"].numpy().astype(np.int32))
        self.status = np.zeros(1, np.int32)

    def verify(self, blk: dict) -> np.ndarray:
        d = self.d
        f = lambda t: np.ascontiguousarray(t.double().numpy())  # noqa: E731
        out = np.zeros((d.B, d.T, d.H, d.dv))
        verify(d, self.state, self.state_idx, self.buf_k, self.buf_v, self.buf_g, self.buf_beta,
               self.buf_len, f(blk["q"]), f(blk["k"]), f(blk["v"]), f(blk["g"]), f(blk["beta"]),
               out, self.status)
        return out

    def accept(self, accepted):
        acc = np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
        accept(self.d, self.buf_len, self.state_idx, acc, self.status)

    def flush(self, force: bool = False):
        flush(self.d, self.state, self.state_idx, self.buf_k, self.buf_v, self.buf_g,
              self.buf_beta, self.buf_len, force, self.status)


# ------------------------------------------------- non-replay baseline
def nr_verify(d: Dims, state, state_idx, q, k, v, g, beta, out, snap, status):
    """The baseline without a buffer: outputs of the draft block from the current
    state, and the state after every draft token stored (binary32) in
    snap [B, H, T, dv, dk].  Never writes ``state``."""
    H = d.H
    args = [_f64(state, (d.n_slot, H, d.dv, d.dk)),
            None if state_idx is None else _i32(state_idx, (d.B,)),
            _f64(q, (d.B, d.T, H, d.dk)), _f64(k, (d.B, d.T, H, d.dk)), _f64(v, (d.B, d.T, H, d.dv)),
            _f64(g, (d.B, d.T, H)), _f64(beta, (d.B, d.T, H)), _f64(out, (d.B, d.T, H, d.dv)),
            _f64(snap, (d.B, H, d.T, d.dv, d.dk)), _i32(status, (1,))]
    return _load().orc_nr_verify(ctypes.byref(d.c()), *[_p(a) for a in args])


def nr_accept(d: Dims, state, state_idx, snap, accepted, status):
    """Restore by copy: state = snap[b, :, p - 1] for p in [1, T]; p = 0 keeps it."""
    args = [_f64(state, (d.n_slot, d.H, d.dv, d.dk)),
            None if state_idx is None else _i32(state_idx, (d.B,)),
            _f64(snap, (d.B, d.H, d.T, d.dv, d.dk)), _i32(accepted, (d.B,)), _i32(status, (1,))]
    return _load().orc_nr_accept(ctypes.byref(d.c()), *[_p(a) for a in args])


class NonReplayLayer:
    """One layer of the non-replay baseline held by the oracle: the current state
    and the snapshots of the last verify."""

    def __init__(self, d: Dims, state, state_idx):
        self.d = d
        self.state = np.array(state, dtype=np.float64, order="C")          # a copy: the layer owns it
        self.state_idx = None if state_idx is None else np.array(state_idx, dtype=np.int32, order="C")
        self.snap = np.zeros((d.B, d.H, d.T, d.dv, d.dk))
        self.status = np.zeros(1, np.int32)

    def verify(self, blk: dict) -> np.ndarray:
        d = self.d
        f = lambda t: np.ascontiguousarray(np.asarray(t, dtype=np.float64))  # noqa: E731
        out = np.zeros((d.B, d.T, d.H, d.dv))
        nr_verify(d, self.state, self.state_idx, f(blk["q"]), f(blk["k"]), f(blk["v"]), f(blk["g"]),
                  f(blk["beta"]), out, self.snap, self.status)
        return out

    def accept(self, accepted):
        acc = np.ascontiguousarray(np.asarray(accepted, dtype=np.int32))
        nr_accept(self.d, self.state, self.state_idx, self.snap, acc, self.status)


# ------------------------------------------------- causal convolution with rollback
@dataclass
class ConvDims:
    B: int
    D: int
    W: int
    T: int
    cap: int
    n_slot: int
    act: int = 1          # 0 identity, 1 SiLU

    def c(self) -> _ConvDims:
        return _ConvDims(self.B, self.D, self.W, self.T, self.cap, self.n_slot, self.act)


def conv_verify(d: ConvDims, ring, pos, state_idx, x, w, bias, y, status):
    """Draft outputs of the causal convolution from the committed window (the W-1
    ring positions before pos) and the draft x; stages x at pos .. pos+T-1 (mod cap)."""
    args = [_f64(ring, (d.n_slot, d.cap, d.D)), _i32(pos, (d.n_slot,)),
            None if state_idx is None else _i32(state_idx, (d.B,)),
            _f64(x, (d.B, d.T, d.D)), _f64(w, (d.D, d.W)),
            None if bias is None else _f64(bias, (d.D,)), _f64(y, (d.B, d.T, d.D)),
            _i32(status, (1,))]
    return _load().orc_conv_verify(ctypes.byref(d.c()), *[_p(a) for a in args])


def conv_accept(d: ConvDims, pos, state_idx, accepted, status):
    """pos += p (mod cap) for 0 <= p <= T: the accepted prefix joins the window."""
    args = [_i32(pos, (d.n_slot,)), None if state_idx is None else _i32(state_idx, (d.B,)),
            _i32(accepted, (d.B,)), _i32(status, (1,))]
    return _load().orc_conv_accept(ctypes.byref(d.c()), *[_p(a) for a in args])


class ConvLayer:
    """One layer's convolution ring and write positions held by the oracle (fp64)."""

    def __init__(self, d: ConvDims, init: dict):
        self.d = d
        f = lambda t: np.ascontiguousarray(t.double().numpy())  # noqa: E731  exact widening
        self.ring = f(init["ring"])
        self.pos = np.ascontiguousarray(init["pos"].numpy().astype(np.int32))
        self.state_idx = np.ascontiguousarray(init["state_idx"].numpy().astype(np.int32))
        self.w = f(init["weight"])
        self.bias = None if init.get("bias") is None else f(init["bias"])
        self.status = np.zeros(1, np.int32)

    def verify(self, x) -> np.ndarray:
        d = self.d
        y = np.zeros((d.B, d.T, d.D))
        conv_verify(d, self.ring, self.pos, self.state_idx,
                    np.ascontiguousarray(x.double().numpy()), self.w, self.bias, y, self.status)
        return y

    def accept(self, accepted):
        conv_accept(self.d, self.pos, self.state_idx,
                    np.ascontiguousarray(np.asarray(accepted, dtype=np.int32)), self.status)


# ------------------------------------------------------ gated RMSNorm + E4M3 codes
def e4m3_decode(code: int) -> float:
    """Value of an E4M3 code (bias 7, subnormals, NaN at exponent 15 / mantissa 7)."""
    return _load().orc_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    """E4M3 code of x: round to nearest, ties to even, saturate at +-448."""
    return _load().orc_e4m3_encode(float(x))


def gated_rmsnorm_fp8(o, z, w, eps: float, inv_scale: float):
    """o, z [rows, d]; w [d].  Returns (codes uint8 [rows, d], y * inv_scale fp64)."""
    o = np.ascontiguousarray(o, dtype=np.float64)
    z = np.ascontiguousarray(z, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, d = o.shape
    assert z.shape == (rows, d) and w.shape == (d,)
    q = np.zeros((rows, d), np.uint8)
    yq = np.zeros((rows, d))
    _load().orc_gated_rmsnorm_fp8(rows, d, _p(o), _p(z), _p(w), float(eps), float(inv_scale),
                                  _p(q), _p(yq))
    return q, yq
