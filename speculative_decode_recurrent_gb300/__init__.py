"""Python binding of libgdnreplay (ReplaySSM verify / accept / flush of Gated
DeltaNet state on sm_103a).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``csrc/gdn_replay.cu`` behind the C ABI declared in ``include/gdnreplay.h``.
PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the shared library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = ["Dims", "GdnError", "load", "gdn_replay_verify", "gdn_replay_accept",
           "gdn_replay_flush", "gdn_replay_verify_fold", "gdn_replay_accept_fold",
           "gdn_replay_kernel_family", "gdn_replay_strerror", "STATUS_BAD_ACCEPT",
           "STATUS_NO_ROOM", "STATUS_BAD_LEN", "STATUS_BAD_SLOT", "STATUS_TIMEOUT",
           "STATUS_DRAIN", "FLAG_TEST_EXPIRE", "FAMILY_TCGEN05", "FAMILY_PERTOKEN", "DTYPE_BF16",
           "DTYPE_F32", "ReplayLayer", "ConvDims", "gdn_conv_verify", "gdn_conv_accept",
           "gdn_gated_rmsnorm_fp8", "ConvLayer", "CONV_ACT_NONE", "CONV_ACT_SILU",
           "gdn_nonreplay_verify", "gdn_nonreplay_accept", "NonReplayLayer"]

DTYPE_BF16, DTYPE_F32 = 0, 1
STATUS_BAD_ACCEPT, STATUS_NO_ROOM, STATUS_BAD_LEN, STATUS_BAD_SLOT, STATUS_TIMEOUT = 1, 2, 4, 8, 16
STATUS_DRAIN = 32
FLAG_TEST_EXPIRE = 1
FAMILY_TCGEN05, FAMILY_PERTOKEN = 1, 2
FAMILY_NAMES = {FAMILY_TCGEN05: "tcgen05", FAMILY_PERTOKEN: "per-token"}
CONV_ACT_NONE, CONV_ACT_SILU = 0, 1
_TORCH_IN = {DTYPE_BF16: torch.bfloat16, DTYPE_F32: torch.float32}


class Dims(ctypes.Structure):
    """Mirror of ``gdn_replay_dims``."""
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("T", ctypes.c_int32), ("cap", ctypes.c_int32),
                ("threshold", ctypes.c_int32), ("n_slot", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("flags", ctypes.c_int32)]

    def __repr__(self):
        return "Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class ConvDims(ctypes.Structure):
    """Mirror of ``gdn_conv_dims`` (include/gdnlayer.h)."""
    _fields_ = [("B", ctypes.c_int32), ("D", ctypes.c_int32), ("W", ctypes.c_int32),
                ("T", ctypes.c_int32), ("cap", ctypes.c_int32), ("n_slot", ctypes.c_int32),
                ("act", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]

    def __repr__(self):
        return "ConvDims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class GdnError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({gdn_replay_strerror(code)})")
        self.code = code


_lib = None


def load(rebuild: bool = False) -> ctypes.CDLL:
    """Build (if stale) and load libgdnreplay.so; raises if that is impossible."""
    global _lib
    if _lib is None or rebuild:
        path = _build.build(force=rebuild)
        if not os.path.exists(path):
            raise RuntimeError(f"libgdnreplay not found at {path}")
        lib = ctypes.CDLL(path)
        P, I = ctypes.c_void_p, ctypes.c_int32
        D = ctypes.POINTER(Dims)
        lib.gdn_replay_verify.argtypes = [D] + [P] * 15
        lib.gdn_replay_accept.argtypes = [D, P, P, P, P, P]
        lib.gdn_replay_flush.argtypes = [D] + [P] * 7 + [I, P, P]
        lib.gdn_replay_verify_fold.argtypes = [D] + [P] * 15
        lib.gdn_replay_accept_fold.argtypes = [D, P, P, P, P, P]
        lib.gdn_replay_strerror.argtypes = [ctypes.c_int]
        lib.gdn_replay_strerror.restype = ctypes.c_char_p
        lib.gdn_replay_version.argtypes = []
        lib.gdn_replay_kernel_family.argtypes = [D]
        CD = ctypes.POINTER(ConvDims)
        lib.gdn_conv_verify.argtypes = [CD] + [P] * 9
        lib.gdn_conv_accept.argtypes = [CD, P, P, P, P, P]
        lib.gdn_gated_rmsnorm_fp8.argtypes = [I, I, P, P, I, P, ctypes.c_float, ctypes.c_float, P, P]
        lib.gdn_nonreplay_verify.argtypes = [D] + [P] * 11
        lib.gdn_nonreplay_accept.argtypes = [D] + [P] * 6
        for f in (lib.gdn_conv_verify, lib.gdn_conv_accept, lib.gdn_gated_rmsnorm_fp8,
                  lib.gdn_nonreplay_verify, lib.gdn_nonreplay_accept):
            f.restype = ctypes.c_int
        for f in (lib.gdn_replay_verify, lib.gdn_replay_accept, lib.gdn_replay_flush,
                  lib.gdn_replay_verify_fold, lib.gdn_replay_accept_fold, lib.gdn_replay_version,
                  lib.gdn_replay_kernel_family):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def gdn_replay_strerror(code: int) -> str:
    return load().gdn_replay_strerror(int(code)).decode()


def gdn_replay_kernel_family(d: Dims) -> int:
    """FAMILY_TCGEN05 or FAMILY_PERTOKEN: the kernels calls with dims d launch."""
    rc = load().gdn_replay_kernel_family(ctypes.byref(d))
    _check("gdn_replay_kernel_family", rc if rc < 0 else 0)
    return rc


def _sizes(d: Dims) -> dict:
    """Elements of each argument for dims d (the dense layouts of gdnreplay.h)."""
    B, H, dk, dv, T, cap, n = d.B, d.H, d.dk, d.dv, d.T, d.cap, d.n_slot
    return {"state": n * H * dv * dk, "state_idx": B, "buf_k": n * H * cap * dk,
            "buf_v": n * H * cap * dv, "buf_g": n * H * cap, "buf_beta": n * H * cap,
            "buf_len": n, "q": B * T * H * dk, "k": B * T * H * dk, "v": B * T * H * dv,
            "g": B * T * H, "beta": B * T * H, "out": B * T * H * dv, "accepted": B, "status": 1}


def _check_sizes(d: Dims, **tensors):
    """Every tensor must hold at least what the kernels read or write for dims d."""
    need = _sizes(d)
    for name, t in tensors.items():
        if isinstance(t, torch.Tensor) and t.numel() < need[name]:
            raise ValueError(f"{name}: needs at least {need[name]} elements for {d}, got {t.numel()}")


def _ptr(t, dtype=None, name=""):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise GdnError(fn, rc)


def gdn_replay_verify(d: Dims, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len,
                      q, k, v, g, beta, out, status, stream=None):
    tin = _TORCH_IN.get(d.in_dtype)
    f32, i32 = torch.float32, torch.int32
    _check_sizes(d, state=state, state_idx=state_idx, buf_k=buf_k, buf_v=buf_v, buf_g=buf_g,
                 buf_beta=buf_beta, buf_len=buf_len, q=q, k=k, v=v, g=g, beta=beta, out=out,
                 status=status)
    rc = load().gdn_replay_verify(
        ctypes.byref(d), _ptr(state, f32, "state"), _ptr(state_idx, i32, "state_idx"),
        _ptr(buf_k, tin, "buf_k"), _ptr(buf_v, tin, "buf_v"), _ptr(buf_g, f32, "buf_g"),
        _ptr(buf_beta, f32, "buf_beta"), _ptr(buf_len, i32, "buf_len"),
        _ptr(q, tin, "q"), _ptr(k, tin, "k"), _ptr(v, tin, "v"), _ptr(g, f32, "g"),
        _ptr(beta, f32, "beta"), _ptr(out, f32, "out"), _ptr(status, i32, "status"),
        _stream(stream))
    _check("gdn_replay_verify", rc)


def gdn_replay_verify_fold(d: Dims, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len,
                           q, k, v, g, beta, out, status, stream=None):
    tin = _TORCH_IN.get(d.in_dtype)
    f32, i32 = torch.float32, torch.int32
    _check_sizes(d, state=state, state_idx=state_idx, buf_k=buf_k, buf_v=buf_v, buf_g=buf_g,
                 buf_beta=buf_beta, buf_len=buf_len, q=q, k=k, v=v, g=g, beta=beta, out=out,
                 status=status)
    rc = load().gdn_replay_verify_fold(
        ctypes.byref(d), _ptr(state, f32, "state"), _ptr(state_idx, i32, "state_idx"),
        _ptr(buf_k, tin, "buf_k"), _ptr(buf_v, tin, "buf_v"), _ptr(buf_g, f32, "buf_g"),
        _ptr(buf_beta, f32, "buf_beta"), _ptr(buf_len, i32, "buf_len"),
        _ptr(q, tin, "q"), _ptr(k, tin, "k"), _ptr(v, tin, "v"), _ptr(g, f32, "g"),
        _ptr(beta, f32, "beta"), _ptr(out, f32, "out"), _ptr(status, i32, "status"),
        _stream(stream))
    _check("gdn_replay_verify_fold", rc)


def gdn_replay_accept_fold(d: Dims, buf_len, state_idx, accepted, status, stream=None):
    i32 = torch.int32
    _check_sizes(d, buf_len=buf_len, state_idx=state_idx, accepted=accepted, status=status)
    rc = load().gdn_replay_accept_fold(ctypes.byref(d), _ptr(buf_len, i32, "buf_len"),
                                       _ptr(state_idx, i32, "state_idx"),
                                       _ptr(accepted, i32, "accepted"), _ptr(status, i32, "status"),
                                       _stream(stream))
    _check("gdn_replay_accept_fold", rc)


def gdn_replay_accept(d: Dims, buf_len, state_idx, accepted, status, stream=None):
    i32 = torch.int32
    _check_sizes(d, buf_len=buf_len, state_idx=state_idx, accepted=accepted, status=status)
    rc = load().gdn_replay_accept(ctypes.byref(d), _ptr(buf_len, i32, "buf_len"),
                                  _ptr(state_idx, i32, "state_idx"),
                                  _ptr(accepted, i32, "accepted"), _ptr(status, i32, "status"),
                                  _stream(stream))
    _check("gdn_replay_accept", rc)


def gdn_replay_flush(d: Dims, state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len, force,
                     status, stream=None):
    tin = _TORCH_IN.get(d.in_dtype)
    f32, i32 = torch.float32, torch.int32
    _check_sizes(d, state=state, state_idx=state_idx, buf_k=buf_k, buf_v=buf_v, buf_g=buf_g,
                 buf_beta=buf_beta, buf_len=buf_len, status=status)
    rc = load().gdn_replay_flush(
        ctypes.byref(d), _ptr(state, f32, "state"), _ptr(state_idx, i32, "state_idx"),
        _ptr(buf_k, tin, "buf_k"), _ptr(buf_v, tin, "buf_v"), _ptr(buf_g, f32, "buf_g"),
        _ptr(buf_beta, f32, "buf_beta"), _ptr(buf_len, i32, "buf_len"), int(bool(force)),
        _ptr(status, i32, "status"), _stream(stream))
    _check("gdn_replay_flush", rc)


class ReplayLayer:
    """Device-resident checkpoint, buffer and lengths of one GDN layer.

    ``init`` is a dict of CPU tensors with the layouts of ``include/gdnreplay.h``
    (state, state_idx, buf_k, buf_v, buf_g, buf_beta, buf_len); they are copied
    to ``device`` once.  A state_idx of None is the identity map (sequence b owns
    slot b).  The methods enqueue the library calls.
    """

    def __init__(self, dims: Dims, init: dict, device="cuda"):
        self.d = dims
        self.t = {n: None if init[n] is None else init[n].to(device).contiguous() for n in
                  ("state", "state_idx", "buf_k", "buf_v", "buf_g", "buf_beta", "buf_len")}
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def verify(self, q, k, v, g, beta, out, stream=None):
        t = self.t
        gdn_replay_verify(self.d, t["state"], t["state_idx"], t["buf_k"], t["buf_v"], t["buf_g"],
                          t["buf_beta"], t["buf_len"], q, k, v, g, beta, out, self.status, stream)

    def accept(self, accepted, stream=None):
        gdn_replay_accept(self.d, self.t["buf_len"], self.t["state_idx"], accepted, self.status,
                          stream)

    def flush(self, force=False, stream=None):
        t = self.t
        gdn_replay_flush(self.d, t["state"], t["state_idx"], t["buf_k"], t["buf_v"], t["buf_g"],
                         t["buf_beta"], t["buf_len"], force, self.status, stream)

    def verify_fold(self, q, k, v, g, beta, out, stream=None):
        t = self.t
        gdn_replay_verify_fold(self.d, t["state"], t["state_idx"], t["buf_k"], t["buf_v"],
                               t["buf_g"], t["buf_beta"], t["buf_len"], q, k, v, g, beta, out,
                               self.status, stream)

    def accept_fold(self, accepted, stream=None):
        gdn_replay_accept_fold(self.d, self.t["buf_len"], self.t["state_idx"], accepted,
                               self.status, stream)


# ---------------------------------------------------------- non-replay baseline
def _check_nr_sizes(d: Dims, **tensors):
    B, H, dk, dv, T, n = d.B, d.H, d.dk, d.dv, d.T, d.n_slot
    need = {"state": n * H * dv * dk, "state_idx": B, "q": B * T * H * dk, "k": B * T * H * dk,
            "v": B * T * H * dv, "g": B * T * H, "beta": B * T * H, "out": B * T * H * dv,
            "snap": B * H * T * dv * dk, "accepted": B, "status": 1}
    for name, t in tensors.items():
        if isinstance(t, torch.Tensor) and t.numel() < need[name]:
            raise ValueError(f"{name}: needs at least {need[name]} elements for {d}, got {t.numel()}")


def gdn_nonreplay_verify(d: Dims, state, state_idx, q, k, v, g, beta, out, snap, status, stream=None):
    """The baseline without a buffer (include/gdnnonreplay.h): outputs of the draft
    block from the current state and the state after every draft token in ``snap``."""
    tin = _TORCH_IN.get(d.in_dtype)
    f32, i32 = torch.float32, torch.int32
    _check_nr_sizes(d, state=state, state_idx=state_idx, q=q, k=k, v=v, g=g, beta=beta, out=out,
                    snap=snap, status=status)
    rc = load().gdn_nonreplay_verify(
        ctypes.byref(d), _ptr(state, f32, "state"), _ptr(state_idx, i32, "state_idx"),
        _ptr(q, tin, "q"), _ptr(k, tin, "k"), _ptr(v, tin, "v"), _ptr(g, f32, "g"),
        _ptr(beta, f32, "beta"), _ptr(out, f32, "out"), _ptr(snap, f32, "snap"),
        _ptr(status, i32, "status"), _stream(stream))
    _check("gdn_nonreplay_verify", rc)


def gdn_nonreplay_accept(d: Dims, state, state_idx, snap, accepted, status, stream=None):
    """Restore by copy: the state after the accepted prefix (snapshot p - 1)."""
    f32, i32 = torch.float32, torch.int32
    _check_nr_sizes(d, state=state, state_idx=state_idx, snap=snap, accepted=accepted, status=status)
    rc = load().gdn_nonreplay_accept(
        ctypes.byref(d), _ptr(state, f32, "state"), _ptr(state_idx, i32, "state_idx"),
        _ptr(snap, f32, "snap"), _ptr(accepted, i32, "accepted"), _ptr(status, i32, "status"),
        _stream(stream))
    _check("gdn_nonreplay_accept", rc)


class NonReplayLayer:
    """Device-resident state of one GDN layer under the non-replay baseline, with
    the snapshot area its verify writes (B x H x T states).  ``snap`` may be shared
    between layers that are stepped one after the other."""

    def __init__(self, dims: Dims, state, state_idx, device="cuda", snap=None):
        self.d = dims
        self.state = state.to(device).contiguous()
        self.state_idx = None if state_idx is None else state_idx.to(device).contiguous()
        n = dims.B * dims.H * dims.T * dims.dv * dims.dk
        self.snap = torch.empty(n, dtype=torch.float32, device=device) if snap is None else snap
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def verify(self, q, k, v, g, beta, out, stream=None):
        gdn_nonreplay_verify(self.d, self.state, self.state_idx, q, k, v, g, beta, out, self.snap,
                             self.status, stream)

    def accept(self, accepted, stream=None):
        gdn_nonreplay_accept(self.d, self.state, self.state_idx, self.snap, accepted, self.status,
                             stream)


# ------------------------------------------------ causal convolution with rollback
def _conv_sizes(d: ConvDims) -> dict:
    return {"ring": d.n_slot * d.cap * d.D, "ring_pos": d.n_slot, "state_idx": d.B,
            "x": d.B * d.T * d.D, "weight": d.D * d.W, "bias": d.D, "y": d.B * d.T * d.D,
            "accepted": d.B, "status": 1}


def _check_conv_sizes(d: ConvDims, **tensors):
    need = _conv_sizes(d)
    for name, t in tensors.items():
        if isinstance(t, torch.Tensor) and t.numel() < need[name]:
            raise ValueError(f"{name}: needs at least {need[name]} elements for {d}, got {t.numel()}")


def gdn_conv_verify(d: ConvDims, ring, ring_pos, state_idx, x, weight, bias, y, status, stream=None):
    tin, tout = _TORCH_IN.get(d.in_dtype), _TORCH_IN.get(d.out_dtype)
    f32, i32 = torch.float32, torch.int32
    _check_conv_sizes(d, ring=ring, ring_pos=ring_pos, state_idx=state_idx, x=x, weight=weight,
                      bias=bias, y=y, status=status)
    rc = load().gdn_conv_verify(
        ctypes.byref(d), _ptr(ring, tin, "ring"), _ptr(ring_pos, i32, "ring_pos"),
        _ptr(state_idx, i32, "state_idx"), _ptr(x, tin, "x"), _ptr(weight, f32, "weight"),
        _ptr(bias, f32, "bias"), _ptr(y, tout, "y"), _ptr(status, i32, "status"), _stream(stream))
    _check("gdn_conv_verify", rc)


def gdn_conv_accept(d: ConvDims, ring_pos, state_idx, accepted, status, stream=None):
    i32 = torch.int32
    _check_conv_sizes(d, ring_pos=ring_pos, state_idx=state_idx, accepted=accepted, status=status)
    rc = load().gdn_conv_accept(ctypes.byref(d), _ptr(ring_pos, i32, "ring_pos"),
                                _ptr(state_idx, i32, "state_idx"), _ptr(accepted, i32, "accepted"),
                                _ptr(status, i32, "status"), _stream(stream))
    _check("gdn_conv_accept", rc)


class ConvLayer:
    """Device-resident convolution ring, write positions, weight and bias of one
    layer (``init``: CPU tensors ring, pos, state_idx, weight, bias; a state_idx of
    None is the identity map)."""

    def __init__(self, dims: ConvDims, init: dict, device="cuda"):
        self.d = dims
        self.t = {n: None if init[n] is None else init[n].to(device).contiguous()
                  for n in ("ring", "pos", "state_idx", "weight")}
        self.t["bias"] = None if init.get("bias") is None else init["bias"].to(device).contiguous()
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def verify(self, x, y, stream=None):
        t = self.t
        gdn_conv_verify(self.d, t["ring"], t["pos"], t["state_idx"], x, t["weight"], t["bias"], y,
                        self.status, stream)

    def accept(self, accepted, stream=None):
        gdn_conv_accept(self.d, self.t["pos"], self.t["state_idx"], accepted, self.status, stream)


# ---------------------------------------------------- gated RMSNorm + E4M3 codes
def gdn_gated_rmsnorm_fp8(o, z, weight, eps: float, inv_scale: float, q, stream=None):
    """o fp32 [rows, d] (any shape whose last dim is d), z bf16/fp32 like o, weight fp32 [d],
    q uint8 like o (E4M3 codes)."""
    d = o.shape[-1]
    rows = o.numel() // d if d else 0
    if z.numel() != o.numel() or q.numel() != o.numel() or weight.numel() != d:
        raise ValueError("o, z and q must have the same number of elements; weight must have d")
    zt = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}.get(z.dtype)
    if zt is None:
        raise TypeError(f"z: expected bfloat16 or float32, got {z.dtype}")
    rc = load().gdn_gated_rmsnorm_fp8(rows, d, _ptr(o, torch.float32, "o"), _ptr(z, None, "z"), zt,
                                      _ptr(weight, torch.float32, "weight"), float(eps),
                                      float(inv_scale), _ptr(q, torch.uint8, "q"), _stream(stream))
    _check("gdn_gated_rmsnorm_fp8", rc)
