"""Shared test plumbing: run the CUDA library and the CPU oracle side by side
on the same seeded inputs and compare them.

Tolerance (floating point): per tensor and per (layer, step),
    max |gpu - ref| <= 2e-3 * max |ref| + 1e-5
with the fp64 oracle as ref.  Integer state (buffer lengths, status words)
and the bytes copied into the buffer must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

RTOL_MAX, ATOL = 2e-3, 1e-5

# max|gpu - ref| / max|ref| of every compared tensor, appended by assert_close as
# (name, ratio); tests that track drift over many steps read it back
DRIFT = []


def gpu_dims(wl: synth.Workload, B=None, n_slot=None):
    import speculative_decode_recurrent_gb300 as lib
    B = wl.B if B is None else B
    return lib.Dims(B=B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.cap, threshold=wl.threshold,
                    n_slot=(B + max(1, B // 4)) if n_slot is None else n_slot,
                    in_dtype=lib.DTYPE_BF16 if wl.in_dtype == "bf16" else lib.DTYPE_F32,
                    scale=wl.scale)


def oracle_dims(wl: synth.Workload, B=None, n_slot=None, threads=8):
    B = wl.B if B is None else B
    return oracle.Dims(B=B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.cap, threshold=wl.threshold,
                       n_slot=(B + max(1, B // 4)) if n_slot is None else n_slot,
                       scale=wl.scale, n_threads=threads)


def assert_close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    mref = float(np.max(np.abs(ref))) if ref.size else 0.0
    bound = RTOL_MAX * mref + ATOL
    DRIFT.append((name, err / mref if mref > 0 else 0.0))
    assert err <= bound, f"{name}: max|d|={err:.3e} > bound {bound:.3e}"
    return err, bound


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


class Pair:
    """GPU layer and oracle layer built from the same seeded initial state."""

    def __init__(self, wl: synth.Workload, layer=0, B=None, device="cuda"):
        import speculative_decode_recurrent_gb300 as lib
        self.wl, self.layer = wl, layer
        self.B = wl.B if B is None else B
        init = synth.initial_layer(wl, layer, B=self.B)
        self.gd = gpu_dims(wl, self.B)
        self.od = oracle_dims(wl, self.B)
        self.gpu = lib.ReplayLayer(self.gd, init, device)
        self.orc = oracle.Layer(self.od, init)
        self.device = device

    def block(self, step):
        return synth.draft_block(self.wl, self.layer, step, B=self.B)

    def step(self, step, force=None, check=True, accepted=None):
        """One verify -> accept -> flush on both sides; compares out, lengths,
        status, and (after the flush) state and buffer."""
        wl = self.wl
        blk = self.block(step)
        acc = blk["accepted"] if accepted is None else torch.as_tensor(accepted, dtype=torch.int32)
        force = wl.forced_flush if force is None else force
        dev = {n: blk[n].to(self.device) for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty(self.B, wl.T, wl.H, wl.dv, dtype=torch.float32, device=self.device)
        self.gpu.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
        o_ref = self.orc.verify(blk)
        self.gpu.accept(acc.to(self.device))
        self.orc.accept(acc.numpy())
        self.gpu.flush(force=force)
        self.orc.flush(force=force)
        torch.cuda.synchronize()
        if check:
            self.compare(out, o_ref, step)
        return out, o_ref, acc

    def fused_step(self, step, check=True, accepted=None):
        """One verify_fold -> accept_fold on the GPU against the oracle's
        flush (threshold) -> verify -> accept, which it must equal."""
        wl = self.wl
        blk = self.block(step)
        acc = blk["accepted"] if accepted is None else torch.as_tensor(accepted, dtype=torch.int32)
        dev = {n: blk[n].to(self.device) for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty(self.B, wl.T, wl.H, wl.dv, dtype=torch.float32, device=self.device)
        self.gpu.verify_fold(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
        self.gpu.accept_fold(acc.to(self.device))
        self.orc.flush(force=False)
        o_ref = self.orc.verify(blk)
        self.orc.accept(acc.numpy())
        torch.cuda.synchronize()
        if check:
            self.compare(out, o_ref, step)
        return out, o_ref, acc

    def compare(self, out, o_ref, step):
        t = self.gpu.t
        tag = f"layer{self.layer}/step{step}"
        np.testing.assert_array_equal(t["buf_len"].cpu().numpy(), self.orc.buf_len, err_msg=tag)
        assert int(self.gpu.status.item()) == int(self.orc.status[0]), tag
        assert_close(f"out {tag}", to_np(out), o_ref)
        assert_close(f"state {tag}", to_np(t["state"]), self.orc.state)
        # the buffer holds copies of inputs: bit-exact
        np.testing.assert_array_equal(to_np(t["buf_k"]), self.orc.buf_k, err_msg=tag)
        np.testing.assert_array_equal(to_np(t["buf_v"]), self.orc.buf_v, err_msg=tag)
        np.testing.assert_array_equal(to_np(t["buf_g"]), self.orc.buf_g, err_msg=tag)
        np.testing.assert_array_equal(to_np(t["buf_beta"]), self.orc.buf_beta, err_msg=tag)


# ---------------------------------------------------------- rounded outputs
def round_bf16(x: np.ndarray) -> np.ndarray:
    """bf16 rounding (nearest, ties to even) of fp64 values.  x is first rounded to
    fp32, which moves it by at most 2^-24 relative: only values within that of a bf16
    midpoint can round differently from a single rounding, and every caller widens its
    comparison by far more than that."""
    r32 = np.asarray(x, np.float64).astype(np.float32)
    bits = r32.view(np.uint32)
    down = (bits & np.uint32(0xFFFF0000))
    up = down + np.uint32(0x10000)
    dv, uv = down.view(np.float32).astype(np.float64), up.view(np.float32).astype(np.float64)
    mid = (dv + uv) / 2
    mag = np.abs(r32.astype(np.float64))
    pick_up = (mag > np.abs(mid)) | ((mag == np.abs(mid)) & ((down >> np.uint32(16)) & np.uint32(1)).astype(bool))
    return np.where(pick_up, uv, dv)


def assert_bf16_rounding(name, got_bf16: torch.Tensor, ref: np.ndarray, band: np.ndarray):
    """got is the bf16 rounding of a value within `band` (absolute, per element) of the
    fp64 reference, so it must lie between the roundings of ref - band and ref + band
    (a single value wherever the band does not reach a rounding midpoint).  Returns the
    count of elements where more than one value is possible."""
    got = got_bf16.float().cpu().double().numpy().reshape(ref.shape)
    lo, hi = round_bf16(ref - band), round_bf16(ref + band)
    ok = (got >= lo) & (got <= hi)
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (f"{name}: {bad.size} elements differ, first at {bad[0]}: got {got.flat[bad[0]]}, "
                           f"ref {ref.flat[bad[0]]}, allowed [{lo.flat[bad[0]]}, {hi.flat[bad[0]]}]")
    return int((lo != hi).sum())


def _e4m3_round(v: np.ndarray, table: np.ndarray) -> np.ndarray:
    """E4M3 code of fp64 values (nearest, ties to the even code, saturated at +-448)
    by search in the table of the 127 non-negative finite values."""
    pos = table[:0x7F]                                  # codes 0x00 .. 0x7E, increasing
    mag = np.minimum(np.abs(v), 448.0)
    i = np.clip(np.searchsorted(pos, mag), 1, 0x7E)     # pos[i-1] < mag <= pos[i]
    lo, hi = pos[i - 1], pos[i]
    mid = (lo + hi) / 2
    code = np.where(mag > mid, i, np.where(mag < mid, i - 1, np.where(i % 2 == 0, i, i - 1)))
    code = np.where(mag <= pos[0], 0, code)
    return code | np.where(np.signbit(v), 0x80, 0)


def assert_e4m3_codes(name, got_codes: np.ndarray, ref_codes: np.ndarray, ref_value: np.ndarray,
                      rel_band: float):
    """E4M3 codes of values within rel_band (relative) of the fp64 ones: each code must be
    the oracle's, or, where that band reaches a rounding midpoint, a code between the
    roundings of the band's ends.  Returns the count of elements with more than one
    possible code."""
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    got = got_codes.reshape(-1).astype(np.int64)
    rc = ref_codes.reshape(-1).astype(np.int64)
    v = ref_value.reshape(-1)
    lo = _e4m3_round(v - rel_band * np.abs(v), table)
    hi = _e4m3_round(v + rel_band * np.abs(v), table)
    assert np.array_equal(_e4m3_round(v, table), rc), f"{name}: the oracle's codes are not its values' rounding"
    gv, lv, hv = table[got], table[lo], table[hi]
    ok = (lo == hi) & (got == rc) | (lo != hi) & (gv >= np.minimum(lv, hv)) & (gv <= np.maximum(lv, hv))
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (f"{name}: {bad.size} codes differ, first at {bad[0]}: got {got[bad[0]]:#x}, "
                           f"ref {rc[bad[0]]:#x} (value {v[bad[0]]!r})")
    return int((lo != hi).sum())
