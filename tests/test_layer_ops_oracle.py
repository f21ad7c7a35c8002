"""Pins for the oracle of the two GDN layer steps either side of the recurrence
("The inference stack behind OCRia", section "Avoiding unnecessary memory
transfers": a faster causal convolution for the GDN layers, and gated RMSNorm
followed by FP8 quantisation).  Each test checks the oracle against something other
than itself: a library routine (torch's conv1d and float8_e4m3fn cast), the format
definition of E4M3 ("Inference Engineering", chapter 5, number formats), closed
forms, a replay of the committed stream from scratch, and hand-worked examples.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layer_ops_hand_examples.txt")


def _golden():
    cases, cur = {}, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "case":
            cur = {}
            cases[rest[0]] = cur
        elif key == "end":
            cur = None
        else:
            cur[key] = rest
    return cases


# ----------------------------------------------------------- causal convolution
def _conv_dims(B, D, W, T, cap, n_slot=None, act=1):
    return oracle.ConvDims(B=B, D=D, W=W, T=T, cap=cap, n_slot=B if n_slot is None else n_slot,
                           act=act)


def _run_verify(d, ring, pos, x, w, bias, idx=None):
    y = np.zeros((d.B, d.T, d.D))
    st = np.zeros(1, np.int32)
    oracle.conv_verify(d, ring, pos, idx, np.ascontiguousarray(x), np.ascontiguousarray(w),
                       None if bias is None else np.ascontiguousarray(bias), y, st)
    return y, int(st[0])


@pytest.mark.parametrize("W,act", [(1, 0), (2, 1), (3, 0), (4, 1)])
def test_conv_matches_torch_conv1d(W, act):
    """Window + draft through torch.nn.functional.conv1d (depthwise, no padding)."""
    rng = np.random.default_rng(10 + W)
    B, D, T, cap = 3, 16, 6, 11
    d = _conv_dims(B, D, W, T, cap, n_slot=5, act=act)
    ring = rng.normal(size=(5, cap, D))
    pos = rng.integers(0, cap, 5).astype(np.int32)
    idx = np.array([4, 0, 2], np.int32)
    x = rng.normal(size=(B, T, D))
    w = rng.normal(size=(D, W))
    bias = rng.normal(size=D)
    y, st = _run_verify(d, ring.copy(), pos.copy(), x, w, bias, idx)
    assert st == 0
    for b in range(B):
        s = idx[b]
        win = [ring[s, (pos[s] - (W - 1) + j) % cap] for j in range(W - 1)]
        seq = np.concatenate([np.array(win).reshape(W - 1, D), x[b]], 0)       # [W-1+T, D]
        ref = torch.nn.functional.conv1d(torch.from_numpy(seq.T[None]), torch.from_numpy(w[:, None, :]),
                                         torch.from_numpy(bias), groups=D)[0].T.numpy()
        if act:
            ref = ref / (1 + np.exp(-ref))
        np.testing.assert_allclose(y[b], ref, rtol=1e-12, atol=1e-12)


def test_conv_identity_and_shift_kernels():
    """w = e_{W-1} gives y = act(x + bias); w = e_0 gives the input W-1 positions back."""
    rng = np.random.default_rng(5)
    B, D, W, T, cap = 2, 8, 4, 5, 9
    d = _conv_dims(B, D, W, T, cap, act=0)
    ring = rng.normal(size=(B, cap, D))
    pos = np.array([0, 7], np.int32)
    x = rng.normal(size=(B, T, D))
    eye_last = np.zeros((D, W)); eye_last[:, W - 1] = 1
    y, _ = _run_verify(d, ring.copy(), pos.copy(), x, eye_last, np.full(D, 0.25))
    np.testing.assert_allclose(y, x + 0.25, rtol=0, atol=0)
    eye_first = np.zeros((D, W)); eye_first[:, 0] = 1
    y, _ = _run_verify(d, ring.copy(), pos.copy(), x, eye_first, None)
    for b in range(B):
        for t in range(T):
            u = t - (W - 1)
            want = x[b, u] if u >= 0 else ring[b, (pos[b] + u) % cap]
            np.testing.assert_array_equal(y[b, t], want)


def test_conv_rollback_equals_straight_run_over_committed_inputs():
    """verify -> accept(p) over many steps (the ring wraps many times): each step's
    outputs equal the convolution of the committed stream (history plus every accepted
    prefix, nothing rejected) followed by the draft, recomputed from scratch."""
    rng = np.random.default_rng(7)
    B, D, W, T, cap = 3, 8, 4, 6, 9                       # cap = W - 1 + T: the tightest ring
    d = _conv_dims(B, D, W, T, cap, act=1)
    hist = [list(rng.normal(size=(W - 1, D))) for _ in range(B)]
    ring = np.zeros((B, cap, D))
    pos = np.array([2, 8, 5], np.int32)
    for b in range(B):
        for j in range(W - 1):
            ring[b, (pos[b] - (W - 1) + j) % cap] = hist[b][j]
    w, bias = rng.normal(size=(D, W)), rng.normal(size=D)
    st = np.zeros(1, np.int32)
    for step in range(25):
        x = rng.normal(size=(B, T, D))
        y = np.zeros((B, T, D))
        oracle.conv_verify(d, ring, pos, None, x, w, bias, y, st)
        for b in range(B):
            seq = np.array(hist[b][-(W - 1):] + list(x[b]))
            for t in range(T):
                acc = bias + sum(w[:, j] * seq[t + j] for j in range(W))
                np.testing.assert_allclose(y[b, t], acc / (1 + np.exp(-acc)), rtol=1e-13, atol=1e-13)
        acc_n = rng.integers(0, T + 1, B).astype(np.int32)
        oracle.conv_accept(d, pos, None, acc_n, st)
        for b in range(B):
            hist[b].extend(list(x[b, :acc_n[b]]))
    assert st[0] == 0


def test_conv_full_rejection_leaves_window_and_outputs():
    rng = np.random.default_rng(8)
    B, D, W, T, cap = 2, 8, 4, 5, 12
    d = _conv_dims(B, D, W, T, cap)
    ring = rng.normal(size=(B, cap, D))
    pos = np.array([3, 11], np.int32)
    w, bias = rng.normal(size=(D, W)), rng.normal(size=D)
    x = rng.normal(size=(B, T, D))
    y1, _ = _run_verify(d, ring, pos, x, w, bias)
    st = np.zeros(1, np.int32)
    oracle.conv_accept(d, pos, None, np.zeros(B, np.int32), st)
    np.testing.assert_array_equal(pos, [3, 11])
    y2, _ = _run_verify(d, ring, pos, x, w, bias)
    np.testing.assert_array_equal(y1, y2)


def test_conv_status_bits():
    d = _conv_dims(2, 8, 4, 4, 8)
    ring = np.zeros((2, 8, 8))
    pos = np.array([8, 0], np.int32)                       # slot 0 out of range
    y = np.full((2, 4, 8), 9.0)
    st = np.zeros(1, np.int32)
    oracle.conv_verify(d, ring, pos, None, np.zeros((2, 4, 8)), np.zeros((8, 4)), None, y, st)
    assert st[0] == 4 and (y[0] == 9.0).all()
    st[0] = 0
    oracle.conv_accept(d, pos, None, np.array([1, 5], np.int32), st)
    assert st[0] == 4 | 1 and pos[1] == 0


@pytest.mark.parametrize("name", ["conv_identity_act_width3", "conv_wraps_the_ring"])
def test_conv_hand_examples(name):
    c = _golden()[name]
    D, W, T, cap = (int(c[k][0]) for k in ("D", "W", "T", "cap"))
    d = _conv_dims(1, D, W, T, cap, act=int(c["act"][0]))
    ring = np.array(c["ring"], float).reshape(1, cap, D)
    pos = np.array([int(c["pos"][0])], np.int32)
    x = np.array(c["x"], float).reshape(1, T, D)
    w = np.array(c["w"], float).reshape(D, W)
    bias = np.full(D, float(c["bias"][0]))
    y, st = _run_verify(d, ring, pos, x, w, bias)
    assert st == 0
    np.testing.assert_array_equal(y.ravel(), np.array(c["y"], float))
    np.testing.assert_array_equal(ring.ravel(), np.array(c["ring_after"], float))
    s = np.zeros(1, np.int32)
    oracle.conv_accept(d, pos, None, np.array([int(c["accept"][0])], np.int32), s)
    assert int(pos[0]) == int(c["pos_after"][0])


# ----------------------------------------------------------------------- E4M3
def _format_value(code):
    """E4M3 from its definition: sign, 4-bit exponent with bias 7, 3-bit mantissa,
    exponent field 0 subnormal."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e4m3_decode_matches_the_format_definition():
    for code in range(256):
        if code & 0x7F == 0x7F:
            assert math.isnan(oracle.e4m3_decode(code))
            continue
        assert oracle.e4m3_decode(code) == _format_value(code), hex(code)
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_every_code_round_trips():
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(code)) == code, hex(code)


def test_e4m3_ties_go_to_the_even_mantissa():
    for code in range(0, 0x7E):
        lo, hi = _format_value(code), _format_value(code + 1)
        mid = (lo + hi) / 2
        want = code if code % 2 == 0 else code + 1
        assert oracle.e4m3_encode(mid) == want, hex(code)
        assert oracle.e4m3_encode(-mid) == want | 0x80
        assert oracle.e4m3_encode(np.nextafter(mid, 0)) == code
        assert oracle.e4m3_encode(np.nextafter(mid, 1e9)) == code + 1


def test_e4m3_saturates():
    for x in (448.0, 449.0, 463.9, 464.0, 1e6, 1e300):
        assert oracle.e4m3_encode(x) == 0x7E and oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -11) == 0x00 and oracle.e4m3_encode(-0.0) == 0x80


def test_e4m3_matches_torch_float8_cast_in_range():
    """torch's float8_e4m3fn conversion (round to nearest even) on random values across
    the whole finite range, subnormals included."""
    rng = np.random.default_rng(11)
    mag = np.exp2(rng.uniform(-12, 8.8, 20000))
    x = np.where(rng.random(20000) < 0.5, -mag, mag)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    np.testing.assert_array_equal(got, ref)


# --------------------------------------------------------- gated RMSNorm + E4M3
def test_norm_constant_row_closed_form():
    """A constant row c: mean(o^2) = c^2, so (eps = 0) y = sign(c) w silu(z)."""
    rng = np.random.default_rng(12)
    d = 64
    o = np.full((3, d), [[-2.5], [0.75], [13.0]])
    z, w = rng.normal(size=(3, d)), rng.normal(size=d)
    _, yq = oracle.gated_rmsnorm_fp8(o, z, w, 0.0, 1.0)
    silu = z / (1 + np.exp(-z))
    np.testing.assert_allclose(yq, np.sign(o) * w * silu, rtol=1e-14, atol=1e-15)


def test_norm_scale_invariance_and_zero_gate():
    rng = np.random.default_rng(13)
    o, z, w = rng.normal(size=(4, 128)), rng.normal(size=(4, 128)), rng.normal(size=128)
    q1, y1 = oracle.gated_rmsnorm_fp8(o, z, w, 0.0, 3.0)
    q2, y2 = oracle.gated_rmsnorm_fp8(o * 1024.0, z, w, 0.0, 3.0)     # power of two: exact
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_allclose(y1, y2, rtol=1e-15)
    q0, y0 = oracle.gated_rmsnorm_fp8(o, np.zeros_like(z), w, 1e-6, 3.0)
    assert (np.abs(y0) == 0).all() and set(np.unique(q0)) <= {0x00, 0x80}


def test_norm_codes_are_the_e4m3_of_the_value():
    rng = np.random.default_rng(14)
    o, z, w = rng.normal(size=(8, 128)), rng.normal(size=(8, 128)), 1 + 0.1 * rng.normal(size=128)
    q, yq = oracle.gated_rmsnorm_fp8(o, z, w, 1e-6, 40.0)
    flat = yq.ravel()
    ref = torch.from_numpy(np.clip(flat, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q.ravel(), ref)


@pytest.mark.parametrize("name", ["norm_unit_rms", "norm_rounding_and_saturation"])
def test_norm_hand_examples(name):
    c = _golden()[name]
    d = int(c["d"][0])
    f = lambda k: np.array(c[k], float).reshape(1, d) if k in ("o", "z") else np.array(c[k], float)  # noqa: E731
    q, _ = oracle.gated_rmsnorm_fp8(f("o"), f("z"), f("w"), float(c["eps"][0]), float(c["inv_scale"][0]))
    assert [int(v) for v in q.ravel()] == [int(h, 16) for h in c["codes"]]
