"""Pins for the oracle of the non-replay baseline (the data movement ReplaySSM
avoids, "The inference stack behind OCRia", section "Making speculative
verification cheaper": without a buffer, a rejection must restore a stored
state).  The baseline stores the state after every draft token and restores
by copying the snapshot of the accepted prefix.

Pinned against: the textbook matrix form of the gated delta rule (Gated Delta
Networks, ICLR 2025) written with numpy matrix products; the ReplaySSM oracle
(checkpoint + buffer + forced flush), which must reach bit-identical outputs
and states; the beta = 0 closed form; and the prefix-acceptance bookkeeping
("Inference Engineering", chapter 5: p = 0 keeps the state, p outside [0, T]
is rejected)."""
import math

import numpy as np
import pytest

import oracle


def _dims(B=2, H=2, dk=8, dv=6, T=5, n_slot=3):
    return oracle.Dims(B=B, H=H, dk=dk, dv=dv, T=T, cap=T, threshold=1, n_slot=n_slot,
                       scale=1.0 / math.sqrt(dk))


def _inputs(d, seed, beta_zero=False):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)  # noqa: E731
    state = np.ascontiguousarray(rng.normal(0, 0.5, (d.n_slot, d.H, d.dv, d.dk)).astype(np.float32)
                                 .astype(np.float64))
    blk = dict(q=unit(rng.normal(size=(d.B, d.T, d.H, d.dk))), k=unit(rng.normal(size=(d.B, d.T, d.H, d.dk))),
               v=rng.normal(size=(d.B, d.T, d.H, d.dv)),
               g=-np.log1p(np.exp(rng.normal(size=(d.B, d.T, d.H)))),
               beta=np.zeros((d.B, d.T, d.H)) if beta_zero else 1 / (1 + np.exp(-rng.normal(size=(d.B, d.T, d.H)))))
    blk = {n: np.ascontiguousarray(a) for n, a in blk.items()}
    state_idx = np.ascontiguousarray(rng.permutation(d.n_slot)[:d.B].astype(np.int32))
    return state, state_idx, blk


def _matrix_form(S, blk, b, h, scale):
    """S <- alpha S (I - beta k k^T) + beta v k^T, o = S (scale q), token by token."""
    snaps, outs = [], []
    for t in range(blk["k"].shape[1]):
        k, v, q = blk["k"][b, t, h], blk["v"][b, t, h], blk["q"][b, t, h]
        a, be = math.exp(blk["g"][b, t, h]), blk["beta"][b, t, h]
        S = a * S @ (np.eye(S.shape[1]) - be * np.outer(k, k)) + be * np.outer(v, k)
        snaps.append(S.copy())
        outs.append(S @ (scale * q))
    return np.array(snaps), np.array(outs)


def test_snapshots_and_outputs_match_the_matrix_form():
    d = _dims()
    state, idx, blk = _inputs(d, 1)
    lay = oracle.NonReplayLayer(d, state, idx)
    out = lay.verify(blk)
    assert lay.status[0] == 0
    np.testing.assert_array_equal(lay.state, state)                  # the verify writes no state
    for b in range(d.B):
        for h in range(d.H):
            snaps, outs = _matrix_form(state[idx[b], h], blk, b, h, d.scale)
            np.testing.assert_allclose(out[b, :, h], outs, rtol=0, atol=1e-12)
            # stored as binary32: the rounding of the exact state, to the last bit
            np.testing.assert_array_equal(lay.snap[b, h], lay.snap[b, h].astype(np.float32).astype(np.float64))
            np.testing.assert_allclose(lay.snap[b, h], snaps, rtol=2.0 ** -23, atol=1e-30)


@pytest.mark.parametrize("p", [0, 1, 3, 5])
def test_restore_by_copy_equals_replay_with_a_forced_flush(p):
    """ReplaySSM (empty buffer, verify, accept p, forced flush) and the baseline
    (verify, accept p) reach the same outputs and the same fp32 state, bit for bit."""
    d = _dims()
    state, idx, blk = _inputs(d, 2)
    nr = oracle.NonReplayLayer(d, state, idx)
    out_nr = nr.verify(blk)
    nr.accept(np.full(d.B, p, np.int32))
    init = dict(state=state, buf_k=np.zeros((d.n_slot, d.H, d.cap, d.dk)),
                buf_v=np.zeros((d.n_slot, d.H, d.cap, d.dv)), buf_g=np.zeros((d.n_slot, d.H, d.cap)),
                buf_beta=np.zeros((d.n_slot, d.H, d.cap)))
    rp_state = init["state"].copy()
    lens = np.zeros(d.n_slot, np.int32)
    st = np.zeros(1, np.int32)
    out_rp = np.zeros((d.B, d.T, d.H, d.dv))
    oracle.verify(d, rp_state, idx, init["buf_k"], init["buf_v"], init["buf_g"], init["buf_beta"], lens,
                  blk["q"], blk["k"], blk["v"], blk["g"], blk["beta"], out_rp, st)
    oracle.accept(d, lens, idx, np.full(d.B, p, np.int32), st)
    oracle.flush(d, rp_state, idx, init["buf_k"], init["buf_v"], init["buf_g"], init["buf_beta"], lens, True, st)
    assert st[0] == 0 and nr.status[0] == 0
    np.testing.assert_array_equal(out_nr, out_rp)
    np.testing.assert_array_equal(nr.state, rp_state)
    if p == 0:
        np.testing.assert_array_equal(nr.state, state)


def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = exp(g_1 + ... + g_t) S_0 (closed form)."""
    d = _dims(B=1, H=1, n_slot=1)
    state, idx, blk = _inputs(d, 3, beta_zero=True)
    lay = oracle.NonReplayLayer(d, state, idx)
    lay.verify(blk)
    G = np.cumsum(blk["g"][0, :, 0])
    for t in range(d.T):
        np.testing.assert_allclose(lay.snap[0, 0, t], math.exp(G[t]) * state[0, 0], rtol=2.0 ** -23, atol=1e-30)


def test_status_bits_and_skipped_rows():
    d = _dims(B=3)
    state, idx, blk = _inputs(d, 4)
    idx = np.ascontiguousarray(np.array([2, 5, 0], np.int32))        # slot 5 does not exist
    lay = oracle.NonReplayLayer(d, state, idx)
    out = lay.verify(blk)
    assert lay.status[0] == oracle.BAD_SLOT
    assert not out[1].any() and not lay.snap[1].any()                 # the bad row is skipped
    lay.status[:] = 0
    before = lay.state.copy()
    lay.accept(np.array([d.T + 1, 2, -1], np.int32))                  # bad count, bad slot, bad count
    assert lay.status[0] == oracle.BAD_ACCEPT | oracle.BAD_SLOT
    np.testing.assert_array_equal(lay.state, before)                  # nothing restored
    lay.status[:] = 0
    lay.accept(np.array([d.T, 0, 1], np.int32))
    assert lay.status[0] == oracle.BAD_SLOT
    np.testing.assert_array_equal(lay.state[2], lay.snap[0, :, d.T - 1])
    np.testing.assert_array_equal(lay.state[0], lay.snap[2, :, 0])
    np.testing.assert_array_equal(lay.state[1], before[1])            # slot of no row: untouched
