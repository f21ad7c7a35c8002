"""Pins for the CPU oracle: brute force, closed forms, hand-worked examples
and the ReplaySSM invariants.  None of these compare the oracle with itself:
each checks it against the mathematics of the gated delta rule (Gated Delta
Networks, ICLR 2025) or the bookkeeping the OCRia inference-stack post
describes in "Making speculative verification cheaper" (checkpoint + buffer,
periodic flush, rollback as a buffer-pointer move) together with the prefix
acceptance rule of "Inference Engineering", chapter 5 (speculative decoding).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_rule_hand_examples.txt")


def dims(dk, dv, *, B=1, H=1, T=1, cap=8, threshold=4, n_slot=None, scale=None, fp32=False, thr=1):
    return oracle.Dims(B=B, H=H, dk=dk, dv=dv, T=T, cap=cap, threshold=threshold,
                       n_slot=B if n_slot is None else n_slot,
                       scale=1.0 / math.sqrt(dk) if scale is None else scale,
                       fp32_mode=fp32, n_threads=thr)


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def matrix_form(S, k, v, g, beta, q, scale):
    """Textbook form: S <- alpha S (I - beta k k^T) + beta v k^T; o = S (scale q)."""
    dk = S.shape[1]
    outs = []
    for t in range(k.shape[0]):
        a = math.exp(g[t])
        P = np.eye(dk) - beta[t] * np.outer(k[t], k[t])
        S = a * S @ P + beta[t] * np.outer(v[t], k[t])
        outs.append(S @ (scale * q[t]))
    return S, np.array(outs)


# ----------------------------------------------------------------- brute force
@pytest.mark.parametrize("dk,dv", [(2, 2), (4, 4), (8, 8), (4, 3), (3, 5), (8, 2)])
def test_rank_one_form_matches_explicit_matrix(dk, dv):
    rng = np.random.default_rng(dk * 100 + dv)
    n = 7
    S0 = rng.normal(0, 0.5, (dv, dk))
    k, q = unit(rng.normal(size=(n, dk))), unit(rng.normal(size=(n, dk)))
    v = rng.normal(size=(n, dv))
    g = -np.log1p(np.exp(rng.normal(size=n)))
    beta = 1 / (1 + np.exp(-rng.normal(size=n)))
    d = dims(dk, dv)
    S = S0.copy()
    o = oracle.recur(d, S, k, v, g, beta, q=q)
    S_ref, o_ref = matrix_form(S0, k, v, g, beta, q, d.scale)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)


def test_exact_rationals_tiny():
    """Exact rational arithmetic (alpha given as an exact binary fraction)."""
    dk, dv = 3, 2
    S0 = [[Fraction(1), Fraction(-2), Fraction(1, 2)], [Fraction(3, 4), Fraction(0), Fraction(5)]]
    toks = [((1, 2, 2), (1, -1), -math.log(2), Fraction(1, 4)),
            ((2, -1, 0), (0, 3), 0.0, Fraction(1, 2))]
    S = [row[:] for row in S0]
    for k, v, g, beta in toks:
        alpha = Fraction(math.exp(g)).limit_denominator(64)
        k = [Fraction(x) for x in k]
        Sk = [sum(S[i][j] * k[j] for j in range(dk)) for i in range(dv)]
        S = [[alpha * S[i][j] - alpha * beta * Sk[i] * k[j] + beta * v[i] * k[j]
              for j in range(dk)] for i in range(dv)]
    Sd = np.array(S0, dtype=float)
    ks = np.array([t[0] for t in toks], float)
    vs = np.array([t[1] for t in toks], float)
    oracle.recur(dims(dk, dv, scale=1.0), Sd, ks, vs, np.array([t[2] for t in toks]),
                 np.array([float(t[3]) for t in toks]))
    np.testing.assert_allclose(Sd, np.array(S, dtype=float), rtol=0, atol=1e-13)


# ------------------------------------------------------------------ closed forms
def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = (prod alpha) S0 and o_t = (prod_{s<=t} alpha_s) S0 (scale q_t)."""
    rng = np.random.default_rng(1)
    dk, dv, n = 16, 12, 9
    S0 = rng.normal(0, 0.1, (dv, dk))
    k, q = unit(rng.normal(size=(n, dk))), unit(rng.normal(size=(n, dk)))
    v = rng.normal(size=(n, dv))
    g = -np.abs(rng.normal(size=n))
    d = dims(dk, dv)
    S = S0.copy()
    o = oracle.recur(d, S, k, v, g, np.zeros(n), q=q)
    cum = np.exp(np.cumsum(g))
    np.testing.assert_allclose(S, cum[-1] * S0, rtol=1e-13, atol=0)
    np.testing.assert_allclose(o, cum[:, None] * (S0 @ (d.scale * q).T).T, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("n", [1, 5, 16])
def test_orthonormal_keys_are_retrieved(n):
    """alpha = 1, beta = 1, orthonormal keys: after writing all n, S k_i = v_i."""
    rng = np.random.default_rng(n)
    dk, dv = 16, 8
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    k = Qm[:, :n].T.copy()
    v = rng.normal(size=(n, dv))
    S = rng.normal(0, 0.1, (dv, dk))
    oracle.recur(dims(dk, dv), S, k, v, np.zeros(n), np.ones(n))
    np.testing.assert_allclose(S @ k.T, v.T, rtol=0, atol=1e-12)


def test_output_reads_post_update_state_with_scale():
    """S0 = 0, one token: o = beta v (k . scale q) (the pre-update state gives 0)."""
    dk, dv = 8, 4
    rng = np.random.default_rng(3)
    k, q = unit(rng.normal(size=(1, dk))), unit(rng.normal(size=(1, dk)))
    v = rng.normal(size=(1, dv))
    d = dims(dk, dv)
    o = oracle.recur(d, np.zeros((dv, dk)), k, v, np.array([-0.3]), np.array([0.7]), q=q)
    np.testing.assert_allclose(o[0], 0.7 * v[0] * (k[0] @ q[0]) * d.scale, rtol=1e-13)


def test_near_reset_gate():
    """g = -20: alpha ~ 2e-9, so S1 = beta v k^T up to 2e-9 relative."""
    dk, dv = 8, 8
    rng = np.random.default_rng(4)
    S = rng.normal(0, 1, (dv, dk))
    k, v = unit(rng.normal(size=(1, dk))), rng.normal(size=(1, dv))
    oracle.recur(dims(dk, dv), S, k, v, np.array([-20.0]), np.array([0.9]))
    np.testing.assert_allclose(S, 0.9 * np.outer(v[0], k[0]), rtol=0, atol=1e-7)


# ---------------------------------------------------------- hand-worked fixture
def _parse_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "tokens": [], "buffer": [], "draft": []}
        elif key == "end":
            cases.append(cur)
        elif key in ("token", "buffer", "draft"):
            tok = {}
            for kv in rest.split():
                name, val = kv.split("=")
                if name == "g" and val.startswith("ln"):
                    tok[name] = math.log(float(val[2:]))
                else:
                    tok[name] = [float(x) for x in val.split(",")]
            cur["tokens" if key == "token" else key].append(tok)
        elif key in ("dk", "dv", "threshold", "accept1_len", "accept0_len"):
            cur[key] = int(rest)
        elif key == "scale":
            cur[key] = float(rest)
        else:
            cur[key] = np.array([[float(x) for x in r.split()] for r in rest.split(";")])
    return cases


def _g(tok):
    return tok["g"] if isinstance(tok["g"], float) else tok["g"][0]


@pytest.mark.parametrize("case", [c for c in _parse_golden() if c["tokens"]], ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    d = dims(case["dk"], case["dv"], scale=case["scale"])
    toks = case["tokens"]
    S = case["S0"].copy()
    o = oracle.recur(d, S, np.array([t["k"] for t in toks]), np.array([t["v"] for t in toks]),
                     np.array([_g(t) for t in toks]), np.array([t["beta"][0] for t in toks]),
                     q=np.array([t["q"] for t in toks]))
    np.testing.assert_allclose(S, case["S"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, case["o"].reshape(o.shape), rtol=0, atol=1e-14)


def _layer_from(case, n_buf_cap=4):
    dk, dv = case["dk"], case["dv"]
    d = dims(dk, dv, T=1, cap=n_buf_cap, threshold=case["threshold"], scale=case["scale"])
    st = case["S0"].reshape(1, 1, dv, dk).copy()
    bk, bv = np.zeros((1, 1, d.cap, dk)), np.zeros((1, 1, d.cap, dv))
    bg, bb = np.zeros((1, 1, d.cap)), np.zeros((1, 1, d.cap))
    for t, tok in enumerate(case["buffer"]):
        bk[0, 0, t], bv[0, 0, t], bg[0, 0, t], bb[0, 0, t] = tok["k"], tok["v"], _g(tok), tok["beta"][0]
    ln = np.array([len(case["buffer"])], np.int32)
    dr = case["draft"][0]
    blk = dict(q=np.array(dr["q"]).reshape(1, 1, 1, dk), k=np.array(dr["k"]).reshape(1, 1, 1, dk),
               v=np.array(dr["v"]).reshape(1, 1, 1, dv), g=np.array([[[_g(dr)]]]),
               beta=np.array([[[dr["beta"][0]]]]))
    return d, st, bk, bv, bg, bb, ln, blk


@pytest.mark.parametrize("p", [0, 1])
def test_hand_worked_bookkeeping(p):
    case = [c for c in _parse_golden() if c["name"] == "replay_bookkeeping"][0]
    d, st, bk, bv, bg, bb, ln, blk = _layer_from(case)
    status = np.zeros(1, np.int32)
    out = np.zeros((1, 1, 1, d.dv))
    oracle.verify(d, st, None, bk, bv, bg, bb, ln, blk["q"], blk["k"], blk["v"], blk["g"], blk["beta"],
                  out, status)
    np.testing.assert_allclose(out.ravel(), case["verify_out"].ravel(), rtol=0, atol=1e-14)
    np.testing.assert_array_equal(st[0, 0], case["S0"])
    oracle.accept(d, ln, None, np.array([p], np.int32), status)
    oracle.flush(d, st, None, bk, bv, bg, bb, ln, False, status)
    assert status[0] == 0
    np.testing.assert_allclose(st[0, 0], case[f"accept{p}_state"], rtol=0, atol=1e-6)
    assert ln[0] == case[f"accept{p}_len"]


# ----------------------------------------------------- batched layout and slots
def _random_layer(d, rng, lens):
    st = rng.normal(0, 0.1, (d.n_slot, d.H, d.dv, d.dk)).astype(np.float32).astype(np.float64)
    bk = unit(rng.normal(size=(d.n_slot, d.H, d.cap, d.dk)))
    bv = rng.normal(size=(d.n_slot, d.H, d.cap, d.dv))
    bg = -np.log1p(np.exp(rng.normal(size=(d.n_slot, d.H, d.cap))))
    bb = 1 / (1 + np.exp(-rng.normal(size=(d.n_slot, d.H, d.cap))))
    return st, bk, bv, bg, bb, np.array(lens, np.int32)


def _random_block(d, rng):
    q = unit(rng.normal(size=(d.B, d.T, d.H, d.dk)))
    k = unit(rng.normal(size=(d.B, d.T, d.H, d.dk)))
    v = rng.normal(size=(d.B, d.T, d.H, d.dv))
    g = -np.log1p(np.exp(rng.normal(size=(d.B, d.T, d.H))))
    beta = 1 / (1 + np.exp(-rng.normal(size=(d.B, d.T, d.H))))
    return q, k, v, g, beta


def test_verify_layout_against_explicit_matrix_form():
    """Batched verify with a slot map equals the textbook form per (b, h),
    with indices taken from the documented layouts."""
    rng = np.random.default_rng(7)
    d = dims(6, 5, B=3, H=2, T=3, cap=9, threshold=6, n_slot=5, thr=2)
    idx = np.array([4, 0, 2], np.int32)
    lens = [2, 0, 0, 0, 6]
    st, bk, bv, bg, bb, ln = _random_layer(d, rng, lens)
    q, k, v, g, beta = _random_block(d, rng)
    out = np.zeros((d.B, d.T, d.H, d.dv))
    status = np.zeros(1, np.int32)
    bk0 = bk.copy()
    oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
    assert status[0] == 0
    for b in range(d.B):
        s = idx[b]
        L = lens[s]
        for h in range(d.H):
            kk = np.concatenate([bk0[s, h, :L], k[b, :, h]])
            vv = np.concatenate([bv[s, h, :L], v[b, :, h]])
            gg = np.concatenate([bg[s, h, :L], g[b, :, h]])
            bt = np.concatenate([bb[s, h, :L], beta[b, :, h]])
            qq = np.concatenate([np.zeros((L, d.dk)), q[b, :, h]])
            _, o_ref = matrix_form(st[s, h], kk, vv, gg, bt, qq, d.scale)
            np.testing.assert_allclose(out[b, :, h], o_ref[L:], rtol=0, atol=1e-12)
            np.testing.assert_array_equal(bk[s, h, L:L + d.T], k[b, :, h])


# ------------------------------------------------------------ ReplaySSM invariants
def _setup(seed, fp32=False, **kw):
    rng = np.random.default_rng(seed)
    base = dict(B=3, H=2, T=4, cap=11, threshold=8, n_slot=4, thr=2)
    base.update(kw)
    d = dims(8, 6, fp32=fp32, **base)
    idx = np.array([3, 1, 0], np.int32)[:d.B]
    lens = [int(x) for x in rng.integers(0, d.threshold, d.n_slot)]
    layer = _random_layer(d, rng, lens)
    if fp32:
        layer = tuple(a.astype(np.float32).astype(np.float64) if a.dtype == np.float64 else a for a in layer)
    return d, idx, rng, layer


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_verify_accept_flush_equals_sequential_run(seed):
    """verify -> accept(p) -> forced flush == straight run over buffer + p accepted tokens
    (bit-exact: the same operations in the same order)."""
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(seed)
    q, k, v, g, beta = _random_block(d, rng)
    p = np.array([d.T, 0, 2], np.int32)
    st0, bk0, bv0, bg0, bb0, ln0 = st.copy(), bk.copy(), bv.copy(), bg.copy(), bb.copy(), ln.copy()
    out = np.zeros((d.B, d.T, d.H, d.dv))
    status = np.zeros(1, np.int32)
    oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
    oracle.accept(d, ln, idx, p, status)
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, True, status)
    assert status[0] == 0
    for b in range(d.B):
        s, L = idx[b], ln0[idx[b]]
        assert ln[s] == 0 or (L + p[b] == 0 and ln[s] == 0)
        for h in range(d.H):
            S = st0[s, h].copy()
            oracle.recur(d, S, bk0[s, h, :L], bv0[s, h, :L], bg0[s, h, :L], bb0[s, h, :L])
            o = oracle.recur(d, S, k[b, :, h], v[b, :, h], g[b, :, h], beta[b, :, h], q=q[b, :, h])
            np.testing.assert_array_equal(out[b, :, h], o)
            S = st0[s, h].copy()
            oracle.recur(d, S, bk0[s, h, :L], bv0[s, h, :L], bg0[s, h, :L], bb0[s, h, :L])
            oracle.recur(d, S, k[b, :p[b], h], v[b, :p[b], h], g[b, :p[b], h], beta[b, :p[b], h])
            np.testing.assert_array_equal(st[s, h], S.astype(np.float32).astype(np.float64))


def test_full_rejection_leaves_everything_bit_identical():
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(11)
    q, k, v, g, beta = _random_block(d, rng)
    st0, ln0, bk0 = st.copy(), ln.copy(), bk.copy()
    status = np.zeros(1, np.int32)
    out = np.zeros((d.B, d.T, d.H, d.dv))
    oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
    oracle.accept(d, ln, idx, np.zeros(d.B, np.int32), status)
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, False, status)
    assert status[0] == 0
    np.testing.assert_array_equal(st, st0)
    np.testing.assert_array_equal(ln, ln0)
    for s in range(d.n_slot):
        np.testing.assert_array_equal(bk[s, :, :ln0[s]], bk0[s, :, :ln0[s]])


def test_flush_empty_is_noop_and_idempotent():
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(12)
    status = np.zeros(1, np.int32)
    ln[:] = 0
    st0 = st.copy()
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, True, status)
    np.testing.assert_array_equal(st, st0)
    ln[idx] = [5, 0, 3]
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, True, status)
    st1, ln1 = st.copy(), ln.copy()
    assert (ln1 == 0).all()
    assert not np.array_equal(st1, st0)
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, True, status)
    np.testing.assert_array_equal(st, st1)
    np.testing.assert_array_equal(ln, ln1)
    assert status[0] == 0


def test_flush_threshold_rule():
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(13)
    ln[:] = 0
    ln[idx] = [d.threshold, d.threshold - 1, d.cap]
    st0 = st.copy()
    status = np.zeros(1, np.int32)
    oracle.flush(d, st, idx, bk, bv, bg, bb, ln, False, status)
    assert list(ln[idx]) == [0, d.threshold - 1, 0]
    np.testing.assert_array_equal(st[idx[1]], st0[idx[1]])
    assert not np.array_equal(st[idx[0]], st0[idx[0]])


def test_flush_schedule_invariance_fp32_mode():
    """In per-operation fp32 mode, flushing every step or only at the threshold
    gives a bit-identical state: the same fp32 operations run either way."""
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(21, fp32=True)
    runs = []
    for every_step in (True, False):
        S, BK, BV, BG, BB, L = st.copy(), bk.copy(), bv.copy(), bg.copy(), bb.copy(), ln.copy()
        r = np.random.default_rng(99)
        status = np.zeros(1, np.int32)
        for step in range(6):
            q, k, v, g, beta = [a.astype(np.float32).astype(np.float64) for a in _random_block(d, r)]
            p = r.integers(0, d.T + 1, d.B).astype(np.int32)
            out = np.zeros((d.B, d.T, d.H, d.dv))
            oracle.verify(d, S, idx, BK, BV, BG, BB, L, q, k, v, g, beta, out, status)
            oracle.accept(d, L, idx, p, status)
            oracle.flush(d, S, idx, BK, BV, BG, BB, L, every_step, status)
        oracle.flush(d, S, idx, BK, BV, BG, BB, L, True, status)
        assert status[0] == 0
        runs.append(S)
    np.testing.assert_array_equal(runs[0], runs[1])


def test_verify_is_pure():
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(31)
    q, k, v, g, beta = _random_block(d, rng)
    st0, ln0 = st.copy(), ln.copy()
    status = np.zeros(1, np.int32)
    outs = []
    for _ in range(2):
        out = np.zeros((d.B, d.T, d.H, d.dv))
        oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
        outs.append(out)
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(st, st0)
    np.testing.assert_array_equal(ln, ln0)


def test_status_bits_and_skips():
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(41)
    ln[:] = 0
    ln[idx] = [d.cap - d.T + 1, 2, 0]          # sequence 0 has no room for the draft
    q, k, v, g, beta = _random_block(d, rng)
    status = np.zeros(1, np.int32)
    out = np.full((d.B, d.T, d.H, d.dv), 7.0)
    oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
    assert status[0] == oracle.NO_ROOM
    assert (out[0] == 7.0).all() and not (out[1] == 7.0).any()
    status[0] = 0
    ln0 = ln.copy()
    oracle.accept(d, ln, idx, np.array([-1, d.T + 1, 3], np.int32), status)
    assert status[0] == oracle.BAD_ACCEPT
    assert list(ln[idx]) == [ln0[idx[0]], ln0[idx[1]], 3]
    status[0] = 0
    oracle.accept(d, ln, idx, np.array([d.T, 0, 0], np.int32), status)   # len + p > cap
    assert status[0] == oracle.BAD_LEN


# ------------------------------------------------- many steps against a plain model
@pytest.mark.parametrize("seed", [11, 12, 13])
def test_many_steps_against_a_matrix_form_model(seed):
    """Twelve decode steps with random accepted counts (0..T), threshold flushes and a
    forced flush every fifth step, against an independent model of the method written
    with the textbook matrix form: per slot a checkpoint (rounded to fp32 when it is
    rewritten) and the list of tokens committed since; a verify runs the matrix form
    from the checkpoint over that list and the draft; an accept appends the first p
    draft tokens; a flush of a list that reached the threshold (any non-empty one when
    forced) replaces the checkpoint by the rounded state after it and empties the list.
    The slot that no sequence owns must never change."""
    d, idx, rng, (st, bk, bv, bg, bb, ln) = _setup(seed, T=3, cap=10, threshold=6)
    model_S = {int(s): st[s].copy() for s in range(d.n_slot)}
    model_list = {int(s): [(bk[s, :, t].copy(), bv[s, :, t].copy(), bg[s, :, t].copy(), bb[s, :, t].copy())
                           for t in range(ln[s])] for s in range(d.n_slot)}
    unused = [s for s in range(d.n_slot) if s not in idx]
    st_unused = st[unused].copy()
    status = np.zeros(1, np.int32)
    folds = 0

    def run(S, toks, q=None):
        """S: [dv, dk] for one head; toks: (k, v, g, beta) per token for that head; the
        output after each token whose query (q[i]) is given."""
        outs = []
        for i, (k, v, g, be) in enumerate(toks):
            S = math.exp(g) * S @ (np.eye(d.dk) - be * np.outer(k, k)) + be * np.outer(v, k)
            if q is not None and q[i] is not None:
                outs.append(S @ (d.scale * q[i]))
        return S, np.array(outs)

    for step in range(12):
        q, k, v, g, beta = _random_block(d, rng)
        out = np.zeros((d.B, d.T, d.H, d.dv))
        oracle.verify(d, st, idx, bk, bv, bg, bb, ln, q, k, v, g, beta, out, status)
        for b in range(d.B):
            s = int(idx[b])
            for h in range(d.H):
                toks = [(kk[h], vv[h], gg[h], be[h]) for kk, vv, gg, be in model_list[s]]
                drafts = [(k[b, t, h], v[b, t, h], g[b, t, h], beta[b, t, h]) for t in range(d.T)]
                _, o = run(model_S[s][h], toks + drafts, q=[None] * len(toks) + list(q[b, :, h]))
                np.testing.assert_allclose(out[b, :, h], o, rtol=1e-9, atol=1e-12)
        p = rng.integers(0, d.T + 1, d.B).astype(np.int32)
        oracle.accept(d, ln, idx, p, status)
        for b in range(d.B):
            s = int(idx[b])
            model_list[s] += [(k[b, t].copy(), v[b, t].copy(), g[b, t].copy(), beta[b, t].copy())
                              for t in range(p[b])]
        force = step % 5 == 4
        oracle.flush(d, st, idx, bk, bv, bg, bb, ln, force, status)
        for b in range(d.B):
            s = int(idx[b])
            n = len(model_list[s])
            if n >= d.threshold or (force and n > 0):
                model_S[s] = np.array([run(model_S[s][h], [(kk[h], vv[h], gg[h], be[h])
                                                           for kk, vv, gg, be in model_list[s]])[0]
                                       for h in range(d.H)]).astype(np.float32).astype(np.float64)
                model_list[s] = []
                folds += 1
            assert ln[s] == len(model_list[s])
            np.testing.assert_allclose(st[s], model_S[s], rtol=2.0 ** -22, atol=1e-30)
        assert status[0] == 0
        np.testing.assert_array_equal(st[unused], st_unused)
    assert folds >= 6
