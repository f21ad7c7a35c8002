"""GPU parity of the non-replay baseline (include/gdnnonreplay.h) against its
fp64 CPU oracle on the same seeded inputs: outputs, every stored snapshot and
the restored state within max|d| <= 2e-3 max|ref| + 1e-5 per tensor and step;
status words exact; nothing written outside the rows and tensors the ABI names."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads
from harness import assert_close, to_np

pytestmark = pytest.mark.gpu
WL = synth.WORKLOADS


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def _dims(wl, B, n_slot):
    import speculative_decode_recurrent_gb300 as lib
    return lib.Dims(B=B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.T, threshold=1, n_slot=n_slot,
                    in_dtype=lib.DTYPE_BF16 if wl.in_dtype == "bf16" else lib.DTYPE_F32, scale=wl.scale)


def _odims(wl, B, n_slot):
    return oracle.Dims(B=B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.T, threshold=1, n_slot=n_slot,
                       scale=wl.scale, n_threads=16)


class NrPair:
    """GPU and oracle layers of the baseline from one seeded initial state; the
    oracle may follow a subset of the batch rows (``rows``), which are independent."""

    def __init__(self, wl, layer=0, rows=None):
        import speculative_decode_recurrent_gb300 as lib
        self.wl = wl
        init = synth.initial_layer(wl, layer)
        self.B, self.n_slot = wl.B, init["state"].shape[0]
        self.layer = layer
        self.gpu = lib.NonReplayLayer(_dims(wl, self.B, self.n_slot), init["state"], init["state_idx"])
        self.rows = np.arange(self.B) if rows is None else np.asarray(rows)
        idx = init["state_idx"].numpy()[self.rows].astype(np.int32)
        self.orc = oracle.NonReplayLayer(_odims(wl, len(self.rows), self.n_slot),
                                         init["state"].double().numpy(), idx)
        self.slots = idx

    def step(self, s):
        wl, r = self.wl, torch.as_tensor(self.rows)
        blk = synth.draft_block(wl, self.layer, s)
        acc = synth.workloads.accepted_counts(wl, self.layer, s)
        out = torch.full((self.B, wl.T, wl.H, wl.dv), float("nan"), device="cuda")
        dev = {n: t.cuda() for n, t in blk.items()}
        self.gpu.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
        o_ref = self.orc.verify({n: blk[n][r].double().numpy() for n in ("q", "k", "v", "g", "beta")})
        torch.cuda.synchronize()
        tag = f"{wl.name}/step{s}"
        assert int(self.gpu.status.item()) == 0, tag
        assert_close(f"out {tag}", to_np(out)[self.rows], o_ref)
        snap = self.gpu.snap.view(self.B, wl.H, wl.T, wl.dv, wl.dk)
        assert_close(f"snap {tag}", to_np(snap[r.cuda()]), self.orc.snap)
        self.gpu.accept(acc.cuda())
        self.orc.accept(acc.numpy()[self.rows])
        torch.cuda.synchronize()
        assert int(self.gpu.status.item()) == 0 and int(self.orc.status[0]) == 0, tag
        assert_close(f"state {tag}", to_np(self.gpu.state)[self.slots], self.orc.state[self.slots])


def test_b8_shape_all_rows():
    """d = 128, bf16, T = 16: every row, every snapshot, six steps."""
    pr = NrPair(dataclasses.replace(WL["b8"], name="b8_nr", B=4, H=8))
    for s in range(6):
        pr.step(s)


def test_decode24_layer_sampled_rows():
    """The decode24 layer at full size on the GPU (B = 32, H = 16); the oracle
    follows four of the batch rows."""
    pr = NrPair(WL["decode24"], layer=23, rows=[0, 7, 19, 31])
    for s in range(3):
        pr.step(s)


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("b8", dict(B=3, H=2, dv=64)),
                                     ("b8", dict(B=3, H=2, dk=64)),
                                     ("b8", dict(B=2, H=2, T=64)),
                                     ("tiny", dict(B=3, H=3, dk=128, dv=128, T=33))])
def test_other_shapes(name, kw):
    """fp32 inputs at d = 64, mixed d_k / d_v, the longest draft (T = 64: 74 KB of
    shared memory), an odd T."""
    wl = dataclasses.replace(WL[name], name=f"{name}_nr", **kw)
    pr = NrPair(wl)
    for s in range(2):
        pr.step(s)


def test_status_bits_rejection_and_guard_bands():
    import speculative_decode_recurrent_gb300 as lib
    wl = dataclasses.replace(WL["b8"], name="b8_nr_st", B=3, H=2)
    init = synth.initial_layer(wl, 0)
    n_slot = init["state"].shape[0]
    d = _dims(wl, 3, n_slot)
    n_state = n_slot * wl.H * wl.dv * wl.dk
    n_snap = 3 * wl.H * wl.T * wl.dv * wl.dk
    guard = 4096
    state = torch.full((n_state + guard,), 7.0, device="cuda")
    state[:n_state] = init["state"].reshape(-1).cuda()
    snap = torch.full((n_snap + guard,), -3.0, device="cuda")
    idx = torch.tensor([int(init["state_idx"][0]), n_slot + 2, int(init["state_idx"][2])],
                       dtype=torch.int32, device="cuda")                          # row 1: no such slot
    blk = {n: t.cuda() for n, t in synth.draft_block(wl, 0, 0).items()}
    out = torch.full((3 * wl.T * wl.H * wl.dv + guard,), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gdn_nonreplay_verify(d, state, idx, blk["q"], blk["k"], blk["v"], blk["g"], blk["beta"],
                             out, snap, status)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.STATUS_BAD_SLOT
    o = out[:3 * wl.T * wl.H * wl.dv].view(3, wl.T, wl.H, wl.dv)
    assert torch.isnan(o[1]).all() and not torch.isnan(o[0]).any() and not torch.isnan(o[2]).any()
    sv = snap[:n_snap].view(3, wl.H, wl.T, wl.dv, wl.dk)
    assert (sv[1] == -3.0).all()                                                  # the skipped row
    assert torch.isnan(out[-guard:]).all() and (snap[-guard:] == -3.0).all() and (state[-guard:] == 7.0).all()
    before = state.clone()
    status.zero_()
    lib.gdn_nonreplay_accept(d, state, idx, snap, torch.tensor([wl.T + 1, 3, -1], dtype=torch.int32,
                                                                device="cuda"), status)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.STATUS_BAD_ACCEPT | lib.STATUS_BAD_SLOT
    assert torch.equal(state, before)                                             # nothing restored
    status.zero_()
    lib.gdn_nonreplay_accept(d, state, idx, snap, torch.tensor([0, 0, wl.T], dtype=torch.int32,
                                                                device="cuda"), status)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.STATUS_BAD_SLOT
    sl0, sl2 = int(idx[0]), int(idx[2])
    st = state[:n_state].view(n_slot, wl.H, wl.dv, wl.dk)
    bt = before[:n_state].view(n_slot, wl.H, wl.dv, wl.dk)
    assert torch.equal(st[sl0], bt[sl0])                                          # p = 0: unchanged
    assert torch.equal(st[sl2], sv[2, :, wl.T - 1])                               # p = T: the last state
    others = [s for s in range(n_slot) if s not in (sl0, sl2)]
    assert torch.equal(st[others], bt[others]) and (state[-guard:] == 7.0).all()
