"""The identity slot map: every entry point takes state_idx = NULL to mean that
sequence b owns slot b (include/gdnreplay.h, include/gdnlayer.h,
include/gdnnonreplay.h).  The GPU runs with NULL and the oracle with the explicit map
0 .. B-1, on the seeded inputs of each workload with its slots rearranged so that
sequence b's data sits in slot b; the slots past B belong to no sequence and must stay
as they were.  Tolerances and exact comparisons as in the other parity tests."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads
from harness import Pair, assert_close, gpu_dims, oracle_dims, to_np
from synth.layer_ops import CONV_WORKLOADS, initial_conv_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def _slot_order(state_idx, n_slot):
    used = state_idx.long()
    rest = torch.tensor([s for s in range(n_slot) if s not in set(used.tolist())], dtype=torch.long)
    return torch.cat([used, rest])


def _identity_replay_init(wl, layer):
    init = synth.initial_layer(wl, layer)
    order = _slot_order(init["state_idx"], init["state"].shape[0])
    out = {n: init[n][order].contiguous() for n in ("state", "buf_k", "buf_v", "buf_g", "buf_beta", "buf_len")}
    out["state_idx"] = torch.arange(wl.B, dtype=torch.int32)
    return out


class IdentityPair(Pair):
    """Pair whose GPU layer passes state_idx = NULL."""

    def __init__(self, wl, layer=0):
        import speculative_decode_recurrent_gb300 as lib
        self.wl, self.layer, self.B, self.device = wl, layer, wl.B, "cuda"
        init = _identity_replay_init(wl, layer)
        self.gd, self.od = gpu_dims(wl), oracle_dims(wl)
        self.gpu = lib.ReplayLayer(self.gd, dict(init, state_idx=None), "cuda")
        self.orc = oracle.Layer(self.od, init)


@pytest.mark.parametrize("name", ["b8", "edge", "tiny"])
def test_three_call_steps_with_the_identity_map(name):
    """tcgen05 kernels at buffers up to 48 and 80 tokens (b8, edge), per-token kernels
    (tiny): verify -> accept -> flush."""
    pr = IdentityPair(synth.WORKLOADS[name])
    for s in range(6):
        pr.step(s)


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_fused_steps_with_the_identity_map(name):
    """verify_fold (fold launch beside the verify of the other sequences) -> accept_fold."""
    pr = IdentityPair(synth.WORKLOADS[name])
    for s in range(6):
        pr.fused_step(s)


def test_nonreplay_with_the_identity_map():
    import speculative_decode_recurrent_gb300 as lib
    wl = dataclasses.replace(synth.WORKLOADS["b8"], name="b8_nr_id", B=3, H=4)
    init = _identity_replay_init(wl, 0)
    n_slot = init["state"].shape[0]
    d = lib.Dims(B=wl.B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.T, threshold=1, n_slot=n_slot,
                 in_dtype=lib.DTYPE_BF16, scale=wl.scale)
    gpu = lib.NonReplayLayer(d, init["state"], None)
    orc = oracle.NonReplayLayer(oracle.Dims(B=wl.B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.T,
                                            threshold=1, n_slot=n_slot, scale=wl.scale, n_threads=8),
                                init["state"].double().numpy(), init["state_idx"].numpy())
    for s in range(3):
        blk = synth.draft_block(wl, 0, s)
        acc = synth.workloads.accepted_counts(wl, 0, s)
        dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty(wl.B, wl.T, wl.H, wl.dv, device="cuda")
        gpu.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
        gpu.accept(acc.cuda())
        o_ref = orc.verify({n: blk[n].double().numpy() for n in ("q", "k", "v", "g", "beta")})
        orc.accept(acc.numpy())
        torch.cuda.synchronize()
        assert int(gpu.status.item()) == 0 and int(orc.status[0]) == 0
        assert_close(f"nr out step{s}", to_np(out), o_ref)
        assert_close(f"nr state step{s}", to_np(gpu.state), orc.state)
        np.testing.assert_array_equal(to_np(gpu.state)[wl.B:], init["state"].double().numpy()[wl.B:])


def test_conv_with_the_identity_map():
    """Causal convolution verify -> accept; fp32 outputs within the arithmetic's band
    (2^-20 of the sum of the absolute terms), ring bytes and positions exact."""
    import speculative_decode_recurrent_gb300 as lib
    from test_gpu_layer_ops import _dims
    from synth.layer_ops import conv_block
    wl = dataclasses.replace(CONV_WORKLOADS["conv_edge"], out_dtype="fp32")
    init = initial_conv_layer(wl, 0)
    order = _slot_order(init["state_idx"], wl.n_slot)
    init = dict(init, ring=init["ring"][order].contiguous(), pos=init["pos"][order].contiguous(),
                state_idx=torch.arange(wl.B, dtype=torch.int32))
    gpu = lib.ConvLayer(_dims(wl), dict(init, state_idx=None))
    orc = oracle.ConvLayer(oracle.ConvDims(B=wl.B, D=wl.D, W=wl.W, T=wl.T, cap=wl.cap, n_slot=wl.n_slot,
                                           act=wl.act), init)
    for s in range(8):
        blk = conv_block(wl, 0, s)
        y = torch.empty(wl.B, wl.T, wl.D, device="cuda")
        xs = blk["x"].double().numpy()
        S = np.zeros((wl.B, wl.T, wl.D))                  # the band, before the ring moves
        for b in range(wl.B):
            win = [orc.ring[b, (orc.pos[b] - (wl.W - 1) + j) % wl.cap] for j in range(wl.W - 1)]
            seq = np.concatenate([np.array(win).reshape(wl.W - 1, wl.D), xs[b]], 0)
            for t in range(wl.T):
                S[b, t] = np.abs(orc.bias) + sum(np.abs(orc.w[:, j] * seq[t + j]) for j in range(wl.W))
        gpu.verify(blk["x"].cuda(), y)
        y_ref = orc.verify(blk["x"])
        gpu.accept(blk["accepted"].cuda())
        orc.accept(blk["accepted"].numpy())
        torch.cuda.synchronize()
        err = np.abs(y.cpu().double().numpy() - y_ref)
        assert (err <= 2.0 ** -20 * S + 1e-7).all(), f"step {s}"
        np.testing.assert_array_equal(gpu.t["pos"].cpu().numpy(), orc.pos)
        np.testing.assert_array_equal(gpu.t["ring"].cpu().double().numpy(), orc.ring)
        assert int(gpu.status.item()) == int(orc.status[0]) == 0
