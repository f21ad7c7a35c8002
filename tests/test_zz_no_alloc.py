"""The baseline step that allocates nothing (gdn_nonreplay_step_static), for callers
that can hand the library their tensors but cannot call cudaMalloc themselves -- a
plugin in a serving engine that reserves all device memory up front through its own
allocator, or a loop that may not pay cudaMalloc's implicit device synchronisation.
It must give what gdn_nonreplay_verify + gdn_nonreplay_accept give with a
caller-allocated snapshot area, call after call, although every call reuses the one
area inside the library.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import ctypes
import dataclasses

import pytest
import torch

import synth
import synth.workloads
from harness import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def _dims(lib, wl):
    return lib.Dims(B=wl.B, H=wl.H, dk=wl.dk, dv=wl.dv, T=wl.T, cap=wl.T, threshold=1,
                    n_slot=wl.n_slot, in_dtype=lib.DTYPE_BF16, scale=wl.scale)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_step_matches_the_allocating_calls_twice_in_a_row():
    import speculative_decode_recurrent_gb300 as lib
    so = lib.load()
    wl = dataclasses.replace(synth.WORKLOADS["b8"], name="b8_static", B=2, H=16)   # 32 MiB: the whole area
    d = _dims(lib, wl)
    assert wl.B * wl.H * wl.T * wl.dv * wl.dk * 4 == 32 << 20
    init = synth.initial_layer(wl, 0)
    ref = lib.NonReplayLayer(d, init["state"], init["state_idx"])                   # torch-allocated snapshots
    state = init["state"].cuda().contiguous()
    idx = init["state_idx"].cuda().contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for s in range(2):
        blk = {n: t.cuda() for n, t in synth.draft_block(wl, 0, s).items()}
        acc = synth.workloads.accepted_counts(wl, 0, s).cuda()
        out_ref = torch.empty(wl.B, wl.T, wl.H, wl.dv, device="cuda")
        ref.verify(blk["q"], blk["k"], blk["v"], blk["g"], blk["beta"], out_ref)
        ref.accept(acc)
        out = torch.full((wl.B, wl.T, wl.H, wl.dv), float("nan"), device="cuda")
        rc = so.gdn_nonreplay_step_static(ctypes.byref(d), _p(state), _p(idx), _p(blk["q"]), _p(blk["k"]),
                                          _p(blk["v"]), _p(blk["g"]), _p(blk["beta"]), _p(acc), _p(out),
                                          _p(status), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, lib.gdn_replay_strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(ref.status.item()) == 0
        assert_close(f"static out step{s}", to_np(out), to_np(out_ref))
        assert_close(f"static state step{s}", to_np(state), to_np(ref.state))


def test_static_step_rejects_steps_beyond_its_area():
    import speculative_decode_recurrent_gb300 as lib
    so = lib.load()
    big = dataclasses.replace(synth.WORKLOADS["b8"], name="b8_static_big", B=3, H=16)  # 48 MiB of snapshots
    fake = ctypes.c_void_p(0x10000)                     # never dereferenced: the size check comes first
    assert so.gdn_nonreplay_step_static(ctypes.byref(_dims(lib, big)), *([fake] * 10), None) == -2
