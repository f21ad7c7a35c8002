"""Long-run GPU parity of the decode-loop sweep (24 GDN layers, B=32, H=16, d=128,
T=16, flush threshold 32), against the fp64 CPU oracle at every step:

* layers 0 and 23 over all 64 steps, in the three-call step (verify -> accept ->
  flush) and in the fused step (verify_fold -> accept_fold), so each sequence goes
  through 12-18 flushes and the error of the tf32 checkpoint contractions has that
  many chances to compound;
* the threshold-64 mix (buffers up to 79 tokens) and a threshold-48 B=8 layer (buffers
  up to 63 tokens) for 48 steps each, so the 80- and 64-token variants of both kernels
  fold every sequence several times;
* the overlapped schedule the benchmark times (verifies on the capturing stream,
  each layer's accept + flush on one of two side streams, captured in a CUDA graph)
  on three layers for 20 steps, every layer compared with its own oracle;
* the wait-expiry path of the tensor-core kernels, forced before anything is issued.

Tolerance as everywhere: max|d| <= 2e-3 max|ref| + 1e-5 per tensor per step; lengths,
status words and buffer bytes bit-exact.  Set GDN_PARITY_LOG to a file name to get
the per-step error ratios max|d| / max|ref| as JSON.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import DRIFT, Pair, assert_close, gpu_dims, oracle_dims, to_np

pytestmark = pytest.mark.gpu
WL = synth.WORKLOADS
_LOG = {}


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


@pytest.fixture(scope="module", autouse=True)
def _drift_log():
    yield
    path = os.environ.get("GDN_PARITY_LOG")
    if path and _LOG:
        with open(path, "w") as f:
            json.dump(_LOG, f, indent=1)


def _record(test, step):
    """Move the ratios appended since the last call into the log under (test, step)."""
    out = max((r for n, r in DRIFT if n.startswith("out")), default=0.0)
    st = max((r for n, r in DRIFT if n.startswith("state")), default=0.0)
    _LOG.setdefault(test, []).append({"step": step, "out": out, "state": st})
    DRIFT.clear()


def _folds(pr, lens_before):
    """Sequences whose buffer was folded in the step just taken (length went down)."""
    idx = pr.gpu.t["state_idx"].long()
    after = pr.gpu.t["buf_len"][idx].cpu().numpy()
    return int((after < lens_before).sum())


@pytest.mark.parametrize("form", ["three_call", "fused"])
@pytest.mark.parametrize("layer", [0, 23])
def test_decode24_all_64_steps(layer, form):
    wl = WL["decode24"]
    pr = Pair(wl, layer=layer)
    name = f"decode24_layer{layer}_{form}"
    DRIFT.clear()
    folds = np.zeros(wl.B, np.int64)
    idx = pr.gpu.t["state_idx"].long()
    for s in range(wl.steps):
        before = pr.gpu.t["buf_len"][idx].cpu().numpy()
        if form == "three_call":
            pr.step(s)
            after = pr.gpu.t["buf_len"][idx].cpu().numpy()
            folds += after < before + pr.block(s)["accepted"].numpy()
        else:
            pr.fused_step(s)
            folds += before >= wl.threshold
        _record(name, s)
    # every sequence went through many flushes: the run exercises the compounding
    assert folds.min() >= 10, folds
    _LOG[name + "_folds_per_sequence"] = [int(folds.min()), int(folds.max())]


@pytest.mark.parametrize("form", ["three_call", "fused"])
def test_edge_48_steps_long_buffers(form):
    """The threshold-64 mix (buffers of up to 79 tokens: the 80-token variants of both
    tensor-core kernels, tokens 64..79 in the second K atom), with extreme gates and
    the forced accepted counts, for 48 steps: every sequence folds several times."""
    wl = WL["edge"]
    pr = Pair(wl)
    name = f"edge_{form}"
    DRIFT.clear()
    idx = pr.gpu.t["state_idx"].long()
    folds = np.zeros(wl.B, np.int64)
    longest = 0
    for s in range(48):
        before = pr.gpu.t["buf_len"][idx].cpu().numpy()
        longest = max(longest, int(before.max()))
        if form == "three_call":
            pr.step(s)
            after = pr.gpu.t["buf_len"][idx].cpu().numpy()
            folds += after < before + pr.block(s)["accepted"].numpy()
        else:
            pr.fused_step(s)
            folds += before >= wl.threshold
        _record(name, s)
    assert folds.min() >= 3, folds
    assert longest + wl.T > 64, longest          # verifies over more than 64 tokens happened
    _LOG[name + "_folds_per_sequence"] = [int(folds.min()), int(folds.max())]


@pytest.mark.parametrize("form", ["three_call", "fused"])
def test_cap63_48_steps(form):
    """B=8 with threshold 48 (buffers of up to 63 tokens: the 64-token variants of both
    tensor-core kernels, four 16-token blocks in the inverse) for 48 steps."""
    import dataclasses
    wl = dataclasses.replace(WL["b8"], name="b8_cap63_long", threshold=48)
    pr = Pair(wl)
    name = f"cap63_{form}"
    DRIFT.clear()
    idx = pr.gpu.t["state_idx"].long()
    folds = np.zeros(wl.B, np.int64)
    longest = 0
    for s in range(48):
        before = pr.gpu.t["buf_len"][idx].cpu().numpy()
        longest = max(longest, int(before.max()))
        if form == "three_call":
            pr.step(s)
            after = pr.gpu.t["buf_len"][idx].cpu().numpy()
            folds += after < before + pr.block(s)["accepted"].numpy()
        else:
            pr.fused_step(s)
            folds += before >= wl.threshold
        _record(name, s)
    assert folds.min() >= 3, folds
    assert longest + wl.T > 48, longest          # verifies over more than 48 tokens happened
    _LOG[name + "_folds_per_sequence"] = [int(folds.min()), int(folds.max())]


def test_overlapped_schedule_in_a_graph_matches_oracle():
    """The benchmark's headline schedule, replayed from one captured graph per step
    on three decode24 layers: every layer's outputs, state, lengths and buffer bytes
    against its own oracle after each step."""
    import speculative_decode_recurrent_gb300 as lib
    from speculative_decode_recurrent_gb300.schedule import StepSchedule
    wl = WL["decode24"]
    n_layers, steps = 3, 20
    pairs = [Pair(wl, layer=l) for l in range(n_layers)]
    dev = torch.device("cuda")
    names = ("q", "k", "v", "g", "beta")
    blk0 = [p.block(0) for p in pairs]
    stat = [{n: b[n].to(dev).clone() for n in names} for b in blk0]
    acc = [b["accepted"].to(dev).clone() for b in blk0]
    outs = [torch.empty(wl.B, wl.T, wl.H, wl.dv, device=dev) for _ in pairs]
    sched = StepSchedule([p.gpu for p in pairs], n_side=2, device=dev)
    cap = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            sched.enqueue_overlap(stat, acc, outs)
    DRIFT.clear()
    for s in range(steps):
        blks = [p.block(s) for p in pairs]
        with torch.cuda.stream(cap):
            for l, b in enumerate(blks):
                for n in names:
                    stat[l][n].copy_(b[n], non_blocking=False)
                acc[l].copy_(b["accepted"])
            graph.replay()
        cap.synchronize()
        for l, (p, b) in enumerate(zip(pairs, blks)):
            o_ref = p.orc.verify(b)
            p.orc.accept(b["accepted"].numpy())
            p.orc.flush(force=False)
            p.compare(outs[l], o_ref, s)
        _record("overlap_schedule_3_layers", s)
    for p in pairs:
        assert int(p.gpu.status.item()) == 0


def test_forced_wait_expiry_skips_the_unit_and_recovers():
    """GDN_FLAG_TEST_EXPIRE: the tensor-core kernels take their wait-expiry exit at the
    first bounded wait, before any copy or tensor-core operation is issued.  The status
    word reports GDN_STATUS_TIMEOUT (not GDN_STATUS_DRAIN: nothing was in flight), the
    outputs, checkpoint and committed buffer are untouched, no length is reset, and the
    next calls without the flag match the oracle again."""
    import speculative_decode_recurrent_gb300 as lib
    wl = WL["b8"]
    pr = Pair(wl)
    t = pr.gpu.t
    assert lib.gdn_replay_kernel_family(pr.gd) == lib.FAMILY_TCGEN05
    st0, ln0 = t["state"].clone(), t["buf_len"].clone()
    bk0 = t["buf_k"].clone()
    blk = pr.block(0)
    dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    sentinel = torch.full((wl.B, wl.T, wl.H, wl.dv), 7.25, device="cuda")
    dx = gpu_dims(wl)
    dx.flags = lib.FLAG_TEST_EXPIRE
    args = (t["state"], t["state_idx"], t["buf_k"], t["buf_v"], t["buf_g"], t["buf_beta"],
            t["buf_len"])
    # verify: every unit skipped
    lib.gdn_replay_verify(dx, *args, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                          sentinel, pr.gpu.status)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == lib.STATUS_TIMEOUT
    assert bool((sentinel == 7.25).all())
    assert torch.equal(t["state"], st0) and torch.equal(t["buf_len"], ln0)
    for sl in range(t["buf_len"].numel()):
        L = int(ln0[sl])
        assert torch.equal(t["buf_k"][sl, :, :L], bk0[sl, :, :L])
    # flush (every used buffer set to the threshold): nothing folded, no length reset
    pr.gpu.status.zero_()
    idx = t["state_idx"].long()
    t["buf_len"][idx] = wl.threshold
    ln1 = t["buf_len"].clone()
    lib.gdn_replay_flush(dx, *args, 0, pr.gpu.status)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == lib.STATUS_TIMEOUT
    assert torch.equal(t["state"], st0) and torch.equal(t["buf_len"], ln1)
    # the fused step: nothing folded, no length changed
    lib.gdn_replay_verify_fold(dx, *args, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                               sentinel, pr.gpu.status)
    lib.gdn_replay_accept_fold(dx, t["buf_len"], t["state_idx"], blk["accepted"].cuda(),
                               pr.gpu.status)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == lib.STATUS_TIMEOUT
    assert torch.equal(t["state"], st0) and torch.equal(t["buf_len"], ln1)
    # recovery: restore the lengths, clear the word, and run normal steps
    t["buf_len"].copy_(ln0)
    pr.gpu.status.zero_()
    torch.cuda.synchronize()
    for s in range(3):
        pr.step(s)
