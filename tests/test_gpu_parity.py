"""GPU parity: libgdnreplay (through its C ABI) against the CPU oracle on the
same seeded inputs.  Outputs and flushed state within
max|d| <= 2e-3 max|ref| + 1e-5 per tensor per (layer, step); lengths, status
words and buffer contents bit-exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import Pair, assert_close, to_np

pytestmark = pytest.mark.gpu
WL = synth.WORKLOADS


@pytest.fixture(autouse=True)
def _gpu(cuda_ok):
    yield


def test_tiny_verify_accept_forced_flush():
    """The tiny workload: B=1, H=2, d=64, T=4, fp32 inputs, 3 buffered tokens,
    one verify, a seeded accept in [0, 4], then a forced flush."""
    Pair(WL["tiny"]).step(0)


@pytest.mark.parametrize("p", [0, 1, 2, 3, 4])
def test_tiny_every_accept_count(p):
    Pair(WL["tiny"]).step(0, accepted=[p])


def test_b8_multistep():
    pr = Pair(WL["b8"])
    for s in range(12):
        pr.step(s)


def test_edge_multistep_extreme_gates_and_forced_accepts():
    """Forced accepts {0,1,8,15,16}, g in {0,-20}, beta near 0 and 1, threshold 64."""
    pr = Pair(WL["edge"])
    for s in range(12):
        pr.step(s)


@pytest.mark.parametrize("layer", [0, 23])
def test_decode24_layers_first_and_last(layer):
    pr = Pair(WL["decode24"], layer=layer)
    for s in range(6):
        pr.step(s)


@pytest.mark.parametrize("form", ["three_call", "fused"])
def test_large_batch_sampled_rows(form):
    """B=128, H=32, T=8 on the GPU at full size for 24 steps (every sampled sequence
    folds at least twice), three-call or fused; the oracle recomputes 12 of the
    sequences (they are independent) for every checked tensor."""
    wl = WL["large"]
    import speculative_decode_recurrent_gb300 as lib
    init = synth.initial_layer(wl, 0)
    from harness import gpu_dims, oracle_dims
    gd = gpu_dims(wl)
    gpu = lib.ReplayLayer(gd, init)
    sample = np.array([0, 1, 9, 23, 37, 50, 64, 77, 90, 100, 111, 127])
    sub = dict(init)
    sub["state_idx"] = init["state_idx"][sample]
    od = oracle_dims(wl, B=len(sample), n_slot=gd.n_slot)
    orc = oracle.Layer(od, sub)
    folds = np.zeros(len(sample), np.int64)
    for s in range(24):                                   # ~3 folds per sequence (T=8, threshold 32)
        blk = synth.draft_block(wl, 0, s)
        dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
        out = torch.empty(wl.B, wl.T, wl.H, wl.dv, device="cuda")
        sblk = {n: blk[n][sample] for n in ("q", "k", "v", "g", "beta")}
        slots = init["state_idx"][sample].long().numpy()
        if form == "three_call":
            gpu.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
            o_ref = orc.verify(sblk)
            gpu.accept(blk["accepted"].cuda())
            orc.accept(blk["accepted"][sample].numpy())
            before = orc.buf_len[slots].copy()
            gpu.flush()
            orc.flush()
            folds += orc.buf_len[slots] < before
        else:
            gpu.verify_fold(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
            gpu.accept_fold(blk["accepted"].cuda())
            before = orc.buf_len[slots].copy()
            orc.flush()
            folds += orc.buf_len[slots] < before
            o_ref = orc.verify(sblk)
            orc.accept(blk["accepted"][sample].numpy())
        torch.cuda.synchronize()
        assert_close(f"out step{s}", to_np(out)[sample], o_ref)
        assert_close(f"state step{s}", to_np(gpu.t["state"])[slots], orc.state[slots])
        np.testing.assert_array_equal(gpu.t["buf_len"].cpu().numpy()[slots], orc.buf_len[slots])
        assert int(gpu.status.item()) == 0
    assert folds.min() >= 2, folds


# ------------------------------------------------------------ exact invariants
def _one_verify(pr, step=0):
    wl = pr.wl
    blk = pr.block(step)
    dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    out = torch.empty(pr.B, wl.T, wl.H, wl.dv, device="cuda")
    pr.gpu.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
    return out, blk


def test_verify_is_pure_and_repeatable():
    pr = Pair(WL["b8"])
    st0 = pr.gpu.t["state"].clone()
    ln0 = pr.gpu.t["buf_len"].clone()
    o1, _ = _one_verify(pr)
    o2, _ = _one_verify(pr)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    assert torch.equal(pr.gpu.t["state"], st0)
    assert torch.equal(pr.gpu.t["buf_len"], ln0)


def test_full_rejection_is_bit_identical():
    pr = Pair(WL["b8"])
    t = pr.gpu.t
    st0, ln0, bk0 = t["state"].clone(), t["buf_len"].clone(), t["buf_k"].clone()
    _one_verify(pr)
    pr.gpu.accept(torch.zeros(pr.B, dtype=torch.int32, device="cuda"))
    pr.gpu.flush(force=False)
    torch.cuda.synchronize()
    assert torch.equal(t["state"], st0)
    assert torch.equal(t["buf_len"], ln0)
    for s in range(t["buf_len"].numel()):
        L = int(ln0[s])
        assert torch.equal(t["buf_k"][s, :, :L], bk0[s, :, :L])
    assert int(pr.gpu.status.item()) == 0


def test_flush_empty_noop_and_idempotent():
    pr = Pair(WL["b8"])
    t = pr.gpu.t
    t["buf_len"].zero_()
    st0 = t["state"].clone()
    pr.gpu.flush(force=True)
    torch.cuda.synchronize()
    assert torch.equal(t["state"], st0)
    t["buf_len"].fill_(5)
    pr.gpu.flush(force=True)
    torch.cuda.synchronize()
    st1 = t["state"].clone()
    assert (t["buf_len"][pr.gpu.t["state_idx"].long()] == 0).all()
    pr.gpu.flush(force=True)
    torch.cuda.synchronize()
    assert torch.equal(t["state"], st1)


def test_status_bits_without_trap():
    """Bad accepted counts and a full buffer are reported in the status word;
    the affected sequences are skipped and nothing traps."""
    pr = Pair(WL["b8"])
    t = pr.gpu.t
    idx = t["state_idx"].long()
    t["buf_len"][idx[0]] = pr.wl.cap - pr.wl.T + 1          # no room for the draft
    out, _ = _one_verify(pr)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == 2
    pr.gpu.status.zero_()
    ln0 = t["buf_len"].clone()
    acc = torch.tensor([-1, pr.wl.T + 1] + [0] * (pr.B - 2), dtype=torch.int32, device="cuda")
    pr.gpu.accept(acc)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == 1
    assert torch.equal(t["buf_len"], ln0)
    pr.gpu.status.zero_()
    t["buf_len"][idx[1]] = pr.wl.cap + 3                    # corrupt length
    pr.gpu.flush(force=False)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) & 4


def test_guard_bands_untouched():
    """Every written tensor gets a NaN tail; the kernels must never touch it."""
    import speculative_decode_recurrent_gb300 as lib
    wl = WL["edge"]
    init = synth.initial_layer(wl, 0)
    from harness import gpu_dims
    d = gpu_dims(wl)
    pad = 4096

    def padded(t):
        flat = torch.full((t.numel() + pad,), float("nan"), dtype=t.dtype, device="cuda") \
            if t.dtype.is_floating_point else torch.full((t.numel() + pad,), -7, dtype=t.dtype,
                                                          device="cuda")
        flat[:t.numel()] = t.reshape(-1).cuda()
        return flat, flat[:t.numel()].view(t.shape)

    names = ("state", "buf_k", "buf_v", "buf_g", "buf_beta", "buf_len")
    store = {n: padded(init[n]) for n in names}
    t = {n: store[n][1] for n in names}
    t["state_idx"] = init["state_idx"].cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(4):
        blk = synth.draft_block(wl, 0, s)
        out_flat, out = padded(torch.zeros(wl.B, wl.T, wl.H, wl.dv))
        dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
        lib.gdn_replay_verify(d, t["state"], t["state_idx"], t["buf_k"], t["buf_v"], t["buf_g"],
                              t["buf_beta"], t["buf_len"], dev["q"], dev["k"], dev["v"], dev["g"],
                              dev["beta"], out, status)
        lib.gdn_replay_accept(d, t["buf_len"], t["state_idx"], blk["accepted"].cuda(), status)
        lib.gdn_replay_flush(d, t["state"], t["state_idx"], t["buf_k"], t["buf_v"], t["buf_g"],
                             t["buf_beta"], t["buf_len"], 0, status)
        torch.cuda.synchronize()
        assert torch.isnan(out_flat[out.numel():].float()).all()
        for n in names:
            tail = store[n][0][init[n].numel():]
            if tail.dtype.is_floating_point:
                assert torch.isnan(tail.float()).all(), n
            else:
                assert (tail == -7).all(), n
    assert int(status.item()) == 0


def test_default_stream_and_side_stream_agree():
    pr1, pr2 = Pair(WL["b8"]), Pair(WL["b8"])
    o1, _ = _one_verify(pr1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, _ = _one_verify(pr2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_checkpoint_resume_bit_identical():
    """State + buffer + lengths are the resumable unit: saving them to the host
    and restoring them continues bit-identically."""
    import speculative_decode_recurrent_gb300 as lib
    wl = WL["b8"]
    init = synth.initial_layer(wl, 0)
    from harness import gpu_dims
    d = gpu_dims(wl)
    a = lib.ReplayLayer(d, init)
    for s in range(3):
        _step_layer(a, wl, s)
    snap = {n: v.cpu().clone() for n, v in a.t.items()}
    b = lib.ReplayLayer(d, snap)
    for s in range(3, 6):
        oa = _step_layer(a, wl, s)
        ob = _step_layer(b, wl, s)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
    for n in a.t:
        assert torch.equal(a.t[n], b.t[n]), n


def _step_layer(layer, wl, s):
    blk = synth.draft_block(wl, 0, s)
    dev = {n: blk[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    out = torch.empty(wl.B, wl.T, wl.H, wl.dv, device="cuda")
    layer.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], out)
    layer.accept(blk["accepted"].cuda())
    layer.flush()
    return out


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_forced_flush_folds_short_buffers(name):
    """flush(force=True) folds every non-empty buffer whatever its length: the first
    step folds 0 .. 47 tokens (initial lengths 0..31 plus the accepted counts), every
    later one 1..16 (edge: also 0, nothing to fold), so the tensor-core fold runs on
    short and partial token blocks; checkpoint, buffer, lengths and outputs against the
    oracle at every step."""
    pr = Pair(WL[name])
    for s in range(6):
        pr.step(s, force=True)


@pytest.mark.parametrize("T", [1, 3, 11])
def test_short_drafts_on_the_tensor_cores(T):
    """Draft blocks of 1, 3 and 11 tokens (the tensor-core kernels take T <= 16; one
    token is the degenerate verify, W a single row), three-call then fused, 8 steps each."""
    import speculative_decode_recurrent_gb300 as lib
    wl = dataclasses.replace(WL["b8"], name=f"b8_T{T}", B=4, H=4, T=T)
    pr = Pair(wl)
    assert lib.gdn_replay_kernel_family(pr.gd) == lib.FAMILY_TCGEN05
    for s in range(8):
        pr.step(s)
    pr = Pair(wl)
    for s in range(8):
        pr.fused_step(s)


def test_one_sequence_odd_heads_on_the_tensor_cores():
    """B = 1, H = 3: in the fused steps where the only sequence folds, every CTA of the
    verify launch beside the fold launch has nothing to do and leaves at once (its CTA
    (0, 0) still waits for the fold launch); 12 steps three-call, 12 fused."""
    wl = dataclasses.replace(WL["b8"], name="b1_h3", B=1, H=3)
    pr = Pair(wl)
    for s in range(12):
        pr.step(s)
    pr = Pair(wl)
    folded = 0
    for s in range(12):
        before = int(pr.gpu.t["buf_len"][pr.gpu.t["state_idx"][0]].item())
        pr.fused_step(s)
        folded += before >= wl.threshold
    assert folded >= 2


@pytest.mark.parametrize("name,threshold", [("b8", 32), ("b8", 48), ("edge", 64), ("b8", 186)])
def test_length_boundaries(name, threshold):
    """Buffer lengths at the edges of each kernel variant (capacity = threshold + 15:
    47, 63, 79 tokens on the tensor cores; 201, the largest the per-token kernels take
    in the fused step at d = 128): a fused step from threshold - 1 (no fold; its verify takes
    the whole capacity), the threshold (folds), the capacity (a full buffer: folds) and
    0; then one where every sequence folds, so the verify launch beside the fold launch
    has nothing to do; a three-call step from threshold - 1, 0, 1 and 15."""
    wl = dataclasses.replace(WL[name], name=f"{name}_edges{threshold}", B=4, H=4, threshold=threshold)
    thr, cap = wl.threshold, wl.cap

    def set_lens(pr, vals):
        idx = pr.gpu.t["state_idx"].long().cpu()
        for b, v in enumerate(vals):
            pr.gpu.t["buf_len"][idx[b]] = v
            pr.orc.buf_len[int(idx[b])] = v

    assert cap == thr + 15
    pr = Pair(wl)
    set_lens(pr, [thr - 1, thr, cap, 0])
    pr.fused_step(0)
    set_lens(pr, [cap - 7, thr + 1, cap, thr])
    pr.fused_step(1)
    pr.fused_step(2)
    pr = Pair(wl)
    set_lens(pr, [thr - 1, 0, 1, 15])
    pr.step(3)
    pr.step(4)


def test_pertoken_largest_shape():
    """The per-token kernels at their largest shape: d = 64, T = 64, capacity 256
    (threshold 193), fp32 inputs; a fused step from lengths 192 (its verify takes all
    256 slots) and 256 (a full buffer folds), then three-call steps with forced flushes
    from 192 and 0."""
    wl = dataclasses.replace(WL["tiny"], name="tiny_max", B=2, H=2, T=64, threshold=193,
                             forced_flush=False)
    assert wl.cap == 256

    def set_lens(pr, vals):
        idx = pr.gpu.t["state_idx"].long().cpu()
        for b, v in enumerate(vals):
            pr.gpu.t["buf_len"][idx[b]] = v
            pr.orc.buf_len[int(idx[b])] = v

    pr = Pair(wl)
    set_lens(pr, [192, 256])
    pr.fused_step(0)
    pr.fused_step(1)
    pr = Pair(wl)
    set_lens(pr, [192, 0])
    pr.step(2, force=True)
    pr.step(3, force=True)


def test_bad_slot_reported_not_dereferenced():
    pr = Pair(WL["b8"])
    pr.gpu.t["state_idx"][3] = pr.gd.n_slot + 100
    _one_verify(pr)
    pr.gpu.accept(torch.zeros(pr.B, dtype=torch.int32, device="cuda"))
    pr.gpu.flush(force=True)
    torch.cuda.synchronize()
    assert int(pr.gpu.status.item()) == 8


# --------------------------------------------- lazy flush: verify_fold + accept_fold
@pytest.mark.parametrize("name,steps", [("b8", 16), ("edge", 12), ("tiny", 1), ("large", 3)])
def test_fused_step_matches_flush_verify_accept(name, steps):
    """verify_fold -> accept_fold equals flush(threshold) -> verify -> accept of the
    oracle at every step (outputs, folded state, lengths, buffer bytes)."""
    wl = WL[name]
    if name == "large":
        pr = Pair(wl, B=16)
    else:
        pr = Pair(wl)
    for s in range(steps):
        pr.fused_step(s)


@pytest.mark.parametrize("layer", [0, 23])
def test_fused_decode24(layer):
    pr = Pair(WL["decode24"], layer=layer)
    for s in range(8):
        pr.fused_step(s)


def test_fused_then_three_call_interleave():
    """Both step forms keep the same buffer/length convention, so they can alternate."""
    pr = Pair(WL["b8"])
    for s in range(10):
        if s % 2:
            pr.fused_step(s)
        else:
            # the three-call step needs len < threshold before verify: flush first
            pr.gpu.flush(force=False)
            pr.orc.flush(force=False)
            pr.step(s)


def test_flush_many_sequences_list_chunks():
    """More sequences than the flush kernel lists at once (1024) and many
    (sequence, head) items per CTA: every flushed unit is folded exactly once."""
    import dataclasses
    import speculative_decode_recurrent_gb300 as lib
    from harness import gpu_dims, oracle_dims
    wl = dataclasses.replace(WL["b8"], name="b1100", B=1100, H=2)
    init = synth.initial_layer(wl, 0)
    init["buf_len"] = torch.where(init["buf_len"] > 0, torch.full_like(init["buf_len"], wl.threshold),
                                  init["buf_len"])            # every used slot flushes
    gd = gpu_dims(wl)
    gpu = lib.ReplayLayer(gd, init)
    gpu.flush(force=False)
    torch.cuda.synchronize()
    assert int(gpu.status.item()) == 0
    used = init["state_idx"].long()
    assert (gpu.t["buf_len"][used] == 0).all()
    sample = np.array([0, 5, 511, 1023, 1024, 1099])
    sub = dict(init)
    sub["state_idx"] = init["state_idx"][sample]
    od = oracle_dims(wl, B=len(sample), n_slot=gd.n_slot)
    orc = oracle.Layer(od, sub)
    orc.flush(force=False)
    slots = init["state_idx"][sample].long().numpy()
    assert_close("state", to_np(gpu.t["state"])[slots], orc.state[slots])


# --------------------------------------------- 64-token buffers (capacity 49..64)
def _cap63(name):
    import dataclasses
    return dataclasses.replace(WL[name], name=name + "_cap63", threshold=48)   # cap = 48 - 1 + 16 = 63


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_cap63_three_call(name):
    """Buffers of up to 63 tokens: the 64-token variants of the verify and of the
    fold (four 16-token blocks in the inverse)."""
    pr = Pair(_cap63(name))
    for s in range(14):
        pr.step(s)


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_cap63_fused(name):
    pr = Pair(_cap63(name))
    for s in range(14):
        pr.fused_step(s)


# ----------------------- short drafts over long buffers (more than 32 buffered rows)
def _short_draft(name):
    import dataclasses
    # cap = 40 - 1 + 8 = 47; accepted counts drawn uniformly in [0, 8]
    return dataclasses.replace(WL[name], name=name + "_t8", T=8, threshold=40, accept_law="uniform")


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_short_draft_long_buffer_three_call(name):
    """T = 8 with buffers of up to 39 tokens: rows past the 32 a thread keeps in
    registers are loaded on a second pass."""
    pr = Pair(_short_draft(name))
    for s in range(14):
        pr.step(s)


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_short_draft_long_buffer_fused(name):
    pr = Pair(_short_draft(name))
    for s in range(14):
        pr.fused_step(s)


# ------------- the per-token kernels at d = 128, bf16 (T = 17 is past the tcgen05 shapes)
def _t17(name):
    import dataclasses
    return dataclasses.replace(WL[name], name=name + "_t17", T=17)


@pytest.mark.parametrize("name", ["b8", "edge"])
def test_pertoken_family_bf16_d128_three_call(name):
    import speculative_decode_recurrent_gb300 as lib
    pr = Pair(_t17(name))
    assert lib.gdn_replay_kernel_family(pr.gd) == lib.FAMILY_PERTOKEN
    for s in range(8):
        pr.step(s)


def test_pertoken_family_bf16_d128_fused():
    pr = Pair(_t17("b8"))
    for s in range(8):
        pr.fused_step(s)
