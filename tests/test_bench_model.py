"""The byte model behind the bench's roofline fractions: the algorithmic HBM bytes of
one layer-step ("The inference stack behind OCRia", section "Making speculative
verification cheaper": the verify reads the checkpoint once and the buffered and
draft inputs, stages the draft and writes the outputs; the accept moves a length; a
flush reads and writes the checkpoint of every sequence whose buffer reached the
threshold, and reads that buffer).  Pinned against hand-counted single-unit cases and
against the per-layer total that the decode24 workload's means give (70.3 MB)."""
import dataclasses

import numpy as np
import pytest

import bench
import synth

WL = synth.WORKLOADS["decode24"]
ST = 128 * 128 * 4                  # one fp32 state [d_v, d_k]
TOK = (128 + 128) * 2 + 4 + 4       # one buffered token: bf16 key and value, fp32 g and beta
DRAFT_IN = 3 * 128 * 2 + 4 + 4      # one draft token read: bf16 q, k, v, fp32 g and beta
OUT = 128 * 4                       # one fp32 output row


def test_one_unit_without_a_flush():
    wl = dataclasses.replace(WL, B=1, H=1)
    v, a, f, new, n_tok = bench.bytes_model(wl, np.array([10]), np.array([5]))
    assert v == ST + 10 * TOK + 16 * DRAFT_IN + 16 * TOK + 16 * OUT
    assert a == 12                  # accepted count, slot and length
    assert f == 8                   # the length read and written back, no fold
    assert new.tolist() == [15] and n_tok == 0


def test_a_flush_reads_and_writes_the_state_once_per_head():
    wl = dataclasses.replace(WL, B=2, H=3)
    v, a, f, new, n_tok = bench.bytes_model(wl, np.array([20, 3]), np.array([16, 2]))
    assert v == 3 * (2 * ST + 23 * TOK + 2 * 16 * (DRAFT_IN + TOK + OUT))
    assert f == 3 * (2 * ST + 36 * TOK) + 2 * 8          # sequence 0 reaches 36 >= 32
    assert new.tolist() == [0, 5] and n_tok == 36


def test_the_fused_step_adds_one_state_write_per_folded_head():
    wl = dataclasses.replace(WL, B=2, H=3)
    lens, acc = np.array([34, 3]), np.array([7, 1])
    v3, _, _, _, _ = bench.bytes_model(wl, lens, np.zeros(2, np.int64))
    vf, a, new, n_folded = bench.bytes_model_fused(wl, lens, acc)
    assert vf == v3 + 3 * ST and n_folded == 1
    assert new.tolist() == [7, 4]                        # folded: 0 + 7; the other: 3 + 1


def test_decode24_means_give_the_per_layer_total():
    """Fed the workload's realised means (flush fraction 0.241, mean length 12.7 before
    the verify, mean flushed length 37.4), the model's terms are the per-layer-step
    byte budget of the decode24 workload: 70.3 MB."""
    B, H, T = WL.B, WL.H, WL.T
    verify = H * (B * ST + TOK * B * 12.7 + B * T * (DRAFT_IN + TOK + OUT))
    flush = H * (2 * ST * B * 0.241 + TOK * B * 0.241 * 37.4)
    assert verify + flush == pytest.approx(70.3e6, rel=2e-3)


def test_decode24_simulated_steps_stay_near_the_budget():
    """The bench's own accounting (initial lengths, cycled accept patterns) over 64 steps
    of four layers: the mean layer-step moves 70.3 MB within 3 %, and about a quarter of
    the sequences flush per step."""
    total, flushed, n = 0.0, 0, 0
    for layer in range(4):
        init = synth.initial_layer(WL, bench.layer_seed(layer, 0))
        lens = init["buf_len"][init["state_idx"].long()].numpy().astype(np.int64)
        pats = [bench._accept_pattern(WL, bench.layer_seed(layer, 0), j) for j in range(bench.ACCEPT_PERIOD)]
        for s in range(64):
            acc = pats[s % bench.ACCEPT_PERIOD]
            v, a, f, new, _ = bench.bytes_model(WL, lens, acc)
            flushed += int(((lens + acc) >= WL.threshold).sum())
            total += v + a + f
            n += 1
            lens = new
    assert total / n == pytest.approx(70.3e6, rel=0.03)
    assert 0.20 <= flushed / (n * WL.B) <= 0.28
