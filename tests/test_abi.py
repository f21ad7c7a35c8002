"""The C-ABI library builds, loads and exports every declared symbol, and its
host-side validation rejects bad arguments before anything is launched.
No test here launches a kernel, so they all run without a GPU."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decode_recurrent_gb300 as lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gdn_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gdn_replay_verify", "gdn_replay_accept", "gdn_replay_flush", "gdn_replay_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol():
    so = lib.load()
    for n in declared_functions():
        assert hasattr(so, n), f"missing export {n}"


def test_dims_struct_layout():
    assert ctypes.sizeof(lib.Dims) == 44
    assert lib.Dims.scale.offset == 36
    assert lib.Dims.flags.offset == 40


def test_kernel_family_query():
    """Host-only: which kernels the dims select, and loud rejection of bad dims."""
    so = lib.load()
    tc = good_dims(T=16, cap=47, threshold=32)
    assert so.gdn_replay_kernel_family(ctypes.byref(tc)) == lib.FAMILY_TCGEN05
    for cap in (16, 48, 49, 64, 65, 79, 80):                   # the three token-capacity variants
        d = good_dims(T=16, cap=cap, threshold=1)
        assert so.gdn_replay_kernel_family(ctypes.byref(d)) == lib.FAMILY_TCGEN05, cap
    for kw in (dict(dk=64, dv=64), dict(in_dtype=lib.DTYPE_F32), dict(T=17, cap=48, threshold=32),
               dict(cap=81, threshold=32)):
        d = good_dims(**kw)
        assert so.gdn_replay_kernel_family(ctypes.byref(d)) == lib.FAMILY_PERTOKEN, kw
    assert so.gdn_replay_kernel_family(ctypes.byref(good_dims(dk=96))) == -2
    assert so.gdn_replay_kernel_family(None) == -1
    assert lib.gdn_replay_kernel_family(tc) == lib.FAMILY_TCGEN05


@pytest.mark.parametrize("flags", [2, 1 << 30, -1])
def test_unknown_flags_rejected(flags):
    so = lib.load()
    d = good_dims(flags=flags)
    assert so.gdn_replay_verify(ctypes.byref(d), *([FAKE] * 14), None) == -2
    assert so.gdn_replay_flush(ctypes.byref(d), *([FAKE] * 7), 0, FAKE, None) == -2
    assert so.gdn_replay_kernel_family(ctypes.byref(d)) == -2


def good_dims(**kw):
    d = dict(B=2, H=2, dk=128, dv=128, T=4, cap=8, threshold=4, n_slot=2, in_dtype=lib.DTYPE_BF16,
             scale=128 ** -0.5)
    d.update(kw)
    return lib.Dims(**d)


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


@pytest.mark.parametrize("kw,code", [
    (dict(dk=96), -2), (dict(dv=32), -2), (dict(T=0), -2), (dict(T=65), -2),
    (dict(cap=3), -2), (dict(cap=257), -2), (dict(threshold=0), -2), (dict(threshold=9), -2),
    (dict(n_slot=1), -2), (dict(H=0), -2), (dict(B=-1), -2), (dict(in_dtype=7), -3),
])
def test_bad_dims_rejected_before_launch(kw, code):
    so = lib.load()
    d = good_dims(**kw)
    assert so.gdn_replay_verify(ctypes.byref(d), *([FAKE] * 14), None) == code
    assert so.gdn_replay_accept(ctypes.byref(d), FAKE, None, FAKE, FAKE, None) == code
    assert so.gdn_replay_flush(ctypes.byref(d), *([FAKE] * 7), 0, FAKE, None) == code


def test_pertoken_shared_memory_capacity():
    """The per-token kernels hold the buffer and the draft in shared memory: at
    dk = dv = 128 and T = 16 they take buffers of up to 217 tokens; at d = 64 the whole
    range up to 256 (even with T = 64)."""
    so = lib.load()
    ok = good_dims(T=16, cap=217, threshold=200)
    assert so.gdn_replay_kernel_family(ctypes.byref(ok)) == lib.FAMILY_PERTOKEN
    big = good_dims(T=16, cap=218, threshold=200)
    assert so.gdn_replay_kernel_family(ctypes.byref(big)) == -2
    assert so.gdn_replay_verify(ctypes.byref(big), *([FAKE] * 14), None) == -2
    d64 = good_dims(dk=64, dv=64, T=64, cap=256, threshold=200)
    assert so.gdn_replay_kernel_family(ctypes.byref(d64)) == lib.FAMILY_PERTOKEN


def test_fold_entry_points_validate():
    so = lib.load()
    d = good_dims(threshold=6)                 # threshold - 1 + T = 9 > cap = 8
    assert so.gdn_replay_verify_fold(ctypes.byref(d), *([FAKE] * 14), None) == -2
    d = good_dims()
    assert so.gdn_replay_verify_fold(None, *([FAKE] * 14), None) == -1
    assert so.gdn_replay_accept_fold(ctypes.byref(d), None, None, FAKE, FAKE, None) == -1
    e = good_dims(B=0, n_slot=0)
    assert so.gdn_replay_verify_fold(ctypes.byref(e), *([None] * 14), None) == 0
    assert so.gdn_replay_accept_fold(ctypes.byref(e), None, None, None, None, None) == 0


def test_null_pointers_rejected():
    so = lib.load()
    d = good_dims()
    assert so.gdn_replay_verify(None, *([FAKE] * 14), None) == -1
    for i in (0, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13):   # index 1 (state_idx) may be NULL
        args = [FAKE] * 14
        args[i] = None
        assert so.gdn_replay_verify(ctypes.byref(d), *args, None) == -1, i
    assert so.gdn_replay_accept(ctypes.byref(d), None, None, FAKE, FAKE, None) == -1
    assert so.gdn_replay_accept(ctypes.byref(d), FAKE, None, None, FAKE, None) == -1
    assert so.gdn_replay_flush(ctypes.byref(d), None, *([FAKE] * 6), 0, FAKE, None) == -1


def test_misaligned_pointers_rejected():
    so = lib.load()
    d = good_dims()
    args = [FAKE] * 14
    args[0] = ctypes.c_void_p(0x10004)      # state must be 16-byte aligned
    assert so.gdn_replay_verify(ctypes.byref(d), *args, None) == -2


def test_empty_batch_is_a_noop():
    so = lib.load()
    d = good_dims(B=0, n_slot=0)
    assert so.gdn_replay_verify(ctypes.byref(d), *([None] * 14), None) == 0
    assert so.gdn_replay_accept(ctypes.byref(d), None, None, None, None, None) == 0
    assert so.gdn_replay_flush(ctypes.byref(d), *([None] * 7), 1, None, None) == 0


def test_strerror():
    for c in (0, -1, -2, -3, -4, -99):
        assert isinstance(lib.gdn_replay_strerror(c), str)


def test_binding_rejects_undersized_tensors_before_launch():
    """The Python binding checks every tensor against the dims (the C ABI takes bare
    pointers and cannot): one element short is refused before anything is launched."""
    import torch
    d = good_dims()
    sizes = lib._sizes(d)
    f32, bf16, i32 = torch.float32, torch.bfloat16, torch.int32
    kinds = {"state": f32, "state_idx": i32, "buf_k": bf16, "buf_v": bf16, "buf_g": f32,
             "buf_beta": f32, "buf_len": i32, "q": bf16, "k": bf16, "v": bf16, "g": f32,
             "beta": f32, "out": f32, "status": i32}
    order = ("state", "state_idx", "buf_k", "buf_v", "buf_g", "buf_beta", "buf_len", "q", "k", "v",
             "g", "beta", "out", "status")
    for short in order:
        args = [torch.zeros(sizes[n] - (1 if n == short else 0), dtype=kinds[n]) for n in order]
        with pytest.raises(ValueError, match=short):
            lib.gdn_replay_verify(d, *args)
    with pytest.raises(ValueError, match="accepted"):
        lib.gdn_replay_accept(d, torch.zeros(sizes["buf_len"], dtype=i32), None,
                              torch.zeros(sizes["accepted"] - 1, dtype=i32), torch.zeros(1, dtype=i32))


# ------------------------------------------ the layer steps either side of the recurrence
def conv_dims(**kw):
    d = dict(B=2, D=64, W=4, T=4, cap=8, n_slot=2, act=lib.CONV_ACT_SILU, in_dtype=lib.DTYPE_BF16,
             out_dtype=lib.DTYPE_BF16)
    d.update(kw)
    return lib.ConvDims(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(D=60), -2), (dict(D=0), -2), (dict(W=0), -2), (dict(W=5), -2), (dict(T=0), -2),
    (dict(T=65), -2), (dict(cap=6), -2), (dict(n_slot=1), -2), (dict(act=2), -2),
    (dict(in_dtype=3), -3), (dict(out_dtype=-1), -3), (dict(B=-1), -2),
])
def test_conv_bad_dims_rejected_before_launch(kw, code):
    so = lib.load()
    d = conv_dims(**kw)
    assert so.gdn_conv_verify(ctypes.byref(d), *([FAKE] * 8), None) == code
    assert so.gdn_conv_accept(ctypes.byref(d), FAKE, None, FAKE, FAKE, None) == code


def test_conv_null_and_empty():
    so = lib.load()
    d = conv_dims()
    for i in (0, 1, 3, 4, 6, 7):                 # state_idx (2) and bias (5) may be NULL
        args = [FAKE] * 8
        args[i] = None
        assert so.gdn_conv_verify(ctypes.byref(d), *args, None) == -1, i
    e = conv_dims(B=0, n_slot=0)
    assert so.gdn_conv_verify(ctypes.byref(e), *([None] * 8), None) == 0
    assert so.gdn_conv_accept(ctypes.byref(e), None, None, None, None, None) == 0


def test_norm_bad_arguments_rejected_before_launch():
    so = lib.load()
    args = [FAKE, FAKE, lib.DTYPE_BF16, FAKE, 1e-6, 1.0, FAKE, None]
    assert so.gdn_gated_rmsnorm_fp8(4, 96, *args) == -2             # d not 64, 128 or 256
    assert so.gdn_gated_rmsnorm_fp8(-1, 128, *args) == -2
    bad_z = list(args); bad_z[2] = 5
    assert so.gdn_gated_rmsnorm_fp8(4, 128, *bad_z) == -3
    bad_s = list(args); bad_s[5] = 0.0
    assert so.gdn_gated_rmsnorm_fp8(4, 128, *bad_s) == -2
    null_q = list(args); null_q[6] = None
    assert so.gdn_gated_rmsnorm_fp8(4, 128, *null_q) == -1
    assert so.gdn_gated_rmsnorm_fp8(0, 128, *([None] * 2), 0, None, 1e-6, 1.0, None, None) == 0


# ---------------------------------------------------------- non-replay baseline
def test_nonreplay_host_validation():
    so = lib.load()
    d = good_dims(T=16, cap=16, threshold=1)
    assert so.gdn_nonreplay_verify(None, *([FAKE] * 10), None) == -1
    for i in (0, 2, 3, 4, 5, 6, 7, 8, 9):                       # state_idx (1) may be NULL
        args = [FAKE] * 10
        args[i] = None
        assert so.gdn_nonreplay_verify(ctypes.byref(d), *args, None) == -1, i
    for i in (0, 2, 3, 4):
        args = [FAKE] * 5
        args[i] = None
        assert so.gdn_nonreplay_accept(ctypes.byref(d), *args, None) == -1, i
    for kw, code in ((dict(dk=96), -2), (dict(T=65, cap=65), -2), (dict(in_dtype=7), -3),
                     (dict(flags=1), -2), (dict(H=0), -2), (dict(n_slot=-1), -2)):
        bad = good_dims(**{**dict(T=16, cap=16, threshold=1), **kw})
        assert so.gdn_nonreplay_verify(ctypes.byref(bad), *([FAKE] * 10), None) == code, kw
        assert so.gdn_nonreplay_accept(ctypes.byref(bad), *([FAKE] * 5), None) == code, kw
    few = good_dims(T=16, cap=16, threshold=1, n_slot=1)       # fewer slots than rows, no slot map
    args = [FAKE] * 10
    args[1] = None
    assert so.gdn_nonreplay_verify(ctypes.byref(few), *args, None) == -2
    assert so.gdn_nonreplay_accept(ctypes.byref(few), FAKE, None, FAKE, FAKE, FAKE, None) == -2
    args = [FAKE] * 10
    args[8] = ctypes.c_void_p(0x10008)                          # snap must be 16-byte aligned
    assert so.gdn_nonreplay_verify(ctypes.byref(d), *args, None) == -2
    e = good_dims(B=0, n_slot=0, T=16, cap=16, threshold=1)
    assert so.gdn_nonreplay_verify(ctypes.byref(e), *([None] * 10), None) == 0
    assert so.gdn_nonreplay_accept(ctypes.byref(e), *([None] * 5), None) == 0


def test_nonreplay_binding_rejects_undersized_snapshots():
    import torch
    d = good_dims(T=4, cap=4, threshold=1)
    small = torch.empty(10, dtype=torch.float32)
    with pytest.raises(ValueError, match="snap"):
        lib.gdn_nonreplay_accept(d, torch.empty(2 * 2 * 128 * 128), None, small,
                                 torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32))
