"""The register budget the overlapped step relies on, checked at compile time.

Three verify CTAs must fit beside one fold CTA on an SM (65 536 registers), and the
verify must keep five CTAs per SM when it runs alone.  ptxas reports the registers
of every kernel; this compiles the tensor-core translation unit for sm_103a (no GPU
needed) and checks them.
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "speculative_decode_recurrent_gb300", "csrc", "gdn_replay_tc.cu")
REGS_PER_SM = 65536
THREADS = 128


def _alloc(regs):
    return (regs + 7) // 8 * 8                      # registers are granted per warp in units of 8


@pytest.fixture(scope="module")
def registers():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        p = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                            "-Xptxas", "-v", "-I", os.path.join(ROOT, "include"), "-c", SRC,
                            "-o", os.path.join(tmp, "tc.o")], capture_output=True, text=True)
    assert p.returncode == 0, p.stderr[-2000:]
    regs, spills, current = {}, {}, None
    for line in p.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and current:
            spills[current] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            regs[current] = int(m.group(1))
            current = None
    regs["__spills__"] = spills
    return regs


def _find(regs, pattern):
    hits = [v for k, v in regs.items() if k != "__spills__" and re.search(pattern, k)]
    assert len(hits) == 1, (pattern, sorted(regs))
    return hits[0]


def test_verify_keeps_five_ctas_per_sm(registers):
    r = _find(registers, r"verify_eq_kernelILi48E")
    assert 5 * THREADS * _alloc(r) <= REGS_PER_SM, r


@pytest.mark.parametrize("draft", [0, 1])
def test_three_verify_ctas_beside_a_fold_cta(registers, draft):
    v = _find(registers, r"verify_eq_kernelILi48E")
    f = _find(registers, rf"fold_eq_kernelILi48ELb{draft}E")
    assert 3 * THREADS * _alloc(v) + THREADS * _alloc(f) <= REGS_PER_SM, (v, f)


def test_tensor_core_kernels_do_not_spill(registers):
    spills = registers["__spills__"]
    tc = {k: v for k, v in spills.items() if "verify_eq_kernel" in k or "fold_eq_kernel" in k}
    assert len(tc) == 9, sorted(spills)              # verify <48|64|80>; fold <48|64|80, draft 0|1>
    assert all(v == 0 for v in tc.values()), tc
