"""The C ABI: every symbol include/lbq.h declares is exported by liblbq.so, and
host-side validation rejects bad arguments before anything touches a GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "lbq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lbq_\w+)\s*\(", src)))


def test_header_declarations_are_exported(lbq):
    from bit_weight_only_lbq_gb300 import build as B
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    declared = _declared()
    assert len(declared) >= 17
    missing = [d for d in declared if d not in exported]
    assert not missing, missing
    assert sorted(lbq.EXPORTS) == declared


def test_status_strings(lbq):
    L = lbq.lib()
    for code, name in lbq.STATUS.items():
        assert L.lbq_status_string(code).decode().startswith(name)
    assert L.lbq_format_version() == 2


def test_host_argument_errors(lbq):
    L = lbq.lib()
    W = np.zeros((4, 64), np.float32)
    buf = np.zeros(1 << 16, np.uint8)
    p = W.ctypes.data
    assert L.lbq_pack_w4(None, 4, 64, None, 0, buf.ctypes.data, buf.size) == 1          # NULL
    assert L.lbq_pack_w4(p, 4, 96, None, 0, buf.ctypes.data, buf.size) == 2             # K % 64
    assert L.lbq_pack_w4(p, 0, 64, None, 0, buf.ctypes.data, buf.size) == 2             # N
    assert L.lbq_pack_w4(p, 4, 64, None, 0, buf.ctypes.data, 10) == 5                   # too small
    bad = np.array([3, 3], np.int32)
    assert L.lbq_pack_w4(p, 4, 64, bad.ctypes.data, 2, buf.ctypes.data, buf.size) == 4  # not ascending
    oob = np.array([64], np.int32)
    assert L.lbq_pack_w2cb(p, 4, 64, oob.ctypes.data, 1, buf.ctypes.data, buf.size) == 4
    Wn = W.copy()
    Wn[1, 2] = np.nan
    assert L.lbq_pack_w4(Wn.ctypes.data, 4, 64, None, 0, buf.ctypes.data, buf.size) == 9
    assert L.lbq_w4_packed_bytes(4, 96, 0) == 0
    idx = np.zeros(1, np.int32)
    n = ctypes.c_int32(0)
    Wh = np.random.default_rng(0).standard_normal((8, 1536)).astype(np.float32)
    st = L.lbq_select_outliers_w4(Wh.ctypes.data, 8, 1536, idx.ctypes.data, 1, ctypes.byref(n))
    assert st == 5 and n.value > 1


def test_device_entry_points_reject_bad_args_without_gpu(lbq):
    """Host validation runs before any CUDA call, so these return on a CPU machine too."""
    L = lbq.lib()
    assert L.lbq_gemv_w4a16(None, 8, 64, 0, 16, 16, 0, None) == 1
    assert L.lbq_gemv_w4a16(16, 8, 96, 0, 16, 16, 0, None) == 2
    assert L.lbq_gemv_w2cb_outlier(16, 8, 64, 65, 16, 16, 0, None) == 2
    assert L.lbq_gemv_w4a16(8, 8, 64, 0, 16, 16, 0, None) == 3          # packed not 16-aligned
    assert L.lbq_gemv_w4a16(16, 8, 64, 0, 16, 16, 7, None) == 10        # bad dtype
    assert L.lbq_gemm_w4a16_smallM(16, 0, 8, 64, 0, 16, 64, 16, 8, 0, None) == 2
    assert L.lbq_gemm_w4a16_smallM(16, 65, 8, 64, 0, 16, 64, 16, 8, 0, None) == 2
    assert L.lbq_gemm_w4a16_smallM(16, 2, 8, 64, 0, 16, 60, 16, 8, 0, None) == 2   # ldx < K
    assert L.lbq_gemm_w4a16_smallM(16, 2, 8, 64, 0, 16, 68, 16, 8, 0, None) == 3   # ldx % 8
    assert L.lbq_gemm_w2cb_outlier_smallM(16, 65, 8, 64, 0, 16, 64, 16, 8, 0, None) == 2
    assert L.lbq_gemm_w2cb_outlier_smallM(16, 2, 8, 64, 0, 16, 60, 16, 8, 0, None) == 2   # ldx < K
    assert L.lbq_gemm_w2cb_outlier_smallM(None, 2, 8, 64, 0, 16, 64, 16, 8, 0, None) == 1


def test_grouped_entry_point_rejects_bad_args_without_gpu(lbq):
    L = lbq.lib()
    P = lbq.Problem
    good = P(16, 8, 64, 0, 0, 16, 64, 16, 8)
    arr = (P * (lbq.LBQ_MAX_GROUP + 1))(*([good] * (lbq.LBQ_MAX_GROUP + 1)))
    assert L.lbq_gemv_grouped(0, None, 1, 1, 0, None, 0) == 1
    assert L.lbq_gemv_grouped(0, arr, 0, 1, 0, None, 0) == 2
    assert L.lbq_gemv_grouped(0, arr, lbq.LBQ_MAX_GROUP + 1, 1, 0, None, 0) == 2
    assert L.lbq_gemv_grouped(5, arr, 1, 1, 0, None, 0) == 10          # unknown kind
    # 2-bit small M passes validation like M = 1 (here it then stops at the
    # device query: no GPU)
    assert L.lbq_gemv_grouped(1, arr, 1, 2, 0, None, 0) == L.lbq_gemv_grouped(1, arr, 1, 1, 0, None, 0) != 0
    assert L.lbq_gemv_grouped(1, arr, 1, 65, 0, None, 0) == 2
    assert L.lbq_gemv_grouped(0, arr, 1, 65, 0, None, 0) == 2
    bad = (P * 2)(good, P(16, 8, 64, 0, 1, 16, 64, 16, 8))             # reserved != 0
    assert L.lbq_gemv_grouped(0, bad, 2, 1, 0, None, 0) == 2
    bad = (P * 2)(good, P(16, 8, 96, 0, 0, 16, 96, 16, 8))             # K % 64
    assert L.lbq_gemv_grouped(0, bad, 2, 1, 0, None, 0) == 2
    bad = (P * 2)(good, P(16, 8, 64, 0, 0, None, 64, 16, 8))           # null x in the second problem
    assert L.lbq_gemv_grouped(0, bad, 2, 1, 0, None, 0) == 1
    bad = (P * 2)(good, P(16, 8, 64, 0, 0, 16, 64, 16, 4))             # ldy < N
    assert L.lbq_gemv_grouped(0, bad, 2, 1, 0, None, 0) == 2


def test_grouped_selection_and_refined_sweep_argument_errors(lbq):
    """lbq_refine_select_grouped and lbq_gemv_grouped_refined validate every
    descriptor on the host before touching a device (fake device addresses)."""
    L = lbq.lib()
    SP, RF, PB = lbq.SelectProblem, lbq.Refinement, lbq.Problem
    x, idx, rb = 0x10000, 0x20000, 0x30000
    ok = SP(x, 4096, 16, 0, idx, rb, 4096)
    assert L.lbq_refine_select_grouped(None, 1, None) == 1                         # NULL array
    assert L.lbq_refine_select_grouped((SP * 1)(ok), 0, None) == 2                 # count
    assert L.lbq_refine_select_grouped((SP * 1)(SP(0, 4096, 16, 0, idx, rb, 4096)), 1, None) == 1
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x, 4096, 0, 0, idx, rb, 4096)), 1, None) == 2    # k
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x, 4096, 257, 0, idx, rb, 4096)), 1, None) == 2  # k > 256
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x, 4096, 16, 1, idx, rb, 4096)), 1, None) == 2   # reserved
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x, 4096, 16, 0, idx, rb, 100)), 1, None) == 2    # N % 64
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x + 1, 4096, 16, 0, idx, rb, 4096)), 1, None) == 3  # x align
    assert L.lbq_refine_select_grouped((SP * 1)(SP(x, 4096, 16, 0, idx, rb + 8, 4096)), 1, None) == 3  # blob align
    prob = (PB * 1)(PB(0x40000, 128, 1024, 0, 0, x, 1024, 0x50000, 128))
    assert L.lbq_gemv_grouped_refined(0, prob, None, 1, 1, None, 0) == 1            # no refinement array
    assert L.lbq_gemv_grouped_refined(0, prob, (RF * 1)(RF(rb, idx, 1025, 0)), 1, 1, None, 0) == 2  # n_sel > K
    assert L.lbq_gemv_grouped_refined(0, prob, (RF * 1)(RF(rb, idx, 4, 1)), 1, 1, None, 0) == 2     # reserved
    assert L.lbq_gemv_grouped_refined(0, prob, (RF * 1)(RF(rb, None, 4, 0)), 1, 1, None, 0) == 1    # idx
    assert L.lbq_gemv_grouped_refined(0, prob, (RF * 1)(RF(rb + 8, idx, 4, 0)), 1, 1, None, 0) == 3  # blob align
    odd = (PB * 1)(PB(0x40000, 100, 1024, 0, 0, x, 1024, 0x50000, 100))
    assert L.lbq_gemv_grouped_refined(0, odd, (RF * 1)(RF(rb, idx, 4, 0)), 1, 1, None, 0) == 2     # N % 64
