"""C-ABI tests that need no GPU: the library loads, exports every entry point
declared in include/nvfp4.h, its layout helpers agree with the oracle, and
argument validation returns the documented status before touching a device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from nvfp4_precision_02_b300 import build, binding
    build.build()
    return binding.lib()


@pytest.fixture(scope="module")
def B():
    from nvfp4_precision_02_b300 import binding
    return binding


def _declared():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(L, B):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), n
    assert sorted(B.EXPORTS) == names


def test_layout_helpers_match_oracle(L, orc):
    for rows, cols in [(1, 16), (127, 48), (128, 64), (129, 1040), (8192, 6144), (33024, 8192)]:
        assert L.nvfp4_sf_bytes(rows, cols) == orc.sf_bytes(rows, cols)
        for r, c in [(0, 0), (rows - 1, cols // 16 - 1), (rows // 2, (cols // 16) // 2)]:
            assert L.nvfp4_sf_offset(r, c, cols) == orc.sf_offset(r, c, cols)
    assert L.nvfp4_sf_bytes_grouped(300, 32, 5) == orc.sf_bytes_grouped(300, 32, 5)
    assert L.nvfp4_sf_bytes(0, 16) == 0


FAKE = 0x10000   # aligned, never dereferenced: validation fails or no device


def _t(rows, cols, codes=FAKE, sf=FAKE, amax=FAKE):
    from nvfp4_precision_02_b300.binding import CTensor
    return CTensor(codes, sf, amax, rows, cols)


def test_quantize_1d_validation(L):
    ok = _t(64, 32)
    f = L.nvfp4_quantize_1d
    assert f(None, 64, 32, 32, 0, 0, None, ctypes.byref(ok), None) == 1                 # NULL x
    assert f(FAKE, 64, 24, 24, 0, 0, None, ctypes.byref(_t(64, 24)), None) == 2          # cols % 16
    assert f(FAKE, 64, 32, 16, 0, 0, None, ctypes.byref(ok), None) == 2                  # ld < cols
    assert f(FAKE + 8, 64, 32, 32, 0, 0, None, ctypes.byref(ok), None) == 3              # misaligned
    assert f(FAKE, 64, 32, 36, 0, 0, None, ctypes.byref(ok), None) == 3                  # ld % 8
    assert f(FAKE, 64, 32, 32, 0, 0, None, ctypes.byref(_t(63, 32)), None) == 2          # shape mismatch
    assert f(FAKE, 64, 32, 32, 0, 0, None, None, None) == 1                              # NULL out
    assert f(FAKE, 64, 32, 32, 0, 0, None, ctypes.byref(_t(64, 32, amax=0)), None) == 1  # NULL amax
    assert f(FAKE, 64, 32, 32, 5, 0, None, ctypes.byref(ok), None) == 2                  # bad mode


def test_other_entry_points_validation(L):
    assert L.nvfp4_quantize_2d(FAKE, 1, 40, 32, 32, None, ctypes.byref(_t(40, 32)), None, None, None) == 2
    assert L.nvfp4_quantize_2d(FAKE, 0, 32, 32, 32, None, ctypes.byref(_t(32, 32)), None, None, None) == 2
    assert L.nvfp4_quantize_2d(FAKE, 1, 32, 64, 64, None, ctypes.byref(_t(32, 64)),
                               ctypes.byref(_t(32, 64)), None, None) == 2                # W^T shape
    assert L.nvfp4_rht_quantize(FAKE, 40, 32, 32, 1, 0, 0, None, ctypes.byref(_t(32, 40)), None) == 2
    assert L.nvfp4_rht_amax(FAKE, 32, 8, 8, 1, None, None) == 1
    a, b = _t(64, 64), _t(48, 64)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(_t(48, 80)), FAKE, 48, 0, None, None) == 2      # K mismatch
    assert L.nvfp4_gemm(ctypes.byref(_t(64, 40)), ctypes.byref(_t(48, 40)), FAKE, 48, 0, None, None) == 2  # K % 16
    # K % 16 == 0 passes the shape checks (then no sm_103 device here: NVFP4_ERR_DEVICE)
    assert L.nvfp4_gemm(ctypes.byref(_t(64, 48)), ctypes.byref(_t(48, 48)), FAKE, 48, 0, None, None) == 4
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), FAKE, 40, 0, None, None) == 2              # ldc < N
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), FAKE + 1, 48, 0, None, None) == 3          # c misaligned
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), None, 48, 0, None, None) == 1
    assert L.nvfp4_grouped_gemm(ctypes.byref(a), None, 4, ctypes.byref(b), 48, FAKE, 48, 0, None, None) == 1
    assert L.nvfp4_grouped_gemm(ctypes.byref(a), FAKE, 2000, ctypes.byref(b), 48, FAKE, 48, 0, None, None) == 7
    assert L.nvfp4_quantize_1d_grouped(FAKE, 64, 32, 32, FAKE, 0, 0, 0, None, ctypes.byref(_t(64, 32)), None) == 7
    assert L.nvfp4_quantize_2d_fused(FAKE, 2, 32, 32, 32, None, 64, ctypes.byref(_t(32, 32)), None, None) == 1
    assert L.nvfp4_quantize_2d_fused(FAKE, 2, 32, 32, 32, FAKE, 4, ctypes.byref(_t(32, 32)), None, None) == 2
    assert L.nvfp4_quantize_2d_fused_workspace(512) == 2064
    assert L.nvfp4_quantize_2d_fused_workspace(5) == 32


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_calls_report_missing_device(L):
    ok = _t(64, 32)
    assert L.nvfp4_quantize_1d(FAKE, 64, 32, 32, 0, 0, None, ctypes.byref(ok), None) == 4
    assert b"device" in L.nvfp4_last_error().lower()
    a, b = _t(64, 64), _t(48, 64)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), FAKE, 48, 0, None, None) == 4


def test_empty_gemm_is_a_no_op(L):
    # M == 0: valid, nothing to launch (returns before any device work)
    a, b = _t(0, 64), _t(48, 64)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), None, 48, 0, None, None) == 0


def test_inject_hook_is_host_side(L, B):
    B.debug_inject(5)
    assert L.nvfp4_quantize_1d(FAKE, 64, 32, 32, 0, 0, None, ctypes.byref(_t(64, 32)), None) == 5
    assert b"injected" in L.nvfp4_last_error()
    # the hook fires once
    assert L.nvfp4_quantize_1d(None, 64, 32, 32, 0, 0, None, ctypes.byref(_t(64, 32)), None) == 1
    with pytest.raises(B.Nvfp4Error) as e:
        B.debug_inject(6)
        B._check(L.nvfp4_gemm(None, None, None, 0, 0, None, None))
    assert e.value.status == 6


def test_status_strings(L):
    for s in range(8):
        assert L.nvfp4_status_string(s)
    assert L.nvfp4_status_string(0) == b"ok"


def test_backward_and_next_row_entry_points_validation(L):
    """Argument checks of the grouped backward, PTQ, FP16 SR and monitoring
    entry points come before any device access."""
    # capacity of the expert-segmented operand: every split fits
    assert L.nvfp4_group_k_capacity(1000, 7) == ((1000 + 63 * 7 + 63) // 64) * 64
    assert L.nvfp4_group_k_capacity(0, 1) == 64 and L.nvfp4_group_k_capacity(5, 0) == 0
    cap = L.nvfp4_group_k_capacity(100, 4)
    g = L.nvfp4_rht_quantize_grouped
    assert g(FAKE, 100, 48, 48, None, 4, cap, 0, 0, 0, None, ctypes.byref(_t(48, cap)), None) == 1     # NULL offsets
    assert g(FAKE, 100, 48, 48, FAKE, 0, cap, 0, 0, 0, None, ctypes.byref(_t(48, cap)), None) == 7     # no groups
    assert g(FAKE, 100, 48, 48, FAKE, 4, cap - 64, 0, 0, 0, None, ctypes.byref(_t(48, cap - 64)), None) == 2
    assert g(FAKE, 100, 48, 48, FAKE, 4, cap + 32, 0, 0, 0, None, ctypes.byref(_t(48, cap + 32)), None) == 2
    assert g(FAKE, 100, 48, 48, FAKE, 4, cap, 0, 7, 0, None, ctypes.byref(_t(48, cap)), None) == 2     # bad mode
    k = L.nvfp4_grouped_gemm_k
    assert k(ctypes.byref(_t(64, 96)), ctypes.byref(_t(64, 96)), FAKE, 2, FAKE, 64, 0, None, None) == 2  # K % 64
    assert k(ctypes.byref(_t(64, 128)), ctypes.byref(_t(64, 192)), FAKE, 2, FAKE, 64, 0, None, None) == 2
    assert k(ctypes.byref(_t(64, 128)), ctypes.byref(_t(64, 128)), None, 2, FAKE, 64, 0, None, None) == 1
    assert k(ctypes.byref(_t(64, 128)), ctypes.byref(_t(64, 128)), FAKE, 0, FAKE, 64, 0, None, None) == 7
    assert k(ctypes.byref(_t(64, 128)), ctypes.byref(_t(64, 128)), FAKE, 2, FAKE, 32, 0, None, None) == 2  # ldc < N
    s = L.nvfp4_sr_fp16
    assert s(FAKE, -1, 0, FAKE, None) == 2 and s(None, 8, 0, FAKE, None) == 1 and s(FAKE, 8, 0, FAKE + 1, None) == 3
    assert s(None, 0, 0, None, None) == 0                                                         # nothing to do
    m = L.nvfp4_quantize_1d_mse
    assert m(FAKE, 64, 24, 24, None, ctypes.byref(_t(64, 24)), None) == 2                          # cols % 16
    assert m(FAKE + 8, 64, 32, 32, None, ctypes.byref(_t(64, 32)), None) == 3                      # misaligned rows
    d = L.nvfp4_dual_amax
    assert d(FAKE, 64, 32, 32, 0, None, FAKE, None) == 1 and d(FAKE, 60, 32, 32, 0, FAKE, FAKE, None) == 2
    z = L.nvfp4_count_zero_codes
    assert z(None, FAKE, None) == 1 and z(ctypes.byref(_t(4, 32)), None, None) == 1
    assert z(ctypes.byref(_t(4, 32)), FAKE + 4, None) == 3                                        # count alignment
