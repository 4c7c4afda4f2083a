"""The allocation-free entry point (nvfp4_quantize_2d_fused_static): the same
fused amax + 2D quantisation of batched weights, with its counters in the
library's fixed scratch array instead of a caller workspace.  It exists for
callers that cannot allocate device memory when they quantise (their memory
is owned by another allocator with no workspace to lend, or the loop must not
call cudaMalloc).  This file is collected last so that a run stopping at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from parity import np_u8


@pytest.fixture(scope="module")
def B():
    from nvfp4_precision_02_b300 import binding, build
    build.build()
    binding.lib()
    return binding


def _weights(batch, rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(batch, rows, cols, generator=g) * 0.02 *
            torch.exp(torch.rand(batch, 1, 1, generator=g) * 6 - 3)).to(torch.bfloat16)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_point(B):
    """Two calls in a row through the C ABI, on different weights, each
    bit-identical (amax, codes, scales, tile scales) to the workspace entry
    point; the second call shows the scratch left by the first is cleared."""
    assert torch.cuda.is_available()
    for seed, (batch, rows, cols) in [(1, (6, 144, 320)), (2, (3, 64, 1040))]:
        w = _weights(batch, rows, cols, seed).cuda()
        qs, ts = B.quantize_2d_fused_static(w, want_tile_sf=True)
        qw, tw = B.quantize_2d_fused(w, want_tile_sf=True)
        torch.cuda.synchronize()
        assert (np_u8(qs.amax) == np_u8(qw.amax)).all()
        assert (np_u8(qs.codes) == np_u8(qw.codes)).all()
        assert (np_u8(qs.sf) == np_u8(qw.sf)).all()
        assert (np_u8(ts) == np_u8(tw)).all()
    assert B.device_status() == 0


def test_static_scratch_rejects_oversized_batch(B):
    """A batch beyond the fixed scratch is refused on the host, before any
    device work, with a message that names the limit."""
    from nvfp4_precision_02_b300.binding import CTensor
    t = CTensor(0x10000, 0x10000, 0x10000, 32, 32)
    st = B.lib().nvfp4_quantize_2d_fused_static(0x10000, B.STATIC_MAX_BATCH + 1, 32, 32, 32, ctypes.byref(t),
                                                None, None)
    assert st == 7
    assert b"static scratch" in B.lib().nvfp4_last_error()
