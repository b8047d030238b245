"""moe_align_block_size_noalloc: the align for callers that cannot allocate
device memory (an engine whose GPU memory is all in its own pool, or code that
must not risk the synchronisation cudaMalloc/cudaFree can bring), with its
scratch in a fixed 1 MiB buffer inside the library.

Checked through the C ABI against moe_align_block_size with a caller
workspace, bit for bit (the align tests' bar), on two calls in a row with
different routings, so the second call cannot lean on what the first left
in the shared buffer.  Sizes needing more scratch than the buffer are refused
before anything is launched.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import cuda, i32, lib, scratch, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.inputs import uniform_routes

pytestmark = pytest.mark.gpu


def _align(ids: np.ndarray, E: int, B: int, noalloc: bool, stream=None):
    R = ids.size
    cap = oes.align_capacity(R, E, B)
    s, b, n, st = i32(cap, -7), i32(cap // B, -7), i32(1, -7), status()
    d_ids = cuda(ids.astype(np.int32))
    if stream is not None:
        stream.wait_stream(torch.cuda.current_stream())   # the buffers above are ready
    if noalloc:
        oes.moe_align_block_size_noalloc(d_ids, R, E, B, 1, s, b, n, st, stream=stream)
    else:
        wsb = oes.moe_align_workspace_size(R, E, B)
        ws = scratch(wsb)
        if stream is not None:
            stream.wait_stream(torch.cuda.current_stream())
        oes.moe_align_block_size(d_ids, R, E, B, 1, s, b, n, st, ws, ws.numel(), stream=stream)
    torch.cuda.synchronize()
    return s.cpu().numpy(), b.cpu().numpy(), int(n.item()), int(st.item())


def _same(got, want):
    assert got[2] == want[2] and got[3] == want[3] == 0
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])


def test_noalloc_matches_workspace_align_on_two_calls_in_a_row():
    lib()
    cases = [(uniform_routes(4096, 10, 512, 77), 512, 128),      # long-prefill shape
             (uniform_routes(8192, 8, 2100, 78), 2100, 64)]      # past 1024 experts
    for ids, E, B in cases:
        assert oes.moe_align_workspace_size(ids.size, E, B) <= oes.OES_ALIGN_NOALLOC_SCRATCH_BYTES
        _same(_align(ids, E, B, noalloc=True), _align(ids, E, B, noalloc=False))


def test_noalloc_decode_width_and_side_stream():
    """Up to 1024 routes take the one-CTA align, which uses the buffer
    differently from the three-kernel path; and a call on a stream other
    than the current one orders its kernels on that stream alone."""
    lib()
    ids = uniform_routes(32, 10, 512, 79)                 # 320 routes: one-CTA path
    for _ in range(2):
        _same(_align(ids, 512, 16, noalloc=True), _align(ids, 512, 16, noalloc=False))
    side = torch.cuda.Stream()
    for ids, E, B in [(uniform_routes(32, 10, 512, 80), 512, 16),
                      (uniform_routes(4096, 10, 512, 81), 512, 128)]:
        _same(_align(ids, E, B, noalloc=True, stream=side), _align(ids, E, B, noalloc=False))


def test_noalloc_refuses_sizes_beyond_its_buffer():
    lib()
    R, E, B = 1 << 24, 4096, 16
    assert oes.moe_align_workspace_size(R, E, B) > oes.OES_ALIGN_NOALLOC_SCRATCH_BYTES
    with pytest.raises(oes.OesError) as e:
        oes.moe_align_block_size_noalloc(16, R, E, B, 1, 16, 16, 16, 0, stream=0)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
