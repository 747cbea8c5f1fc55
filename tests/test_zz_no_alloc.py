"""dflash2_topk_noalloc: top-k for callers that cannot allocate device memory.

Hosts such as an engine that plans all device memory itself (and gives plugins no
allocator) or a decode loop that cannot afford cudaMalloc's implicit synchronisation
cannot pass dflash2_topk a workspace.  The no-allocation variant keeps its scratch in
the library's own fixed device array.  Here it is called through the C ABI twice in a
row, on different logits, and must return exactly what dflash2_topk returns (top-k of
identical float32 logits is compared bit for bit throughout these tests).  This file
is collected last so that a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_drafter_gb300 import dflash2 as df

pytestmark = pytest.mark.gpu

DF2_ERR_UNSUPPORTED = 2


def _logits(rng, R, V):
    lg = rng.standard_normal((R, V)).astype(np.float32)
    lg[:, 11] = lg[:, 5]  # exact duplicates: lower id first
    lg[0, :12] = 3.5  # a run of equal maxima
    return torch.from_numpy(lg).cuda()


def test_topk_noalloc_matches_workspace_topk_on_two_calls():
    lib = df.library()
    rng = np.random.default_rng(2024)
    for R, V, k in ((16, 151936, 8), (64, 262144, 16)):
        logits = _logits(rng, R, V)
        want_ids, want_vals = df.dflash2_topk(logits, k)
        ids = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
        vals = torch.zeros((R, k), dtype=torch.float32, device="cuda")
        dims = df.make_dims(R, 1, 8, V, k, 8)
        st = lib.dflash2_topk_noalloc(ctypes.byref(dims), logits.data_ptr(), ids.data_ptr(), vals.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
        assert st == 0, df.dflash2_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(ids, want_ids)
        assert torch.equal(vals.view(torch.int32), want_vals.view(torch.int32))


def test_topk_noalloc_rejects_sizes_beyond_its_array():
    lib = df.library()
    dims = df.make_dims(1024, 1, 8, 262144, 16, 8)  # 1024 rows x KP 16 > 4096
    st = lib.dflash2_topk_noalloc(ctypes.byref(dims), 0x1000, 0x2000, 0x3000, None)
    assert st == DF2_ERR_UNSUPPORTED
