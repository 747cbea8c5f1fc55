"""dflash2_topk_noalloc: top-k for callers that cannot allocate device memory.

Hosts such as an engine that plans all device memory itself (and gives plugins no
allocator) or a decode loop that cannot afford cudaMalloc's implicit synchronisation
cannot pass dflash2_topk a workspace.  The no-allocation variant keeps its scratch in
the library's own fixed device array.  Here it is called through the C ABI twice in a
row, on different logits, and must return exactly what dflash2_topk returns and exactly
what the oracle's full sort returns (top-k of identical float32 logits is compared bit
for bit throughout these tests).  The largest request the array admits (B*T*KP = 4096,
which fills the whole array and puts the id lists at its end) is among the cases.  This
file is collected last so that a stop-at-first-failure run has already run everything
else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_drafter_gb300 import dflash2 as df

pytestmark = pytest.mark.gpu

DF2_ERR_UNSUPPORTED = 2


def _logits(rng, R, V):
    lg = rng.standard_normal((R, V)).astype(np.float32)
    lg[:, 11] = lg[:, 5]  # exact duplicates: lower id first
    lg[0, :12] = 3.5  # a run of equal maxima
    return lg


def _call_noalloc(lib, logits, R, V, k):
    ids = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
    vals = torch.zeros((R, k), dtype=torch.float32, device="cuda")
    dims = df.make_dims(R, 1, 8, V, k, 8)
    st = lib.dflash2_topk_noalloc(ctypes.byref(dims), logits.data_ptr(), ids.data_ptr(), vals.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == 0, df.dflash2_status_string(st)
    torch.cuda.synchronize()
    return ids, vals


# (R, V, k): two ordinary requests, then the largest the array admits with KP = 32 and
# with KP = 16 (R * KP = 4096)
CASES = ((16, 151936, 8), (64, 262144, 16), (128, 151936, 32), (256, 151936, 16))


@pytest.mark.parametrize("R,V,k", CASES)
def test_topk_noalloc_matches_workspace_topk_and_oracle_on_two_calls(R, V, k):
    lib = df.library()
    rng = np.random.default_rng(2024 + R + k)
    for call in range(2):
        lg = _logits(rng, R, V)
        logits = torch.from_numpy(lg).cuda()
        want_ids, want_vals = df.dflash2_topk(logits, k)
        ids, vals = _call_noalloc(lib, logits, R, V, k)
        assert torch.equal(ids, want_ids), f"call {call}"
        assert torch.equal(vals.view(torch.int32), want_vals.view(torch.int32)), f"call {call}"
        o_ids, o_vals = oracle.topk(lg, k)
        assert np.array_equal(ids.cpu().numpy(), o_ids), f"call {call}"
        assert np.array_equal(vals.cpu().numpy().view(np.uint32), o_vals.view(np.uint32)), f"call {call}"


def test_topk_noalloc_rejects_sizes_beyond_its_array():
    """A request over the array's limit is refused before any launch; the buffers are real
    (small) device tensors, so nothing could go astray even if the check were missing."""
    lib = df.library()
    R, V, k = 512, 64, 16  # R * KP = 8192 > 4096
    logits = torch.zeros((R, V), dtype=torch.float32, device="cuda")
    ids = torch.full((R, k), -1, dtype=torch.int32, device="cuda")
    vals = torch.zeros((R, k), dtype=torch.float32, device="cuda")
    dims = df.make_dims(R, 1, 8, V, k, 8)
    st = lib.dflash2_topk_noalloc(ctypes.byref(dims), logits.data_ptr(), ids.data_ptr(), vals.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert st == DF2_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(ids == -1), "a refused call wrote its outputs"

