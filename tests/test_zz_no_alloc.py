"""fathom_topk_noalloc: the top-k for callers that cannot provide or allocate
device scratch (its scratch is a fixed array inside the library).  Called
through the C ABI twice in a row on different inputs; each result must equal
fathom_topk's (bit-exact indices and values, the tolerance of the top-k tests).
Sizes beyond the fixed scratch are refused before anything is launched.

This file is collected last so that a failure here cannot hide another test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _call_noalloc(L, scores, k):
    rows, n = scores.shape
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((rows, k), float("nan"), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.fathom_topk_noalloc(rows, n, k, ctypes.c_void_p(scores.data_ptr()), ctypes.c_void_p(idx.data_ptr()),
                               ctypes.c_void_p(vals.data_ptr()), stream)
    return rc, idx, vals


def test_topk_noalloc_matches_topk_on_two_calls(gpu_lib):
    F = gpu_lib
    L = F.load()
    rng = np.random.default_rng(2026)
    cases = [
        (8, 300_000, 2048, rng.standard_normal((8, 300_000)).astype(np.float32)),
        (3, 70_001, 512, rng.choice(np.linspace(-1, 1, 16).astype(np.float32), (3, 70_001))),  # heavy ties
    ]
    for rows, n, k, s in cases:  # two calls in a row, different shapes and contents
        sd = torch.from_numpy(s).cuda()
        rc, idx, vals = _call_noalloc(L, sd, k)
        assert rc == 0, L.fathom_last_error()
        ref_idx, ref_vals = F.topk(sd, k, with_values=True)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.equal(vals.view(torch.int32), ref_vals.view(torch.int32))


def test_topk_noalloc_rejects_sizes_beyond_its_scratch(gpu_lib):
    L = gpu_lib.load()
    big = ctypes.c_size_t()
    assert L.fathom_topk_workspace_bytes(288, 1 << 20, 2048, ctypes.byref(big)) == 0
    assert big.value > (8 << 20)
    scores = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    rc = L.fathom_topk_noalloc(288, 1 << 20, 2048, ctypes.c_void_p(scores.data_ptr()),
                               ctypes.c_void_p(scores.data_ptr()), None, None)
    assert rc == 1
    assert b"scratch" in L.fathom_last_error()
