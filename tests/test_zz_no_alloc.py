"""moe_permute_noalloc: the permutation for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (or size and pass a workspace): code in a
host callback or under an embedding runtime's allocator lock, or a process
whose device memory is owned entirely by another framework.  This entry point
takes only the inputs and outputs and keeps its scratch in a fixed array
inside the library.  The test checks it through the C ABI against the
workspace-taking moe_permute, bit for bit, on two calls in a row (the second
must not see the first call's leftovers), and that sizes above its limit are
refused on the host.  The file name sorts last so that a run stopping at the
first failure has already run every other test.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import quantized_routed_expert_sigmoid_gb300 as moe
from quantized_routed_expert_sigmoid_gb300 import _native as N

pytestmark = pytest.mark.gpu


def _ids(T, k, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1)
    p[E // 3] = 0.0                                   # one expert never chosen
    p /= p.sum()
    return np.stack([np.sort(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]).astype(np.int32)


def _with_workspace(ids, E):
    T, k = ids.shape
    P = T * k
    d = torch.from_numpy(ids).cuda()
    sp = torch.empty(P, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pp = torch.empty(P, dtype=torch.int32, device="cuda")
    nb = moe.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    moe.moe_permute(d, T, k, E, sp, off, pp, ws, nb)
    torch.cuda.synchronize()
    return sp.cpu(), off.cpu(), pp.cpu()


def _no_alloc(ids, E):
    T, k = ids.shape
    P = T * k
    d = torch.from_numpy(ids).cuda()
    sp = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pp = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    moe.moe_permute_noalloc(d, T, k, E, sp, off, pp)
    torch.cuda.synchronize()
    return sp.cpu(), off.cpu(), pp.cpu()


def test_noalloc_matches_workspace_permute_twice():
    # first call: many chunks (exercises the arrival ticket and per-chunk bases);
    # second call: a different size on the same scratch, which must start clean
    # the largest accepted size (65,536 pairs in 64 chunks over 1024 experts) fills every
    # chunk-base word of the fixed array
    for (T, k, E, seed) in ((3000, 8, 128, 1), (700, 8, 256, 2), (1, 8, 128, 3), (8192, 8, 1024, 4)):
        ids = _ids(T, k, E, seed)
        ref = _with_workspace(ids, E)
        got = _no_alloc(ids, E)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        assert int(got[1][E]) == T * k


def test_noalloc_rejects_sizes_above_its_limit():
    with pytest.raises(N.MoeError) as ei:
        moe.moe_permute_noalloc(16, 8193, 8, 128, 16, 16, 16)      # 65,544 pairs > 65,536
    assert ei.value.status == N.MOE_ERR_INVALID_ARG
    assert "65536" in str(ei.value)
