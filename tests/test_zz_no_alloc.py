"""tv_accept_noalloc: acceptance for callers that cannot allocate device memory.

It must give exactly what tv_accept gives (argmax, accepted length, path and
bonus token are integers: bit-exact), on two calls in a row with different
inputs, so that scratch left by the first call cannot leak into the second.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload


def _workload(seed, nb, B, V):
    rng = np.random.default_rng(seed)
    trees = [wl.tree_best_first(rng, B, child_cap=3, max_depth=B) for _ in range(nb)]
    return wl.make_workload("noalloc", nb, B, 8, 2, 128, V, [5] * nb, trees, seed, extra_pages=1)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    for seed, (nb, B, V) in ((1, (3, 64, 50021)), (2, (2, 200, 4096))):
        d = DevWorkload(_workload(seed, nb, B, V))
        mask, _ = d.mask()
        ref = tv.accept(d.logits, d.draft, d.parent, mask, status=d.status)
        got = tv.accept_noalloc(d.logits, d.draft, d.parent, mask, status=d.status)
        torch.cuda.synchronize()
        assert d.status.item() == 0
        for r, g in zip(ref, got):
            assert torch.equal(r, g)


@pytest.mark.gpu
def test_noalloc_rejects_too_many_rows():
    # real device buffers sized for the oversized call, so that a regression of the row
    # limit would give a wrong return code, not kernels writing through made-up addresses
    B, V = 256, 100
    big = tv.binding.NOALLOC_MAX_ROWS // B + 1
    dev = "cuda"
    logits = torch.zeros((big * B, V), dtype=torch.int16, device=dev)
    draft = torch.zeros((big, B), dtype=torch.int32, device=dev)
    parent = torch.arange(-1, B - 1, dtype=torch.int32, device=dev).repeat(big, 1)
    am = torch.zeros(big * B, dtype=torch.int32, device=dev)
    n_acc = torch.zeros(big, dtype=torch.int32, device=dev)
    path = torch.zeros((big, B), dtype=torch.int32, device=dev)
    bonus = torch.zeros(big, dtype=torch.int32, device=dev)
    P = C.c_void_p
    rc = tv.lib().tv_accept_noalloc(P(logits.data_ptr()), V, P(draft.data_ptr()), P(parent.data_ptr()), None, B,
                                    big, P(am.data_ptr()), P(n_acc.data_ptr()), P(path.data_ptr()),
                                    P(bonus.data_ptr()), None, None)
    torch.cuda.synchronize()
    assert rc == 3  # TV_ERR_UNSUPPORTED_SHAPE
    assert int(n_acc.abs().sum()) == 0  # nothing was enqueued
