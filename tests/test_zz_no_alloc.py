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
    nb, B = 2, 256
    assert nb * B <= tv.binding.NOALLOC_MAX_ROWS
    big = tv.binding.NOALLOC_MAX_ROWS // B + 1
    P = C.c_void_p
    fake = [P(0x10000)] * 9
    rc = tv.lib().tv_accept_noalloc(fake[0], 100, fake[1], fake[2], fake[3], B, big, fake[4], fake[5], fake[6],
                                    fake[7], None, None)
    assert rc == 3  # TV_ERR_UNSUPPORTED_SHAPE
