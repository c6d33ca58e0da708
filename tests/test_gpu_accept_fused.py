"""GPU parity of tv_accept_fused (argmax and greedy acceptance in one kernel) with the oracle.

Bit-exact like tv_accept: argmax of every row, accepted length, path and bonus.  Cases
cover sequences whose rows share a CTA (B smaller than a row group), rows split into
several chunks, an unaligned vocabulary, the mask given or built in-kernel from the
parent array, the workspace counters returning to zero across calls, a non-topological
parent array, and replay inside a CUDA graph.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload
from tests.test_gpu_parity import _workload

pytestmark = pytest.mark.gpu


def _check(w, am, n_acc, path, bonus):
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am)
    assert np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(path.cpu().numpy(), r_path)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)


@pytest.mark.parametrize("with_mask", [True, False])
@pytest.mark.parametrize("nb,B,V", [(9, 1, 7), (6, 3, 300), (5, 7, 3), (4, 16, 4096), (3, 33, 1001), (2, 64, 5),
                                    (2, 256, 4099), (1, 256, 151936), (2, 3, 300001)])
def test_accept_fused_bit_exact(nb, B, V, with_mask):
    rng = np.random.default_rng(nb * 7919 + B * 1000 + V)
    w = _workload(B + V + nb, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    if V <= 7:  # tiny vocab: many ties and many accepted edges
        w.logits[:] = wl.f32_to_bf16(rng.integers(0, 3, size=w.logits.shape).astype(np.float32))
        w.draft[:] = rng.integers(0, V, size=w.draft.shape)
    d = DevWorkload(w)
    mask = d.mask()[0] if with_mask else None
    out = tv.accept_fused(d.logits, d.draft, d.parent, mask, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    _check(w, *out)


def test_accept_fused_reuses_its_workspace():
    """Counters return to zero: consecutive calls on one workspace (different inputs) all match."""
    nb, B, V = 5, 48, 2000
    ws = torch.zeros(tv.accept_fused_workspace_size(V, B, nb), dtype=torch.uint8, device="cuda")
    for seed in range(4):
        w = _workload(100 + seed, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
        d = DevWorkload(w)
        out = tv.accept_fused(d.logits, d.draft, d.parent, None, status=d.status, workspace=ws)
        torch.cuda.synchronize()
        assert d.status.item() == 0
        _check(w, *out)
    counters = ws[nb * B * 8:].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0


def test_accept_fused_reports_non_topological_parent():
    nb, B, V = 2, 8, 50
    w = _workload(7, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    w.parent[1, 4] = 6  # a later node as parent
    d = DevWorkload(w)
    am, n_acc, path, bonus = tv.accept_fused(d.logits, d.draft, d.parent, None, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 2  # TV_ERR_NOT_TOPOLOGICAL
    # the bad sequence falls back to the root alone; the good one is exact
    assert n_acc[1].item() == 0 and path[1].cpu().tolist() == [0] + [-1] * (B - 1)
    assert bonus[1].item() == int(oracle.argmax(w.logits[B:B + 1])[0])
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits[:B], w.draft[:1], w.parent[:1])
    assert n_acc[0].item() == r_n[0] and path[0].cpu().tolist() == r_path[0].tolist()


def test_accept_fused_in_a_cuda_graph():
    nb, B, V = 4, 64, 30000
    w = _workload(11, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    d = DevWorkload(w)
    ws = torch.zeros(tv.accept_fused_workspace_size(V, B, nb), dtype=torch.uint8, device="cuda")
    out = (torch.empty(nb * B, dtype=torch.int32, device="cuda"), torch.empty(nb, dtype=torch.int32, device="cuda"),
           torch.empty((nb, B), dtype=torch.int32, device="cuda"), torch.empty(nb, dtype=torch.int32, device="cuda"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tv.accept_fused(d.logits, d.draft, d.parent, None, status=d.status, out=out, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tv.accept_fused(d.logits, d.draft, d.parent, None, status=d.status, out=out, workspace=ws, stream=s)
    for t in out:
        t.fill_(-7)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert d.status.item() == 0
    _check(w, *out)
