"""GPU parity for the commit of the accepted branch (tv_kv_commit) against the oracle.

The commit only moves bf16 rows, so the caches and the new committed lengths are
compared bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload, i32_dev

pytestmark = pytest.mark.gpu


def _root_path(parent, v):
    out = []
    while v != -1:
        out.append(int(v))
        v = int(parent[v])
    return out[::-1]


def _outcome(rng, parent, pick=None):
    nb, B = parent.shape
    n_acc = np.zeros(nb, np.int32)
    path = np.full((nb, B), -1, np.int32)
    for b in range(nb):
        v = int(rng.integers(0, B)) if pick is None else pick(b, B)
        p = _root_path(parent[b], v)
        n_acc[b] = len(p) - 1
        path[b, :len(p)] = p
    return n_acc, path


def _check(w, n_acc, path):
    d = DevWorkload(w)
    new_pl = tv.kv_commit(d.k.view(torch.int16), d.v.view(torch.int16), d.bt, d.pl, i32_dev(n_acc), i32_dev(path),
                          status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    k_ref, v_ref, pl_ref = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, n_acc, path)
    assert np.array_equal(new_pl.cpu().numpy(), pl_ref)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k_ref)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v_ref)


CASES = [  # (nb, B, Hkv, prefixes)
    (1, 1, 8, [100]),
    (3, 16, 8, [0, 15, 33]),
    (2, 64, 4, [4096, 7]),
    (4, 256, 8, [1, 300, 16, 5000]),
    (2, 255, 1, [31, 64]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"nb{c[0]}_B{c[1]}_Hkv{c[2]}" for c in CASES])
@pytest.mark.parametrize("kind", ["random", "deepest", "none"])
def test_kv_commit_bit_exact(case, kind):
    nb, B, Hkv, prefix = case
    rng = np.random.default_rng(B * 7 + nb)
    trees = [wl.tree_best_first(rng, B, child_cap=2, max_depth=B) if b % 2 else
             np.array([-1] + [int(rng.integers(max(0, i - 3), i)) for i in range(1, B)], np.int32)
             for b in range(nb)]
    w = wl.make_workload("commit", nb, B, 2 * Hkv, Hkv, 128, 8, prefix, trees, seed=B + nb, extra_pages=2,
                         with_logits=False)
    if kind == "random":
        n_acc, path = _outcome(rng, w.parent)
    elif kind == "deepest":  # the last node: long paths whose rows mostly move
        n_acc, path = _outcome(rng, w.parent, pick=lambda b, B: B - 1)
    else:
        n_acc, path = _outcome(rng, w.parent, pick=lambda b, B: 0)
    _check(w, n_acc, path)


def test_kv_commit_chain_accepted_in_full_moves_nothing():
    B = 40
    w = wl.make_workload("commit", 2, B, 8, 4, 128, 8, [17, 0], [np.arange(-1, B - 1, dtype=np.int32)] * 2, seed=3,
                         extra_pages=1, with_logits=False)
    path = np.tile(np.arange(B, dtype=np.int32), (2, 1))
    _check(w, np.full(2, B - 1, np.int32), path)


def test_kv_commit_after_device_acceptance():
    """mask -> accept -> commit on the device, fed by the device's own n_acc and path."""
    w = wl.make_workload("commit", 3, 48, 16, 4, 128, 300, [129, 0, 777],
                         lambda r: wl.tree_best_first(r, 48, child_cap=3, max_depth=12), seed=21, extra_pages=2)
    d = DevWorkload(w)
    mask, _ = d.mask()
    am, n_acc, path, bonus = d.accept(mask)
    new_pl = tv.kv_commit(d.k.view(torch.int16), d.v.view(torch.int16), d.bt, d.pl, n_acc, path, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    _, r_n, r_path, _ = oracle.accept(w.logits, w.draft, w.parent)
    k_ref, v_ref, pl_ref = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, r_n, r_path)
    assert np.array_equal(new_pl.cpu().numpy(), pl_ref)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k_ref)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v_ref)


def test_kv_commit_reports_a_bad_path():
    B = 8
    w = wl.make_workload("commit", 2, B, 4, 2, 128, 8, [5, 9], [np.arange(-1, B - 1, dtype=np.int32)] * 2, seed=5,
                         extra_pages=1, with_logits=False)
    d = DevWorkload(w)
    path = np.full((2, B), -1, np.int32)
    path[0, :3] = [0, 1, 2]
    path[1, :3] = [0, 3, 3]  # not increasing
    new_pl = tv.kv_commit(d.k.view(torch.int16), d.v.view(torch.int16), d.bt, d.pl, i32_dev(np.array([2, 2])),
                          i32_dev(path), status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 1  # TV_ERR_INVALID_ARG
    assert new_pl.cpu().numpy().tolist() == [5 + 3, 9]  # the bad sequence stays uncommitted
