"""GPU parity at the five benchmark workloads' full sizes, in the benchmark's launch configuration.

Each workload (the seeded inputs bench.py times) runs through the C ABI exactly as the
benchmark launches it (default CTA count = one per SM, split-KV merge included).  Masks,
depths, argmax, accepted length/path/bonus are compared bit-exactly over every row, and
the attention output element by element over every row, query head and column against
the fp64 oracle (within the c13 tolerances), for the mask-array form and for the step's
form that derives the ancestor bits from the parent array (which must be bit-identical
to it).  The commit of the accepted branch (tv_kv_commit) runs last, on the device's own
acceptance outputs, and both whole caches are compared bit-exactly with the oracle's
commit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import tree_speculative_decoding_tv_gb300 as tv
from tests.helpers import DevWorkload, assert_attn_close

pytestmark = pytest.mark.gpu

CONFIGS = [1, 2, 3, 4, 5]


@pytest.mark.parametrize("config", CONFIGS)
def test_config_full_size(config):
    w = wl.config(config, seed=1234)
    d = DevWorkload(w)
    mask, depth = d.mask()
    O, L = d.attn(mask)
    O2, L2 = tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, parent=d.parent)
    am, n_acc, path, bonus = d.accept(None)
    torch.cuda.synchronize()
    assert d.status.item() == 0

    ref_mask, ref_depth = oracle.build_mask(w.parent)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), ref_mask)
    assert np.array_equal(depth.cpu().numpy(), ref_depth)

    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am)
    assert np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(path.cpu().numpy(), r_path)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)

    # every row of every (sequence, kv head) unit against the fp64 oracle
    O_ref, L_ref = oracle.attn_workload(w)
    assert_attn_close(O, L, O_ref, L_ref, w)
    del O_ref, L_ref
    # the step's form (ancestor bits from the parent array) gives the same bits
    assert torch.equal(O2.view(torch.int16), O.view(torch.int16)) and torch.equal(L2, L)

    # commit of the accepted branch, fed by the device's own acceptance: bit-exact caches and lengths
    new_pl = tv.kv_commit(d.k.view(torch.int16), d.v.view(torch.int16), d.bt, d.pl, n_acc, path, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    k_ref, v_ref, pl_ref = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, r_n, r_path)
    assert np.array_equal(new_pl.cpu().numpy(), pl_ref)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k_ref)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v_ref)
