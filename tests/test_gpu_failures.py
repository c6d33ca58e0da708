"""Failure detection on the GPU, without faulting or hanging it.

The library's kernels never trap: data-dependent problems go to a device status word
and every device-side wait has a time limit.  These tests drive both paths on purpose:
  - a block-table entry that points outside the cache, inside the range the attention
    needs, must report TV_ERR_INVALID_ARG (the kernel bounds-checks every page id and
    reads zeros instead), while entries past the needed range are never read;
  - a kernel whose barrier wait can never complete (tv_selftest_wait: nothing arrives)
    must give up after its limit, report TV_ERR_TIMEOUT, free its tensor memory and
    leave the context usable for the next call.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload, assert_attn_close

pytestmark = pytest.mark.gpu


def _small(seed=3):
    rng = np.random.default_rng(seed)
    trees = [wl.tree_window(rng, 24, 4) for _ in range(2)]
    return wl.make_workload("failures", 2, 24, 8, 2, 128, 1000, [100, 37], trees, seed)


@pytest.mark.parametrize("bad", ["num_blocks", "negative"])
def test_block_id_out_of_range_is_reported(bad):
    w = _small()
    d = DevWorkload(w)
    bt = d.bt.clone()
    bt[1, 2] = w.num_blocks if bad == "num_blocks" else -7  # page 2 of sequence 1 is needed (P = 37)
    O, L = tv.attn(d.q, d.k, d.v, bt, d.pl, None, status=d.status, parent=d.parent)
    torch.cuda.synchronize()
    assert d.status.item() == 1  # TV_ERR_INVALID_ARG
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
    # sequence 0 is untouched by the bad entry and still matches the oracle
    O_ref, L_ref = oracle.attn_workload(w)
    rows = np.arange(w.B)
    assert_attn_close(O[:w.B], L[:w.B], O_ref[rows], L_ref[rows], w)


def test_block_table_entries_past_the_needed_range_are_not_read():
    w = _small()
    d = DevWorkload(w)
    O_ref, L_ref = tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, parent=d.parent)
    wide = torch.full((w.nb, w.max_pages + 5), 1 << 30, dtype=torch.int32, device="cuda")
    wide[:, :w.max_pages] = d.bt
    for b in range(w.nb):  # poison every entry a sequence does not need
        need = (int(w.prefix_lens[b]) + w.B + 15) // 16
        wide[b, need:] = -(1 << 20)
    O, L = tv.attn(d.q, d.k, d.v, wide, d.pl, None, status=d.status, parent=d.parent)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    assert torch.equal(O.view(torch.int16), O_ref.view(torch.int16)) and torch.equal(L, L_ref)


def test_bounded_wait_times_out_cleanly_and_the_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tv.selftest_wait(1000, status)  # 1 ms on a barrier nothing arrives at
    torch.cuda.synchronize()
    assert status.item() == 5  # TV_ERR_TIMEOUT
    # again: its tensor memory was freed, so a second allocation succeeds at once
    status.zero_()
    tv.selftest_wait(200, status)
    torch.cuda.synchronize()
    assert status.item() == 5
    # and the context still runs the real kernels correctly
    w = _small(seed=4)
    d = DevWorkload(w)
    O, L = tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, parent=d.parent)
    am, n_acc, path, bonus = d.accept(None)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    O_ref, L_ref = oracle.attn_workload(w)
    assert_attn_close(O, L, O_ref, L_ref, w)
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am) and np.array_equal(path.cpu().numpy(), r_path)
