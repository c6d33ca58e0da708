"""The folded forms of the step: the mask build inside the attention, and the whole verify step
as attention (from the parent array) + split-KV merge + one-kernel acceptance.

With mask_d NULL the attention derives each row's ancestor bits from the parent array; the
bits, and so every score that is kept or dropped, are the same as with tv_build_mask's
array, and the arithmetic is unchanged, so O and LSE must be bit-identical to the unfolded
call (which the parity tests hold to the oracle).  The folded step's acceptance outputs are
compared with the oracle bit-exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload
from tests.test_gpu_parity import ATTN_CASES, _workload

pytestmark = pytest.mark.gpu


def _attn_both(d, num_ctas=0):
    mask, _ = d.mask()
    O1, L1 = d.attn(mask, num_ctas=num_ctas)
    O2, L2 = tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, num_ctas=num_ctas, parent=d.parent)
    torch.cuda.synchronize()
    return O1, L1, O2, L2


@pytest.mark.parametrize("case", ATTN_CASES, ids=[f"nb{c[0]}_B{c[1]}_Hq{c[2]}_Hkv{c[3]}" for c in ATTN_CASES])
@pytest.mark.parametrize("num_ctas", [0, 7])
def test_attention_from_parents_is_bit_identical(case, num_ctas):
    nb, B, Hq, Hkv, prefix = case
    w = _workload(7 * B + nb, nb, B, Hq, Hkv, prefix, V=8)
    d = DevWorkload(w)
    O1, L1, O2, L2 = _attn_both(d, num_ctas)
    assert d.status.item() == 0
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1, L2)


@pytest.mark.parametrize("kind", ["chain", "star"])
def test_attention_from_parents_special_trees(kind):
    w = _workload(3, 2, 256, 32, 8, [300, 0], V=8, kind=kind)
    d = DevWorkload(w)
    O1, L1, O2, L2 = _attn_both(d)
    assert d.status.item() == 0
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)) and torch.equal(L1, L2)


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
def test_attention_from_parents_full_size(config):
    w = wl.config(config, seed=99, with_logits=False)
    d = DevWorkload(w)
    O1, L1, O2, L2 = _attn_both(d)
    assert d.status.item() == 0
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16)) and torch.equal(L1, L2)


def test_attention_from_parents_reports_non_topological():
    w = _workload(5, 2, 40, 8, 2, [100, 64], V=8)
    w.parent[1, 30] = 35  # a later node as parent
    d = DevWorkload(w)
    tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, parent=d.parent)
    torch.cuda.synchronize()
    assert d.status.item() == 2  # TV_ERR_NOT_TOPOLOGICAL


def test_attention_needs_mask_or_parent():
    w = _workload(5, 1, 8, 8, 2, [10], V=8)
    d = DevWorkload(w)
    with pytest.raises(tv.TVError):
        tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status)


@pytest.mark.parametrize("config", [1, 3])
def test_folded_step_matches_oracle(config):
    """attention from parents + tv_accept_fused without a mask: two launches."""
    w = wl.config(config, seed=5)
    d = DevWorkload(w)
    O, L = tv.attn(d.q, d.k, d.v, d.bt, d.pl, None, status=d.status, parent=d.parent)
    am, n_acc, path, bonus = tv.accept_fused(d.logits, d.draft, d.parent, None, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am) and np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(path.cpu().numpy(), r_path) and np.array_equal(bonus.cpu().numpy(), r_bonus)
    mask, _ = d.mask()
    O1, L1 = d.attn(mask)
    torch.cuda.synchronize()
    assert torch.equal(O.view(torch.int16), O1.view(torch.int16)) and torch.equal(L, L1)


@pytest.mark.parametrize("nb,B,V", [(9, 1, 7), (5, 7, 3), (4, 16, 4096), (3, 33, 1001), (2, 256, 4099)])
def test_accept_without_mask_bit_exact(nb, B, V):
    """tv_accept with mask_d NULL builds the ancestor bits from the parent array itself."""
    rng = np.random.default_rng(nb * 31 + B + V)
    w = _workload(B + V + 3 * nb, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    if V <= 7:
        w.logits[:] = wl.f32_to_bf16(rng.integers(0, 3, size=w.logits.shape).astype(np.float32))
        w.draft[:] = rng.integers(0, V, size=w.draft.shape)
    d = DevWorkload(w)
    am, n_acc, path, bonus = tv.accept(d.logits, d.draft, d.parent, None, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am) and np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(path.cpu().numpy(), r_path) and np.array_equal(bonus.cpu().numpy(), r_bonus)


def test_accept_without_mask_reports_non_topological():
    nb, B, V = 2, 8, 50
    w = _workload(7, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    w.parent[0, 0] = 3  # the root must have parent -1
    d = DevWorkload(w)
    am, n_acc, path, bonus = tv.accept(d.logits, d.draft, d.parent, None, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 2
    assert n_acc[0].item() == 0 and path[0].cpu().tolist() == [0] + [-1] * (B - 1)
    assert np.array_equal(am.cpu().numpy(), oracle.argmax(w.logits))
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits[B:], w.draft[1:], w.parent[1:])
    assert n_acc[1].item() == r_n[0] and path[1].cpu().tolist() == r_path[0].tolist()
