"""GPU parity for best-first draft-tree construction (tv_build_tree) against the oracle.

Parents, tokens and scores are compared bit-exactly: both sides accumulate the
scores in fp32 in the same order, so they take the same decisions.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv

pytestmark = pytest.mark.gpu


def _tables(seed, nb, Dmax, K, ties=False):
    rng = np.random.default_rng(seed)
    lp = np.log(rng.dirichlet([0.3] * K, size=(nb, Dmax)) + 1e-12).astype(np.float32)
    if ties:  # few distinct values: many equal scores, so the tie-break decides
        lp = np.round(lp * 2) / 2
    lp = -np.sort(-lp, axis=-1)
    tok = rng.integers(0, 151936, size=(nb, Dmax, K)).astype(np.int32)
    return np.ascontiguousarray(lp), tok


CASES = [  # (nb, Dmax, K, B, w)
    (1, 16, 8, 256, 1),    # the 8B workload's budget
    (1, 16, 8, 256, 4),
    (8, 12, 3, 64, 1),
    (8, 12, 3, 64, 16),
    (32, 15, 2, 16, 1),
    (4, 24, 4, 256, 32),
    (3, 3, 5, 100, 7),
    (2, 1, 40, 41, 1),     # depth 1: a star
    (2, 255, 1, 256, 3),   # one candidate per depth: a chain
]


@pytest.mark.parametrize("case", CASES, ids=[f"nb{c[0]}_D{c[1]}_K{c[2]}_B{c[3]}_w{c[4]}" for c in CASES])
@pytest.mark.parametrize("ties", [False, True])
def test_build_tree_bit_exact(case, ties):
    nb, Dmax, K, B, w = case
    lp, tok = _tables(sum(case) + ties, nb, Dmax, K, ties)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    parent, token, score = tv.build_tree(torch.from_numpy(lp).cuda(), torch.from_numpy(tok).cuda(), B, w,
                                         status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    r_parent, r_token, r_score = oracle.build_tree(lp, tok, B, w)
    assert np.array_equal(parent.cpu().numpy(), r_parent)
    assert np.array_equal(token.cpu().numpy(), r_token)
    assert np.array_equal(score.cpu().numpy(), r_score)


def test_built_tree_feeds_the_mask_build():
    lp, tok = _tables(3, 4, 16, 8)
    parent, token, _ = tv.build_tree(torch.from_numpy(lp).cuda(), torch.from_numpy(tok).cuda(), 256, 2)
    mask, depth = tv.build_mask(parent)
    torch.cuda.synchronize()
    r_parent, _, _ = oracle.build_tree(lp, tok, 256, 2)
    r_mask, r_depth = oracle.build_mask(r_parent)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), r_mask)
    assert np.array_equal(depth.cpu().numpy(), r_depth)


def test_build_tree_reports_unsorted_log_probs():
    lp, tok = _tables(4, 2, 4, 4)
    lp[1, 2] = lp[1, 2][::-1].copy()  # sequence 1, depth 3: ascending
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tv.build_tree(torch.from_numpy(lp).cuda(), torch.from_numpy(tok).cuda(), 50, 1, status=status)
    torch.cuda.synchronize()
    assert status.item() == 1  # TV_ERR_INVALID_ARG
