"""GPU parity at the five benchmark workloads' full sizes, in the benchmark's launch configuration.

Each workload (the seeded inputs bench.py times) runs through the C ABI exactly as the
benchmark launches it (default CTA count = one per SM, split-KV merge included).  Masks,
depths, argmax, accepted length/path/bonus are compared bit-exactly over every row.  The
attention output is compared element by element on sampled (sequence, kv head) units,
each of which the fp64 oracle recomputes from a slice of the inputs (that unit's query
heads and kv-head slice of the paged cache); every other row is checked for finiteness
and for the LSE lower bound that holds at any size (a row sees at least one key, so
LSE >= the largest scaled score, which is >= the score of the row's own tree key).  The
commit of the accepted branch (tv_kv_commit) runs last, on the device's own acceptance
outputs, and both whole caches are compared bit-exactly with the oracle's commit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.helpers import DevWorkload, assert_attn_close, bf16_host

pytestmark = pytest.mark.gpu

# (config, sampled (sequence, kv head) units); first, last and interior units, so that
# row tiles cut between CTAs (split-KV pieces + merge) are among them
UNITS = {
    1: [(0, 0), (0, 3), (0, 7)],
    2: [(0, 0), (0, 5)],
    3: [(0, 0), (3, 4), (7, 7)],
    4: [(0, 0), (13, 2), (31, 3)],
    5: [(0, 0), (3, 7)],
}


def _unit_oracle(w, b, g):
    """fp64 oracle O, LSE for sequence b and kv head g only, from sliced inputs."""
    G = w.Hq // w.Hkv
    q = w.q[b * w.B:(b + 1) * w.B, g * G:(g + 1) * G]
    kc = w.k_cache[:, g:g + 1]
    vc = w.v_cache[:, g:g + 1]
    return oracle.attn(q, kc, vc, w.block_table[b:b + 1], w.prefix_lens[b:b + 1], w.parent[b:b + 1], G, 1)


@pytest.mark.parametrize("config", sorted(UNITS))
def test_config_full_size(config):
    w = wl.config(config, seed=1234)
    d = DevWorkload(w)
    mask, depth = d.mask()
    O, L = d.attn(mask)
    am, n_acc, path, bonus = d.accept(mask)
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

    G = w.Hq // w.Hkv
    O_all = O.view(w.nb, w.B, w.Hq, w.D)
    L_all = L.view(w.nb, w.B, w.Hq)
    for b, g in UNITS[config]:
        O_ref, L_ref = _unit_oracle(w, b, g)
        O_u = O_all[b, :, g * G:(g + 1) * G].reshape(w.B, G, w.D)
        L_u = L_all[b, :, g * G:(g + 1) * G].reshape(w.B, G)
        assert_attn_close(O_u, L_u, O_ref, L_ref, w)

    # commit of the accepted branch, fed by the device's own acceptance: bit-exact caches and lengths
    import tree_speculative_decoding_tv_gb300 as tv
    new_pl = tv.kv_commit(d.k.view(torch.int16), d.v.view(torch.int16), d.bt, d.pl, n_acc, path, status=d.status)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    k_ref, v_ref, pl_ref = oracle.kv_commit(w.k_cache, w.v_cache, w.block_table, w.prefix_lens, r_n, r_path)
    assert np.array_equal(new_pl.cpu().numpy(), pl_ref)
    assert np.array_equal(d.k.view(torch.int16).cpu().numpy().view(np.uint16), k_ref)
    assert np.array_equal(d.v.view(torch.int16).cpu().numpy().view(np.uint16), v_ref)
    del k_ref, v_ref

    # any size: finite outputs, and LSE >= the scaled score of the row's own key (its tree slot)
    assert torch.isfinite(O).all() and torch.isfinite(L).all()
    q = bf16_host(d.q).reshape(w.nb, w.B, w.Hq, w.D)
    scale = 1.0 / np.sqrt(w.D)
    L_h = L_all.cpu().numpy()
    for b in range(w.nb):
        P = int(w.prefix_lens[b])
        for i in (0, w.B - 1):
            t = P + i
            page = w.block_table[b, t // 16]
            for h in (0, w.Hq - 1):
                k = wl.bf16_to_f32(w.k_cache[page, h // G, t % 16]).astype(np.float64)
                assert L_h[b, i, h] >= scale * float(q[b, i, h] @ k) - 1e-3
