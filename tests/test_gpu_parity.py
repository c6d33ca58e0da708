"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bars: masks, depths, argmax, accepted length/path/bonus bit-exact; attention
O within max|dO| <= 2e-2 (bf16 output vs fp64 oracle) and LSE within 1e-3
(natural log), element by element.
"""
import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import DevWorkload, assert_attn_close

pytestmark = pytest.mark.gpu


def _trees(seed, B, nb, kind="mixed"):
    rng = np.random.default_rng(seed)
    out = []
    for b in range(nb):
        k = (b + seed) % 3 if kind == "mixed" else {"chain": 3, "star": 4}[kind]
        if k == 0:
            out.append(wl.tree_window(rng, B, 4))
        elif k == 1:
            out.append(wl.tree_best_first(rng, B, child_cap=4, max_depth=B))
        elif k == 2:
            out.append(np.array([-1] + [int(rng.integers(0, i)) for i in range(1, B)], np.int32))
        elif k == 3:
            out.append(np.arange(-1, B - 1, dtype=np.int32))
        else:
            out.append(np.array([-1] + [0] * (B - 1), np.int32))
    return out


def _workload(seed, nb, B, Hq, Hkv, prefix, V=1000, kind="mixed", shuffle=True):
    return wl.make_workload("parity", nb, B, Hq, Hkv, 128, V, prefix, _trees(seed, B, nb, kind), seed,
                            shuffle_pages=shuffle, extra_pages=2)


# -------------------------------------------------------------------- ancestor masks

@pytest.mark.parametrize("B", [1, 2, 15, 16, 17, 31, 32, 33, 64, 100, 255, 256])
def test_mask_bit_exact(B):
    w = _workload(B, nb=5, B=B, Hq=8, Hkv=2, prefix=[3] * 5, V=16)
    d = DevWorkload(w)
    mask, depth = d.mask()
    torch.cuda.synchronize()
    ref_mask, ref_depth = oracle.build_mask(w.parent)
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), ref_mask)
    assert np.array_equal(depth.cpu().numpy(), ref_depth)
    assert d.status.item() == 0


def test_mask_reports_non_topological_parent():
    parent = torch.tensor([[-1, 0, 1, 2], [-1, 2, 0, 1], [0, 0, 1, 2]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    import tree_speculative_decoding_tv_gb300 as tv
    tv.build_mask(parent, status=status)
    torch.cuda.synchronize()
    assert status.item() == 2  # TV_ERR_NOT_TOPOLOGICAL


# ------------------------------------------------------- argmax and acceptance

# (100, 32768): rows of exactly 8 chunks (one per warp of a CTA); (200, 40961): 1200 ragged,
# unaligned rows of 11 chunks; (3, 65537): 17 chunks, the last one a single element
@pytest.mark.parametrize("B,V", [(1, 7), (7, 3), (16, 4096), (33, 1001), (64, 5), (256, 4099), (3, 300001),
                                 (100, 32768), (200, 40961), (3, 65537)])
def test_accept_bit_exact(B, V):
    rng = np.random.default_rng(B * 1000 + V)
    nb = 6
    w = _workload(B + V, nb=nb, B=B, Hq=8, Hkv=2, prefix=[1] * nb, V=V)
    if V <= 7:  # tiny vocab: many ties and many accepted edges
        w.logits[:] = wl.f32_to_bf16(rng.integers(0, 3, size=w.logits.shape).astype(np.float32))
        w.draft[:] = rng.integers(0, V, size=w.draft.shape)
    d = DevWorkload(w)
    mask, _ = d.mask()
    am, n_acc, path, bonus = d.accept(mask)
    torch.cuda.synchronize()
    r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
    assert np.array_equal(am.cpu().numpy(), r_am)
    assert np.array_equal(n_acc.cpu().numpy(), r_n)
    assert np.array_equal(path.cpu().numpy(), r_path)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)
    assert d.status.item() == 0


@pytest.mark.parametrize("V", [1003, 2048, 4104])
def test_argmax_edge_values(V):
    # ties, signed zeros, NaNs, infinities; V = 1003 leaves rows unaligned, V = 4104 splits each
    # row over two chunks whose keys the acceptance kernel combines
    rows = np.full((6, V), 0xBF80, dtype=np.uint16)            # -1.0 everywhere
    rows[0, [5, 700]] = 0x4000                                   # tie between 5 and 700 -> 5
    rows[1, :] = 0x8000
    rows[1, 900] = 0x0000                                        # -0 everywhere, +0 late -> index 0
    rows[2, [10, 600]] = 0x7FC0                                  # NaNs -> first NaN (10)
    rows[2, 3] = 0x7F80                                          # +inf before the NaN
    rows[3, :] = 0xFF80                                          # all -inf -> 0
    rows[4, V - 1] = 0x3F80                                      # max in the tail -> V-1
    rows[5, 0] = 0xFFC1                                          # negative NaN first -> 0
    nb, B = 1, 6
    parent = np.array([[-1, 0, 1, 2, 3, 4]], np.int32)
    logits = torch.from_numpy(rows.view(np.int16)).cuda()
    d_parent = torch.from_numpy(parent).cuda()
    import tree_speculative_decoding_tv_gb300 as tv
    mask, _ = tv.build_mask(d_parent)
    draft = torch.zeros((nb, B), dtype=torch.int32, device="cuda")
    am, *_ = tv.accept(logits, draft, d_parent, mask)
    torch.cuda.synchronize()
    ref = oracle.argmax(rows)
    assert am.cpu().numpy().tolist() == ref.tolist() == [5, 0, 10, 0, V - 1, 0]


def test_argmax_edge_values_across_spans():
    """V = 151936 (38 chunks of 4096): ties, signed zeros, NaNs and infinities whose candidates
    sit in chunks that different warps reduce, combined through the row's key."""
    V = 151936
    rows = np.full((6, V), 0xBF80, dtype=np.uint16)            # -1.0 everywhere
    rows[0, [5, V - 3]] = 0x4000                                 # tie, first and last chunk -> 5
    rows[1, :] = 0x8000
    rows[1, 100000] = 0x0000                                     # -0 everywhere, +0 late -> index 0
    rows[2, [140000, 150000]] = 0x7FC0                           # NaNs late -> the first NaN
    rows[2, 3] = 0x7F80                                          # +inf early, in another chunk
    rows[3, :] = 0xFF80                                          # all -inf -> 0
    rows[4, [40000, 80000, V - 1]] = [0x3F80, 0x3F80, 0x4000]    # max in the tail -> V-1
    rows[5, 4096 * 16 + 1] = 0x4100                              # a single maximum mid-row
    nb, B = 1, 6
    parent = np.array([[-1, 0, 1, 2, 3, 4]], np.int32)
    logits = torch.from_numpy(rows.view(np.int16)).cuda()
    d_parent = torch.from_numpy(parent).cuda()
    import tree_speculative_decoding_tv_gb300 as tv
    mask, _ = tv.build_mask(d_parent)
    draft = torch.zeros((nb, B), dtype=torch.int32, device="cuda")
    am, *_ = tv.accept(logits, draft, d_parent, mask)
    torch.cuda.synchronize()
    ref = oracle.argmax(rows)
    assert am.cpu().numpy().tolist() == ref.tolist() == [5, 0, 140000, 0, V - 1, 4096 * 16 + 1]


# --------------------------------------------------- attention and split-KV merge

ATTN_CASES = [
    # (nb, B, Hq, Hkv, prefixes)
    (1, 16, 32, 8, [512]),               # the 8B shape with budget 16
    (1, 1, 8, 2, [200]),                 # single node: decode attention
    (2, 17, 8, 1, [0, 37]),              # P = 0, ragged tails, G = 8
    (3, 33, 4, 4, [129, 1, 300]),        # G = 1, tree straddling tiles
    (2, 64, 16, 8, [1000, 77]),          # G = 2
    (1, 255, 32, 8, [250]),              # B = 255, several M tiles
    (1, 256, 16, 1, [130]),              # G = 16, 32 M tiles
    (2, 100, 32, 4, [513, 2047]),        # G = 8, 30B-A3B shape
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=[f"nb{c[0]}_B{c[1]}_Hq{c[2]}_Hkv{c[3]}" for c in ATTN_CASES])
@pytest.mark.parametrize("num_ctas", [0, 1, 5])
def test_attention_parity(case, num_ctas):
    nb, B, Hq, Hkv, prefix = case
    w = _workload(7 * B + nb, nb, B, Hq, Hkv, prefix, V=8)
    d = DevWorkload(w)
    mask, _ = d.mask()
    O, L = d.attn(mask, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert d.status.item() == 0
    O_ref, L_ref = oracle.attn_workload(w)
    assert_attn_close(O, L, O_ref, L_ref, w)


@pytest.mark.parametrize("kind", ["chain", "star"])
def test_attention_special_trees(kind):
    w = _workload(3, 2, 48, 32, 8, [300, 0], V=8, kind=kind)
    d = DevWorkload(w)
    mask, _ = d.mask()
    O, L = d.attn(mask)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attn_workload(w)
    assert_attn_close(O, L, O_ref, L_ref, w)


def test_attention_many_ctas_ragged_prefixes():
    """Ragged prefixes with more CTAs than tiles per row tile: every row tile is split and merged."""
    prefix = [5000, 1, 2222, 4097, 0, 129]
    w = _workload(11, 6, 40, 32, 8, prefix, V=8)
    d = DevWorkload(w)
    mask, _ = d.mask()
    for ctas in (0, 7, 300):
        O, L = d.attn(mask, num_ctas=ctas)
        torch.cuda.synchronize()
        O_ref, L_ref = oracle.attn_workload(w) if ctas == 0 else (O_ref, L_ref)
        assert_attn_close(O, L, O_ref, L_ref, w)
    assert d.status.item() == 0


# tv_attn's workspace per CTA: 128 bytes of arrival counters, four 32 KB fp16 partial
# outputs and their four 512-byte LSE rows
ATTN_WS_BLOCK = 128 + 4 * 32768 + 4 * 512


def test_attention_workspace_reused_across_shapes():
    """One workspace, zeroed once, serves split-KV calls of different shapes and CTA counts
    (pair tiles, a single-tile unit, ragged prefixes), merged in place or by the merge
    kernel: every call matches the oracle, leaves every arrival counter zero, and a repeated
    call gives bit-identical outputs (the merge does not depend on which CTA lands last)."""
    cases = [
        # (workload, CTA counts): 300 and 0 (one per SM) take the merge kernel here, 7 and
        # fewer merge in place (fewer CTA groups than twice the units)
        (_workload(21, 6, 40, 32, 8, [5000, 1, 2222, 4097, 0, 129], V=8), (300, 7, 0)),  # pairs, ragged
        (_workload(22, 2, 16, 32, 8, [4000, 1500], V=8), (300, 7, 0)),                   # one M tile per unit
        (_workload(23, 1, 256, 32, 8, [3000], V=8), (300, 7, 0)),                        # four pair tiles per unit
        # two units, one 157 KV tiles long: on 3 CTAs it is cut into three pieces (one from
        # a CTA whose whole share lies inside it), merged in place
        (_workload(24, 2, 16, 8, 1, [20000, 10], V=8), (3, 2, 300)),
    ]
    ws = torch.zeros(300 * ATTN_WS_BLOCK, dtype=torch.uint8, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for w, ctas_list in cases:
        d = DevWorkload(w)
        mask, _ = d.mask()
        O_ref, L_ref = oracle.attn_workload(w)
        for ctas in ctas_list:
            O, L = tv.attn(d.q, d.k, d.v, d.bt, d.pl, mask, status=d.status, num_ctas=ctas, workspace=ws)
            O2, L2 = tv.attn(d.q, d.k, d.v, d.bt, d.pl, mask, status=d.status, num_ctas=ctas, workspace=ws)
            torch.cuda.synchronize()
            assert d.status.item() == 0
            assert_attn_close(O, L, O_ref, L_ref, w)
            assert torch.equal(O.view(torch.int16), O2.view(torch.int16)) and torch.equal(L, L2)
            n = ctas if ctas > 0 else sms
            counters = ws[: n * ATTN_WS_BLOCK].view(n, ATTN_WS_BLOCK)[:, :128]
            assert int(counters.count_nonzero()) == 0


def test_attention_long_prefix_many_pieces():
    """A 65536-token prefix over 8 single-tile units: one CTA per SM cuts every row tile into
    about twenty pieces (the merge kernel's batches of four, several times over); 15 CTAs
    (fewer groups than twice the units) merge each tile's two or three pieces in place."""
    w = _workload(25, 1, 16, 32, 8, [65536], V=8)
    d = DevWorkload(w)
    mask, _ = d.mask()
    O_ref, L_ref = oracle.attn_workload(w)
    ws = torch.zeros(300 * ATTN_WS_BLOCK, dtype=torch.uint8, device="cuda")
    for ctas in (0, 15):
        O, L = tv.attn(d.q, d.k, d.v, d.bt, d.pl, mask, status=d.status, num_ctas=ctas, workspace=ws)
        torch.cuda.synchronize()
        assert d.status.item() == 0
        assert_attn_close(O, L, O_ref, L_ref, w)


def test_attention_explicit_scale():
    w = _workload(12, 1, 20, 8, 2, [77], V=8)
    d = DevWorkload(w)
    mask, _ = d.mask()
    O, L = d.attn(mask, scale=0.02)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle.attn_workload(w, scale=0.02)
    assert_attn_close(O, L, O_ref, L_ref, w)


def test_attention_reports_short_block_table():
    w = _workload(13, 2, 16, 8, 2, [40, 10], V=8)
    d = DevWorkload(w)
    mask, _ = d.mask()
    d.pl[1] = 10_000  # prefix longer than the block table covers
    d.attn(mask)
    torch.cuda.synchronize()
    assert d.status.item() == 1  # TV_ERR_INVALID_ARG


def test_accept_workspace_is_left_zeroed_and_reused():
    """tv_accept combines per-row maxima into zeroed keys and resets them after the walk:
    two calls in a row on one workspace (different vocabularies and trees) are both
    bit-exact, and the workspace is all zero after each."""
    ws = None
    for seed, (nb, B, V) in ((11, (3, 40, 9000)), (12, (2, 256, 151936)), (13, (5, 7, 33))):
        rng = np.random.default_rng(seed)
        trees = [wl.tree_best_first(rng, B, child_cap=3, max_depth=B) for _ in range(nb)]
        w = wl.make_workload("ws-reuse", nb, B, 8, 2, 128, V, [3] * nb, trees, seed, extra_pages=1)
        d = DevWorkload(w)
        need = tv.accept_workspace_size(V, B, nb)
        if ws is None:
            ws = torch.zeros(2 * 256 * 8 * 8, dtype=torch.uint8, device="cuda")
        assert need <= ws.numel()
        am, n_acc, path, bonus = tv.accept(d.logits, d.draft, d.parent, None, status=d.status, workspace=ws)
        torch.cuda.synchronize()
        assert d.status.item() == 0
        r_am, r_n, r_path, r_bonus = oracle.accept(w.logits, w.draft, w.parent)
        assert np.array_equal(am.cpu().numpy(), r_am)
        assert np.array_equal(n_acc.cpu().numpy(), r_n)
        assert np.array_equal(path.cpu().numpy(), r_path)
        assert np.array_equal(bonus.cpu().numpy(), r_bonus)
        assert int(ws.count_nonzero()) == 0
