"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching a device."""
import ctypes as C
import os
import re

import pytest

import tree_speculative_decoding_tv_gb300 as tv
from tree_speculative_decoding_tv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


@pytest.fixture(scope="module")
def L():
    from tree_speculative_decoding_tv_gb300 import build
    build.build()
    return tv.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TV_API\s+[\w\s\*]*?\b(tv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_symbols() == sorted(binding.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_status_strings(L):
    names = [tv.status_str(i) for i in range(7)]
    assert names == ["TV_OK", "TV_ERR_INVALID_ARG", "TV_ERR_NOT_TOPOLOGICAL", "TV_ERR_UNSUPPORTED_SHAPE",
                     "TV_ERR_CUDA", "TV_ERR_TIMEOUT", "TV_ERR_UNIMPLEMENTED"]
    assert tv.status_str(99) == "TV_ERR_UNKNOWN"
    assert L.tv_version() == 100


FAKE = 0x10000  # an aligned non-null address that is never dereferenced: every case below fails validation first


def test_build_mask_argument_checks(L):
    P = C.c_void_p
    assert L.tv_build_mask(P(FAKE), 16, 0, P(FAKE), None, None, None) == 0        # nb = 0: nothing to do
    assert L.tv_build_mask(P(FAKE), 0, 1, P(FAKE), None, None, None) == 3         # B = 0
    assert L.tv_build_mask(P(FAKE), 257, 1, P(FAKE), None, None, None) == 3       # B > 256
    assert L.tv_build_mask(None, 16, 1, P(FAKE), None, None, None) == 1           # null parent
    assert L.tv_build_mask(P(FAKE), 16, 1, None, None, None, None) == 1           # null mask
    assert L.tv_build_mask(P(FAKE + 2), 16, 1, P(FAKE), None, None, None) == 1    # misaligned parent
    assert L.tv_build_mask(P(FAKE), 16, -1, P(FAKE), None, None, None) == 1       # nb < 0


def _args(**kw):
    a = dict(q_d=FAKE, k_cache_d=FAKE, v_cache_d=FAKE, block_table_d=FAKE, prefix_lens_d=FAKE, mask_d=FAKE,
             o_d=FAKE, lse_d=FAKE, dev_status_d=None, nb=1, B=16, Hq=32, Hkv=8, D=128, page_size=16,
             num_blocks=40, max_pages=40, scale=0.0, num_ctas=0)
    a.update(kw)
    return binding.AttnArgs(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), 3), (dict(page_size=32), 3), (dict(B=0), 3), (dict(B=257), 3),
    (dict(Hq=24, Hkv=8), 3),                      # G = 3 unsupported
    (dict(Hq=30, Hkv=8), 1),                      # Hq not a multiple of Hkv
    (dict(Hq=64, Hkv=2), 3),                      # G = 32 unsupported
    (dict(q_d=None), 1), (dict(lse_d=None), 1), (dict(mask_d=None), 1),
    (dict(q_d=FAKE + 8), 1),                      # q not 16-byte aligned
    (dict(o_d=FAKE + 4), 1),
    (dict(num_blocks=0), 1), (dict(nb=-1), 1), (dict(num_ctas=-2), 1),
    (dict(max_pages=1 << 27), 3),
])
def test_attn_argument_checks(L, kw, code):
    a = _args(**kw)
    assert L.tv_attn(C.byref(a), C.c_void_p(FAKE), 1 << 30, None) == code
    assert L.tv_attn_workspace_size(C.byref(a)) == 0


def test_attn_null_args(L):
    assert L.tv_attn(None, None, 0, None) == 1
    assert L.tv_attn_workspace_size(None) == 0
    assert L.tv_attn_launches(None) == 0


@pytest.mark.parametrize("kw", [dict(num_ctas=1), dict(num_ctas=152), dict(nb=4, B=256, max_pages=2064,
                                num_blocks=8256, num_ctas=300), dict(nb=32, B=16, Hkv=4, num_ctas=7)])
def test_attn_workspace_is_one_fixed_block_per_cta(L, kw):
    """tv_attn's workspace is one block per CTA whatever the shape: 128 bytes of arrival
    counters, four 32 KB fp16 partial outputs and their four 512-byte LSE rows, so a
    block's counters sit at the same offset for every call that shares the workspace."""
    a = _args(**kw)
    assert L.tv_attn_workspace_size(C.byref(a)) == kw["num_ctas"] * (128 + 4 * 32768 + 4 * 512)


@pytest.mark.parametrize("kw,launches", [
    # 4 sequences x 8 kv heads, 256-node trees (4 pair tiles per unit), 32K prefixes, 152 CTAs:
    # 38 groups over 32 units, so a split tile has about two parts and is merged in place
    (dict(nb=4, B=256, max_pages=2064, num_blocks=8256, num_ctas=152), 1),
    # one sequence: 38 groups over 8 units, many parts per split tile: the merge kernel runs
    (dict(nb=1, B=256, max_pages=272, num_blocks=272, num_ctas=152), 2),
    # 8 sequences x 8 kv heads, 64-node trees (one pair tile per unit): 152 groups, 64 units
    (dict(nb=8, B=64, max_pages=1030, num_blocks=8240, num_ctas=152), 2),
    # 32 sequences x 4 kv heads, 16-node trees: 152 groups over 128 units
    (dict(nb=32, B=16, Hkv=4, max_pages=514, num_blocks=16448, num_ctas=152), 1),
    # every unit fits the grid and the block table covers few KV tiles: nothing is split
    (dict(nb=1, B=16, max_pages=33, num_blocks=33, num_ctas=152), 1),
    # fewer CTAs than pair tiles per unit: one group, nothing is split
    (dict(nb=1, B=256, max_pages=272, num_blocks=272, num_ctas=3), 1),
    (dict(nb=0, num_ctas=152), 0),                 # nothing to do
    (dict(B=0, num_ctas=152), 0),                  # invalid
])
def test_attn_launch_count(L, kw, launches):
    """tv_attn_launches (host-only with an explicit CTA count): one kernel when split tiles
    have about two parts or none, the merge kernel too when they have more."""
    assert L.tv_attn_launches(C.byref(_args(**kw))) == launches


def test_accept_argument_checks(L):
    P = C.c_void_p
    ok = [P(FAKE)] * 4
    base = dict(logits=P(FAKE), V=100, draft=P(FAKE), parent=P(FAKE), mask=P(FAKE), B=16, nb=1)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_accept(d["logits"], d["V"], d["draft"], d["parent"], d["mask"], d["B"], d["nb"], *ok, None,
                           d.get("ws", P(FAKE)), d.get("ws_bytes", 1 << 30), None)

    assert call(nb=0) == 0
    assert call(V=0) == 1
    assert call(B=0) == 3 and call(B=300) == 3
    assert call(logits=None) == 1 and call(parent=None) == 1 and call(mask=P(FAKE + 2)) == 1
    assert call(logits=P(FAKE + 1)) == 1
    assert call(draft=P(FAKE + 2)) == 1
    assert call(ws=None) == 1 and call(ws_bytes=8) == 1 and call(ws=P(FAKE + 4)) == 1
    # one 8-byte argmax key per logits row, whatever V
    assert L.tv_accept_workspace_size(151936, 256, 1) == 256 * 8
    assert L.tv_accept_workspace_size(4096, 16, 2) == 32 * 8
    assert L.tv_accept_workspace_size(0, 16, 1) == 0 and L.tv_accept_workspace_size(10, 300, 1) == 0


def test_accept_entry_points_reject_a_vocabulary_near_int_max(L):
    # the kernels index a row with 32-bit ints: V must stay 8192 below INT32_MAX
    P = C.c_void_p
    f = P(FAKE)
    for V in (2**31 - 1, 2**31 - 8192):
        assert L.tv_accept(f, V, f, f, f, 16, 1, f, f, f, f, None, f, 1 << 40, None) == 3
        assert L.tv_accept_fused(f, V, f, f, f, 16, 1, f, f, f, f, None, f, 1 << 40, None) == 3
        assert L.tv_accept_noalloc(f, V, f, f, f, 16, 1, f, f, f, f, None, None) == 3
    # the unit count (rows x 4096-logit units) must stay below 2^31 as well
    assert L.tv_accept_noalloc(f, 2**31 - 8193, f, f, f, 256, 32, f, f, f, f, None, None) == 3


def test_selftest_wait_argument_checks(L):
    P = C.c_void_p
    assert L.tv_selftest_wait(0, P(FAKE), None) == 1
    assert L.tv_selftest_wait(1000001, P(FAKE), None) == 1
    assert L.tv_selftest_wait(1000, None, None) == 1
    assert L.tv_selftest_wait(1000, P(FAKE + 2), None) == 1


def test_accept_fused_argument_checks(L):
    P = C.c_void_p
    ok = [P(FAKE)] * 4
    base = dict(logits=P(FAKE), V=100, draft=P(FAKE), parent=P(FAKE), mask=P(FAKE), B=16, nb=1)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_accept_fused(d["logits"], d["V"], d["draft"], d["parent"], d["mask"], d["B"], d["nb"], *ok, None,
                                 d.get("ws", P(FAKE)), d.get("ws_bytes", 1 << 30), None)

    assert call(nb=0) == 0
    assert call(V=0) == 1
    assert call(B=0) == 3 and call(B=300) == 3
    assert call(logits=None) == 1 and call(parent=None) == 1
    assert call(mask=P(FAKE + 2)) == 1 and call(logits=P(FAKE + 1)) == 1
    assert call(ws=None) == 1 and call(ws_bytes=16 * 8) == 1 and call(ws=P(FAKE + 4)) == 1
    # keys, then one 32-bit counter per sequence
    assert L.tv_accept_fused_workspace_size(151936, 256, 1) == 256 * 8 + 4
    assert L.tv_accept_fused_workspace_size(4096, 16, 3) == 48 * 8 + 12
    assert L.tv_accept_fused_workspace_size(0, 16, 1) == 0


def test_kv_commit_argument_checks(L):
    P = C.c_void_p
    base = dict(k=P(FAKE), v=P(FAKE), bt=P(FAKE), pl=P(FAKE), n=P(FAKE), path=P(FAKE), nb=2, B=16, Hkv=8, D=128,
                page=16, blocks=64, pages=8, out=P(FAKE + 4096))

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_kv_commit(d["k"], d["v"], d["bt"], d["pl"], d["n"], d["path"], d["nb"], d["B"], d["Hkv"], d["D"],
                              d["page"], d["blocks"], d["pages"], d["out"], None, None)

    assert call(nb=0) == 0                                    # nothing to do, nothing enqueued
    assert call(nb=-1) == 1 and call(Hkv=0) == 1 and call(blocks=0) == 1
    assert call(B=0) == 3 and call(B=257) == 3 and call(D=64) == 3 and call(page=32) == 3
    assert call(k=None) == 1 and call(path=None) == 1 and call(out=None) == 1
    assert call(out=P(FAKE)) == 1                             # new prefix lengths may not overwrite the old
    assert call(k=P(FAKE + 8)) == 1 and call(n=P(FAKE + 2)) == 1


def test_build_tree_argument_checks(L):
    P = C.c_void_p
    base = dict(lp=P(FAKE), tk=P(FAKE), nb=2, D=16, K=8, B=256, w=1, par=P(FAKE), tok=P(FAKE), sc=P(FAKE))

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_build_tree(d["lp"], d["tk"], d["nb"], d["D"], d["K"], d["B"], d["w"], d["par"], d["tok"], d["sc"],
                               None, None)

    assert call(nb=0) == 0
    assert call(nb=-1) == 1 and call(D=0) == 1 and call(K=0) == 1 and call(w=0) == 1
    assert call(B=0) == 3 and call(B=257) == 3 and call(K=40000) == 3
    assert call(lp=None) == 1 and call(sc=None) == 1 and call(tk=P(FAKE + 2)) == 1
    assert call(D=1, K=8, B=10) == 1          # the full tree of depth 1 holds 9 nodes
    assert call(D=1, K=8, B=9, nb=0) == 0 and call(D=2, K=2, B=8, nb=0) == 1


def test_gdn_tree_argument_checks(L):
    P = C.c_void_p
    base = dict(q=P(FAKE), k=P(FAKE), v=P(FAKE), a=P(FAKE), b=P(FAKE), s=P(FAKE), par=P(FAKE), nb=1, B=128, H=32, D=128,
                o=P(FAKE), ws=P(FAKE), wsb=1 << 30)

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_gdn_tree(d["q"], d["k"], d["v"], d["a"], d["b"], d["s"], d["par"], d["nb"], d["B"], d["H"], d["D"],
                             d["o"], d["ws"], d["wsb"], None, None)

    assert call(nb=0) == 0
    assert call(nb=-1) == 1 and call(H=0) == 1
    assert call(B=0) == 3 and call(B=257) == 3 and call(D=64) == 3
    assert call(q=None) == 1 and call(s=None) == 1 and call(o=None) == 1
    assert call(k=P(FAKE + 8)) == 1 and call(s=P(FAKE + 4)) == 1 and call(a=P(FAKE + 2)) == 1
    assert call(ws=None) == 1 and call(wsb=16) == 1
    # per (sequence, head, value-column slice of 32): records [B][B]; B > 128 adds two [B][32] row slices
    assert L.tv_gdn_tree_workspace_size(1, 128, 32, 128) == 32 * 4 * 128 * 128 * 16
    assert L.tv_gdn_tree_workspace_size(2, 256, 4, 128) == 2 * 4 * 4 * (256 * 256 * 16 + 2 * 256 * 32 * 4)
    assert L.tv_gdn_tree_workspace_size(1, 128, 32, 64) == 0


def test_gdn_commit_argument_checks(L):
    P = C.c_void_p
    base = dict(k=P(FAKE), v=P(FAKE), a=P(FAKE), b=P(FAKE), s=P(FAKE), n=P(FAKE), path=P(FAKE), nb=1, B=128, H=32,
                D=128, o=P(FAKE))

    def call(**kw):
        d = dict(base)
        d.update(kw)
        return L.tv_gdn_commit(d["k"], d["v"], d["a"], d["b"], d["s"], d["n"], d["path"], d["nb"], d["B"], d["H"],
                               d["D"], d["o"], None, None)

    assert call(nb=0) == 0
    assert call(nb=-1) == 1 and call(H=0) == 1
    assert call(B=0) == 3 and call(B=257) == 3 and call(D=64) == 3
    assert call(k=None) == 1 and call(path=None) == 1 and call(o=None) == 1
    assert call(k=P(FAKE + 8)) == 1 and call(s=P(FAKE + 2)) == 1 and call(n=P(FAKE + 1)) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_accept_binding_refuses_pageable_or_host_tree_arrays():
    """The acceptance wrappers put outputs and workspaces on the tree arrays' device; host tree
    arrays, or logits in pageable host memory, are refused before anything is launched."""
    import torch
    import tree_speculative_decoding_tv_gb300 as tv
    logits = torch.zeros((4, 16), dtype=torch.bfloat16)
    parent = torch.tensor([[-1, 0, 1, 2]], dtype=torch.int32)
    draft = torch.zeros((1, 4), dtype=torch.int32)
    for fn in (tv.accept, tv.accept_fused, tv.accept_noalloc):
        with pytest.raises(ValueError):
            fn(logits, draft, parent, None)
