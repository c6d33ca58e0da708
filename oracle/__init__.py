"""CPU oracle for tree verification (fp64, plain C in ``tv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
The CUDA library neither links nor calls anything here, and nothing here
imports the CUDA package.

Functions (numpy in, numpy out):
  build_mask(parent)                         -> (mask uint32 [nb][B][W], depth int32 [nb][B])
  attn(w_like args...)                       -> (O float64 [nb*B][Hq][D], LSE float64 [nb*B][Hq])
  lse_merge(O_parts, lse_parts)              -> (O, LSE)
  argmax(logits_bf16)                        -> int32 [rows]
  accept(logits, draft, parent)              -> (argmax, n_acc, path, bonus)
  build_tree(logp, tokens, B, w)              -> (parent, token, score)   best-first, top-w rounds
  gdn_tree(q, k, v, alpha, beta, S0, parent)  -> O float64 [nb*B][H][D]  (Gated DeltaNet state per root path)
  kv_commit(k_cache, v_cache, block_table, prefix_lens, n_acc, path)
                                             -> (k_cache', v_cache', new prefix_lens)  (copies)
Every pinned property of these functions is listed in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tv_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libtvoracle.so")
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile tv_oracle.c with the host C compiler (plain -O2, IEEE fp64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = C.CDLL(_LIB)
        P = C.c_void_p
        lib.tvo_build_mask.argtypes = [P, C.c_int, C.c_int, P, P]
        lib.tvo_attn.argtypes = [P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                 C.c_int, C.c_int, C.c_int, C.c_double, C.c_long, C.c_long, P, P,
                                 C.c_int, P]
        lib.tvo_lse_merge.argtypes = [C.c_int, C.c_long, C.c_int, P, P, P, P]
        lib.tvo_argmax.argtypes = [P, C.c_long, C.c_long, P]
        lib.tvo_accept.argtypes = [P, C.c_long, P, P, C.c_int, C.c_int, P, P, P, P]
        lib.tvo_kv_commit.argtypes = [P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                      C.c_int, P]
        lib.tvo_build_tree.argtypes = [P, P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P]
        lib.tvo_gdn_tree.argtypes = [P, P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, P]
        lib.tvo_gdn_commit.argtypes = [P, P, P, P, P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, P]
        for f in (lib.tvo_build_mask, lib.tvo_attn, lib.tvo_lse_merge, lib.tvo_argmax, lib.tvo_accept,
                  lib.tvo_kv_commit, lib.tvo_build_tree, lib.tvo_gdn_tree, lib.tvo_gdn_commit):
            f.restype = C.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc == 1:
        raise OracleError(f"{what}: bad argument")
    if rc == 2:
        raise OracleError(f"{what}: parent array is not a topologically ordered single-root tree")
    if rc:
        raise OracleError(f"{what}: error {rc}")


def build_mask(parent):
    parent = _c(parent, np.int32)
    if parent.ndim == 1:
        parent = parent[None]
    nb, B = parent.shape
    W = (B + 31) // 32
    mask = np.zeros((nb, B, W), dtype=np.uint32)
    depth = np.zeros((nb, B), dtype=np.int32)
    _check(_load().tvo_build_mask(_ptr(parent), B, nb, _ptr(mask), _ptr(depth)), "build_mask")
    return mask, depth


def attn(q, k_cache, v_cache, block_table, prefix_lens, parent, Hq: int, Hkv: int,
         scale: float = 0.0, key_range=(0, -1), threads: int = 0, return_threads: bool = False):
    """Tree-causal paged attention over every node and query head (fp64 results)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    block_table = _c(block_table, np.int32)
    prefix_lens = _c(prefix_lens, np.int32).reshape(-1)
    parent = _c(parent, np.int32)
    nb, B = parent.shape
    D = q.shape[-1]
    page = k_cache.shape[2]
    num_blocks = k_cache.shape[0]
    assert q.shape == (nb * B, Hq, D)
    assert k_cache.shape == (num_blocks, Hkv, page, D) and v_cache.shape == k_cache.shape
    O = np.zeros((nb * B, Hq, D), dtype=np.float64)
    LSE = np.zeros((nb * B, Hq), dtype=np.float64)
    used = C.c_int(0)
    rc = _load().tvo_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(prefix_lens),
                          _ptr(parent), nb, B, Hq, Hkv, D, page, block_table.shape[1], num_blocks,
                          float(scale), int(key_range[0]), int(key_range[1]), _ptr(O), _ptr(LSE),
                          int(threads), C.byref(used))
    _check(rc, "attn")
    if return_threads:
        return O, LSE, used.value
    return O, LSE


def attn_workload(w, **kw):
    """attn() on a workloads.Workload."""
    return attn(w.q, w.k_cache, w.v_cache, w.block_table, w.prefix_lens, w.parent, w.Hq, w.Hkv, **kw)


def lse_merge(O_parts, lse_parts):
    O_parts = _c(O_parts, np.float64)
    lse_parts = _c(lse_parts, np.float64)
    U = O_parts.shape[0]
    D = O_parts.shape[-1]
    rows = lse_parts[0].size
    O = np.zeros(O_parts.shape[1:], dtype=np.float64)
    lse = np.zeros(lse_parts.shape[1:], dtype=np.float64)
    _check(_load().tvo_lse_merge(U, rows, D, _ptr(O_parts), _ptr(lse_parts), _ptr(O), _ptr(lse)), "lse_merge")
    return O, lse


def argmax(logits):
    logits = _c(logits, np.uint16)
    rows, V = logits.shape
    am = np.zeros(rows, dtype=np.int32)
    _check(_load().tvo_argmax(_ptr(logits), rows, V, _ptr(am)), "argmax")
    return am


def accept(logits, draft, parent):
    parent = _c(parent, np.int32)
    if parent.ndim == 1:
        parent = parent[None]
    nb, B = parent.shape
    draft = _c(draft, np.int32).reshape(nb, B)
    logits = _c(logits, np.uint16).reshape(nb * B, -1)
    V = logits.shape[1]
    am = np.zeros(nb * B, dtype=np.int32)
    n_acc = np.zeros(nb, dtype=np.int32)
    path = np.zeros((nb, B), dtype=np.int32)
    bonus = np.zeros(nb, dtype=np.int32)
    _check(_load().tvo_accept(_ptr(logits), V, _ptr(draft), _ptr(parent), B, nb, _ptr(am), _ptr(n_acc),
                              _ptr(path), _ptr(bonus)), "accept")
    return am, n_acc, path, bonus


def kv_commit(k_cache, v_cache, block_table, prefix_lens, n_acc, path):
    """Commit of the accepted branch on copies of the caches; returns (k, v, new prefix_lens)."""
    k = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    v = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    block_table = _c(block_table, np.int32)
    prefix_lens = _c(prefix_lens, np.int32).reshape(-1)
    n_acc = _c(n_acc, np.int32).reshape(-1)
    path = _c(path, np.int32)
    nb, B = path.shape
    num_blocks, Hkv, page, D = k.shape
    new_pl = np.zeros(nb, dtype=np.int32)
    _check(_load().tvo_kv_commit(_ptr(k), _ptr(v), _ptr(block_table), _ptr(prefix_lens), _ptr(n_acc), _ptr(path),
                                 nb, B, Hkv, D, page, block_table.shape[1], num_blocks, _ptr(new_pl)), "kv_commit")
    return k, v, new_pl


def build_tree(logp, tokens, B, w=1):
    """Best-first tree (top-w rounds) from per-depth candidates logp/tokens [nb][Dmax][K].
    Returns parent, token int32 [nb][B] and score float32 [nb][B]; node 0 is the root."""
    logp = _c(logp, np.float32)
    tokens = _c(tokens, np.int32)
    nb, Dmax, K = logp.shape
    parent = np.zeros((nb, B), np.int32)
    token = np.zeros((nb, B), np.int32)
    score = np.zeros((nb, B), np.float32)
    _check(_load().tvo_build_tree(_ptr(logp), _ptr(tokens), nb, Dmax, K, B, w, _ptr(parent), _ptr(token),
                                  _ptr(score)), "build_tree")
    return parent, token, score


def gdn_tree(q, k, v, alpha, beta, S0, parent):
    """Gated DeltaNet outputs of every tree node (fp64), each from its own root path's state."""
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    alpha, beta, S0 = _c(alpha, np.float32), _c(beta, np.float32), _c(S0, np.float32)
    parent = _c(parent, np.int32)
    nb, B = parent.shape
    H, D = q.shape[1], q.shape[2]
    assert q.shape == (nb * B, H, D) and S0.shape == (nb, H, D, D) and alpha.shape == (nb * B, H)
    O = np.zeros((nb * B, H, D), np.float64)
    _check(_load().tvo_gdn_tree(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(parent),
                                nb, B, H, D, _ptr(O)), "gdn_tree")
    return O


def gdn_commit(k, v, alpha, beta, S0, n_acc, path):
    """New committed Gated DeltaNet state (fp64 [nb][H][D][D]): the recurrence applied from S0
    along path[b][0 .. n_acc[b]] (the accepted root path, root first)."""
    k, v = _c(k, np.uint16), _c(v, np.uint16)
    alpha, beta, S0 = _c(alpha, np.float32), _c(beta, np.float32), _c(S0, np.float32)
    n_acc = _c(n_acc, np.int32).reshape(-1)
    path = _c(path, np.int32)
    nb, B = path.shape
    H, D = k.shape[1], k.shape[2]
    assert k.shape == (nb * B, H, D) and S0.shape == (nb, H, D, D) and alpha.shape == (nb * B, H)
    S = np.zeros((nb, H, D, D), np.float64)
    _check(_load().tvo_gdn_commit(_ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0), _ptr(n_acc), _ptr(path),
                                  nb, B, H, D, _ptr(S)), "gdn_commit")
    return S
