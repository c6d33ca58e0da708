"""Thin ctypes binding over libtreeverify's C ABI (include/treeverify.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (device memory and streams come from torch);
the functions keep the C names: build_mask, attn, accept.  There is no CPU
path: if the library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreeverify.so")

TV_OK = 0
TV_ERR_INVALID_ARG = 1
TV_ERR_NOT_TOPOLOGICAL = 2
TV_ERR_UNSUPPORTED_SHAPE = 3
TV_ERR_CUDA = 4
TV_ERR_TIMEOUT = 5
TV_ERR_UNIMPLEMENTED = 6

EXPORTED = ("tv_status_str", "tv_version", "tv_build_mask", "tv_attn_workspace_size", "tv_attn", "tv_attn_launches",
            "tv_accept_workspace_size", "tv_accept", "tv_accept_fused_workspace_size", "tv_accept_fused",
            "tv_accept_noalloc", "tv_kv_commit", "tv_build_tree", "tv_gdn_tree_workspace_size", "tv_gdn_tree", "tv_gdn_commit",
            "tv_selftest_wait")
NOALLOC_MAX_ROWS = 8192  # TV_ACCEPT_NOALLOC_MAX_ROWS


class TVError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_str(code)} ({code})")


class AttnArgs(C.Structure):
    """Mirror of tv_attn_args."""
    _fields_ = [
        ("q_d", C.c_void_p), ("k_cache_d", C.c_void_p), ("v_cache_d", C.c_void_p),
        ("block_table_d", C.c_void_p), ("prefix_lens_d", C.c_void_p), ("mask_d", C.c_void_p),
        ("o_d", C.c_void_p), ("lse_d", C.c_void_p), ("dev_status_d", C.c_void_p),
        ("nb", C.c_int32), ("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("D", C.c_int32),
        ("page_size", C.c_int32), ("num_blocks", C.c_int32), ("max_pages", C.c_int32),
        ("scale", C.c_float), ("num_ctas", C.c_int32), ("parent_d", C.c_void_p),
    ]


_lib = None


def lib() -> C.CDLL:
    """Load libtreeverify.so (built by build.build()); raises if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtreeverify.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        P, I = C.c_void_p, C.c_int32
        L.tv_status_str.argtypes = [I]
        L.tv_status_str.restype = C.c_char_p
        L.tv_version.argtypes = []
        L.tv_version.restype = I
        L.tv_build_mask.argtypes = [P, I, I, P, P, P, P]
        L.tv_build_mask.restype = I
        L.tv_attn_workspace_size.argtypes = [C.POINTER(AttnArgs)]
        L.tv_attn_workspace_size.restype = C.c_size_t
        L.tv_attn_launches.argtypes = [C.POINTER(AttnArgs)]
        L.tv_attn_launches.restype = C.c_int32
        L.tv_attn.argtypes = [C.POINTER(AttnArgs), P, C.c_size_t, P]
        L.tv_attn.restype = I
        L.tv_accept_workspace_size.argtypes = [I, I, I]
        L.tv_accept_workspace_size.restype = C.c_size_t
        L.tv_accept.argtypes = [P, I, P, P, P, I, I, P, P, P, P, P, P, C.c_size_t, P]
        L.tv_accept.restype = I
        L.tv_accept_fused_workspace_size.argtypes = [I, I, I]
        L.tv_accept_fused_workspace_size.restype = C.c_size_t
        L.tv_accept_fused.argtypes = [P, I, P, P, P, I, I, P, P, P, P, P, P, C.c_size_t, P]
        L.tv_accept_fused.restype = I
        L.tv_accept_noalloc.argtypes = [P, I, P, P, P, I, I, P, P, P, P, P, P]
        L.tv_accept_noalloc.restype = I
        L.tv_kv_commit.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P]
        L.tv_kv_commit.restype = I
        L.tv_build_tree.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
        L.tv_build_tree.restype = I
        L.tv_gdn_tree_workspace_size.argtypes = [I, I, I, I]
        L.tv_gdn_tree_workspace_size.restype = C.c_size_t
        L.tv_gdn_tree.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, P, C.c_size_t, P, P]
        L.tv_gdn_tree.restype = I
        L.tv_gdn_commit.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P, P, P]
        L.tv_gdn_commit.restype = I
        L.tv_selftest_wait.argtypes = [C.c_uint32, P, P]
        L.tv_selftest_wait.restype = I
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().tv_status_str(int(code)).decode()


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != TV_OK:
        raise TVError(rc, what)


def build_mask(parent: torch.Tensor, status: torch.Tensor | None = None, mask: torch.Tensor | None = None,
               depth: torch.Tensor | None = None, stream=None):
    """tv_build_mask: parent int32 [nb][B] (cuda) -> (mask uint32-as-int32 [nb][B][W], depth int32 [nb][B])."""
    nb, B = parent.shape
    W = (B + 31) // 32
    if mask is None:
        mask = torch.empty((nb, B, W), dtype=torch.int32, device=parent.device)
    if depth is None:
        depth = torch.empty((nb, B), dtype=torch.int32, device=parent.device)
    rc = lib().tv_build_mask(_p(parent), B, nb, _p(mask), _p(depth), _p(status), _stream(stream))
    _check(rc, "tv_build_mask")
    return mask, depth


def attn_args(q, k_cache, v_cache, block_table, prefix_lens, mask, o, lse, status=None, scale: float = 0.0,
              num_ctas: int = 0, parent=None) -> AttnArgs:
    """mask may be None when parent is given (the attention derives the ancestor bits itself)."""
    nbB, Hq, D = q.shape
    num_blocks, Hkv, page, _ = k_cache.shape
    nb = prefix_lens.shape[0]
    B = nbB // nb if nb else 0
    return AttnArgs(q_d=q.data_ptr(), k_cache_d=k_cache.data_ptr(), v_cache_d=v_cache.data_ptr(),
                    block_table_d=block_table.data_ptr(), prefix_lens_d=prefix_lens.data_ptr(),
                    mask_d=(mask.data_ptr() if mask is not None else None), o_d=o.data_ptr(), lse_d=lse.data_ptr(),
                    dev_status_d=(status.data_ptr() if status is not None else None),
                    nb=nb, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=page, num_blocks=num_blocks,
                    max_pages=block_table.shape[1], scale=float(scale), num_ctas=int(num_ctas),
                    parent_d=(parent.data_ptr() if parent is not None else None))


def attn_workspace_size(args: AttnArgs) -> int:
    return int(lib().tv_attn_workspace_size(C.byref(args)))


def attn_launches(args: AttnArgs) -> int:
    """Kernel launches tv_attn enqueues for these arguments (1, or 2 with the merge kernel)."""
    return int(lib().tv_attn_launches(C.byref(args)))


def attn(q, k_cache, v_cache, block_table, prefix_lens, mask, status=None, scale: float = 0.0, num_ctas: int = 0,
         o=None, lse=None, workspace=None, stream=None, parent=None):
    """tv_attn: returns (O bf16 [nb*B][Hq][D], LSE fp32 [nb*B][Hq]); mask=None with parent
    given folds the mask build into the attention.  A workspace passed in must have been
    zeroed once before its first use (every call leaves its counters zero); without one,
    a zeroed workspace is allocated for this call."""
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    a = attn_args(q, k_cache, v_cache, block_table, prefix_lens, mask, o, lse, status, scale, num_ctas, parent)
    need = attn_workspace_size(a)
    if need == 0:  # invalid arguments: let the library say which
        _check(lib().tv_attn(C.byref(a), None, 0, _stream(stream)), "tv_attn")
        return o, lse
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    rc = lib().tv_attn(C.byref(a), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "tv_attn")
    return o, lse


def _logits_ok(logits, parent):
    """The device every output and workspace lives on: the tree arrays'.  The logits may be
    on that device or in pinned host memory (the kernel then reads them over the host link);
    pageable host memory is refused."""
    if not parent.is_cuda:
        raise ValueError("parent (and draft) must be device tensors")
    if not logits.is_cuda and not logits.is_pinned():
        raise ValueError("logits must be a device tensor or pinned host memory")
    return parent.device


def accept_workspace_size(V: int, B: int, nb: int) -> int:
    return int(lib().tv_accept_workspace_size(int(V), int(B), int(nb)))


def accept(logits, draft, parent, mask, status=None, out=None, workspace=None, stream=None):
    """tv_accept: returns (argmax [nb*B], n_acc [nb], path [nb][B], bonus [nb]) int32 tensors.

    A workspace passed in must have been zeroed once before its first use (every call
    leaves it zeroed); without one, a zeroed workspace is allocated for this call.
    """
    nb, B = parent.shape
    V = logits.shape[-1]
    dev = _logits_ok(logits, parent)
    if out is None:
        out = (torch.empty(nb * B, dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev),
               torch.empty((nb, B), dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev))
    am, n_acc, path, bonus = out
    need = accept_workspace_size(V, B, nb)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.zeros(max(need, 8), dtype=torch.uint8, device=dev)
    rc = lib().tv_accept(_p(logits), V, _p(draft), _p(parent), _p(mask), B, nb, _p(am), _p(n_acc), _p(path),
                         _p(bonus), _p(status), _p(workspace), workspace.numel() * workspace.element_size(),
                         _stream(stream))
    _check(rc, "tv_accept")
    return am, n_acc, path, bonus


def accept_fused_workspace_size(V: int, B: int, nb: int) -> int:
    return int(lib().tv_accept_fused_workspace_size(int(V), int(B), int(nb)))


def accept_fused(logits, draft, parent, mask=None, status=None, out=None, workspace=None, stream=None):
    """tv_accept_fused: tv_accept's results from one kernel; mask may be None (built from parent).

    A workspace passed in must have had its counters zeroed once (the library keeps
    them zero); without one, a zeroed workspace is allocated for this call.
    """
    nb, B = parent.shape
    V = logits.shape[-1]
    dev = _logits_ok(logits, parent)
    if out is None:
        out = (torch.empty(nb * B, dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev),
               torch.empty((nb, B), dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev))
    am, n_acc, path, bonus = out
    need = accept_fused_workspace_size(V, B, nb)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.zeros(max(need, 8), dtype=torch.uint8, device=dev)
    rc = lib().tv_accept_fused(_p(logits), V, _p(draft), _p(parent), _p(mask), B, nb, _p(am), _p(n_acc), _p(path),
                               _p(bonus), _p(status), _p(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "tv_accept_fused")
    return am, n_acc, path, bonus


def accept_noalloc(logits, draft, parent, mask, status=None, out=None, stream=None):
    """tv_accept_noalloc: tv_accept on the library's own fixed scratch (no workspace).

    For callers that cannot allocate device memory (stream capture, runtimes
    with a fixed memory plan); at most NOALLOC_MAX_ROWS logits rows per call,
    and calls must not overlap on the GPU (they share the scratch).
    """
    nb, B = parent.shape
    V = logits.shape[-1]
    dev = _logits_ok(logits, parent)
    if out is None:
        out = (torch.empty(nb * B, dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev),
               torch.empty((nb, B), dtype=torch.int32, device=dev), torch.empty(nb, dtype=torch.int32, device=dev))
    am, n_acc, path, bonus = out
    rc = lib().tv_accept_noalloc(_p(logits), V, _p(draft), _p(parent), _p(mask), B, nb, _p(am), _p(n_acc), _p(path),
                                 _p(bonus), _p(status), _stream(stream))
    _check(rc, "tv_accept_noalloc")
    return am, n_acc, path, bonus


def kv_commit(k_cache, v_cache, block_table, prefix_lens, n_acc, path, new_prefix_lens=None, status=None,
              stream=None):
    """tv_kv_commit: moves the accepted path's K/V into place (caches updated in place);
    returns new_prefix_lens int32 [nb]."""
    num_blocks, Hkv, page, D = k_cache.shape
    nb, B = path.shape
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty(nb, dtype=torch.int32, device=k_cache.device)
    rc = lib().tv_kv_commit(_p(k_cache), _p(v_cache), _p(block_table), _p(prefix_lens), _p(n_acc), _p(path), nb, B,
                            Hkv, D, page, num_blocks, block_table.shape[1], _p(new_prefix_lens), _p(status),
                            _stream(stream))
    _check(rc, "tv_kv_commit")
    return new_prefix_lens


def build_tree(logp, tokens, B, w=1, out=None, status=None, stream=None):
    """tv_build_tree: logp fp32 / tokens int32 [nb][Dmax][K] (cuda) -> (parent, token int32 [nb][B],
    score fp32 [nb][B])."""
    nb, Dmax, K = logp.shape
    dev = logp.device
    if out is None:
        out = (torch.empty((nb, B), dtype=torch.int32, device=dev), torch.empty((nb, B), dtype=torch.int32, device=dev),
               torch.empty((nb, B), dtype=torch.float32, device=dev))
    parent, token, score = out
    rc = lib().tv_build_tree(_p(logp), _p(tokens), nb, Dmax, K, B, w, _p(parent), _p(token), _p(score), _p(status),
                             _stream(stream))
    _check(rc, "tv_build_tree")
    return parent, token, score


def gdn_tree(q, k, v, alpha, beta, S0, parent, out=None, workspace=None, status=None, stream=None):
    """tv_gdn_tree: q/k/v bf16 [nb*B][H][D], alpha/beta fp32 [nb*B][H], S0 fp32 [nb][H][D][D],
    parent int32 [nb][B] (cuda) -> O fp32 [nb*B][H][D]."""
    nb, B = parent.shape
    H, D = q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((nb * B, H, D), dtype=torch.float32, device=q.device)
    need = int(lib().tv_gdn_tree_workspace_size(nb, B, H, D))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    rc = lib().tv_gdn_tree(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(S0), _p(parent), nb, B, H, D, _p(out),
                           _p(workspace), workspace.numel() * workspace.element_size(), _p(status), _stream(stream))
    _check(rc, "tv_gdn_tree")
    return out


def gdn_commit(k, v, alpha, beta, S0, n_acc, path, out=None, status=None, stream=None):
    """tv_gdn_commit: the new committed state (fp32 [nb][H][D][D]) after the accepted path;
    out may be S0 itself (committed in place)."""
    nb, B = path.shape
    H, D = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty_like(S0)
    rc = lib().tv_gdn_commit(_p(k), _p(v), _p(alpha), _p(beta), _p(S0), _p(n_acc), _p(path), nb, B, H, D, _p(out),
                             _p(status), _stream(stream))
    _check(rc, "tv_gdn_commit")
    return out


def selftest_wait(limit_us: int, status: torch.Tensor, stream=None):
    """tv_selftest_wait: a kernel whose bounded wait runs out; status gets TV_ERR_TIMEOUT."""
    _check(lib().tv_selftest_wait(int(limit_us), _p(status), _stream(stream)), "tv_selftest_wait")
