"""GPU parity of tv_gdn_tree (Gated DeltaNet tree verification) against the fp64 oracle.

Every output element is compared.  Tolerance: the device works in fp32 (bf16 q/k/v
read exactly).  Each output element is gamma_i (S0^T q_i)_c plus one term per node
on i's root path, and each of those is a length-128 fp32 dot product (or a product
of them) whose rounding error is at most 128 * 2^-24 times the sum of the absolute
products, which these inputs bound by 4 (unit q and k, |S0| entries under 0.6, |v|
and |u| under 3).  A node at depth d therefore stays within
tol(d) = (d + 2) * 128 * 2^-24 * 4 of the exact value (5.5e-4 at depth 16), which
the tests apply node by node.  A dropped ancestor term moves an output by about
beta |k_i.k_j| |u_j| ~ 0.02, a wrong gate power by ~0.1 |S0^T q| ~ 0.005.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl
from tests.helpers import bf16_dev, i32_dev

pytestmark = pytest.mark.gpu

TOL16 = 18 * 128 * 2.0 ** -24 * 4


def _tol(parent):
    """Per-node tolerance [nb*B][1][1] from each node's depth."""
    nb, B = parent.shape
    dep = np.zeros((nb, B))
    for b in range(nb):
        for i in range(1, B):
            dep[b, i] = dep[b, parent[b, i]] + 1
    return ((dep + 2) * 128 * 2.0 ** -24 * 4).reshape(nb * B, 1, 1)


def _assert_close(got, ref, parent):
    err = np.abs(got - ref) - _tol(parent)
    assert np.isfinite(got).all()
    assert err.max() <= 0, f"error over tolerance by {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"


def _dev(w):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dict(q=bf16_dev(w.q), k=bf16_dev(w.k), v=bf16_dev(w.v), alpha=f(w.alpha), beta=f(w.beta), S0=f(w.S0),
                parent=i32_dev(w.parent))


def _run(w, status=None):
    d = _dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status is None else status
    O = tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], status=st)
    torch.cuda.synchronize()
    return O, int(st.item())


def _chain(B):
    return np.arange(-1, B - 1, dtype=np.int32)


def _star(B):
    p = np.zeros(B, np.int32)
    p[0] = -1
    return p


def _random_tree(B):
    def gen(r):
        p = np.empty(B, np.int32)
        p[0] = -1
        for i in range(1, B):
            p[i] = r.integers(max(0, i - 8), i)  # a recent node: deep and bushy
        return p
    return gen


CASES = {
    "single node": (1, 1, 3, lambda r: np.array([-1], np.int32)),
    "chain of 33 (ragged row tile)": (2, 33, 2, lambda r: _chain(33)),
    "star of 64": (1, 64, 2, lambda r: _star(64)),
    "best-first 48, 3 sequences": (3, 48, 4, lambda r: wl.tree_best_first(r, 48, child_cap=4, max_depth=16)),
    "random 200": (1, 200, 2, _random_tree(200)),
    "best-first 256 (largest tree)": (1, 256, 2, lambda r: wl.tree_best_first(r, 256, child_cap=4, max_depth=16)),
    "chain of 256": (1, 256, 1, lambda r: _chain(256)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_gdn_tree_matches_oracle(case):
    nb, B, H, trees = CASES[case]
    w = wl.make_gdn_workload(case, nb, B, H, 128, trees, seed=zlib.crc32(case.encode()))
    O, st = _run(w)
    assert st == 0
    ref = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    _assert_close(O.cpu().numpy().astype(np.float64), ref, w.parent)


def test_gdn_tree_full_size():
    """The benchmarked workload (1 sequence, 128-node best-first tree, 32 heads of 128), every element."""
    w = wl.gdn_config(seed=4321)
    O, st = _run(w)
    assert st == 0
    ref = oracle.gdn_tree(w.q, w.k, w.v, w.alpha, w.beta, w.S0, w.parent)
    _assert_close(O.cpu().numpy().astype(np.float64), ref, w.parent)


def test_gdn_tree_sibling_relabelling_permutes_outputs():
    """At any size: relabelling nodes by another topological order permutes the outputs
    (each node's output depends only on its own root path)."""
    w = wl.make_gdn_workload("relabel", 1, 96, 8, 128,
                             lambda r: wl.tree_best_first(r, 96, child_cap=4, max_depth=16), seed=77)
    rng = np.random.default_rng(5)
    par = w.parent[0]
    # a random topological order: repeatedly take a random node whose parent is already placed
    placed, order = {-1}, []
    avail = [0]
    children = {i: [j for j in range(w.B) if par[j] == i] for i in range(w.B)}
    while avail:
        x = avail.pop(int(rng.integers(len(avail))))
        order.append(x)
        placed.add(x)
        avail += children[x]
    old_of_new = np.array(order)
    new_of_old = np.argsort(old_of_new)
    new_parent = np.array([-1 if par[o] < 0 else new_of_old[par[o]] for o in old_of_new], np.int32)
    w2 = wl.GdnWorkload(name="relabelled", nb=1, B=w.B, H=w.H, D=w.D, q=w.q[old_of_new], k=w.k[old_of_new],
                        v=w.v[old_of_new], alpha=w.alpha[old_of_new], beta=w.beta[old_of_new], S0=w.S0,
                        parent=new_parent[None])
    O1, s1 = _run(w)
    O2, s2 = _run(w2)
    assert s1 == 0 and s2 == 0
    d = (O2.cpu() - O1.cpu()[torch.from_numpy(old_of_new)]).abs().max().item()
    assert d <= 2 * TOL16  # best-first trees here are at most 16 deep


def test_gdn_tree_rejects_non_topological_parent():
    w = wl.make_gdn_workload("bad", 2, 16, 2, 128, lambda r: _chain(16), seed=3)
    w.parent[1, 5] = 9  # a later node as parent
    O, st = _run(w)
    assert st == 2  # TV_ERR_NOT_TOPOLOGICAL


def test_gdn_tree_empty_batch_is_a_no_op():
    z = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    a = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    S0 = torch.empty((0, 4, 128, 128), dtype=torch.float32, device="cuda")
    parent = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    O = tv.gdn_tree(z, z, z, a, a, S0, parent)
    torch.cuda.synchronize()
    assert O.shape == (0, 4, 128)


def test_gdn_tree_in_a_cuda_graph():
    """The two launches capture and replay in a CUDA graph; the replay matches the eager call."""
    w = wl.gdn_config(seed=11)
    d = _dev(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    O = torch.empty((w.nb * w.B, w.H, w.D), dtype=torch.float32, device="cuda")
    ws = torch.empty(tv.lib().tv_gdn_tree_workspace_size(w.nb, w.B, w.H, w.D), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], out=O, workspace=ws,
                    status=st, stream=s)
    torch.cuda.synchronize()
    eager = O.clone()
    O.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tv.gdn_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], d["parent"], out=O, workspace=ws,
                    status=st, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(O, eager)
