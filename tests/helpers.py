"""Shared test helpers: move a workloads.Workload to the GPU and run the library on it."""
import numpy as np
import torch

import tree_speculative_decoding_tv_gb300 as tv
import workloads as wl


def bf16_dev(u16: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).to(dev).view(torch.bfloat16)


def i32_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return wl.bf16_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


class DevWorkload:
    def __init__(self, w: wl.Workload, dev="cuda"):
        self.w = w
        self.q = bf16_dev(w.q, dev)
        self.k = bf16_dev(w.k_cache, dev)
        self.v = bf16_dev(w.v_cache, dev)
        self.bt = i32_dev(w.block_table, dev)
        self.pl = i32_dev(w.prefix_lens, dev)
        self.parent = i32_dev(w.parent, dev)
        self.draft = i32_dev(w.draft, dev)
        self.logits = bf16_dev(w.logits, dev) if w.logits.size else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def mask(self):
        return tv.build_mask(self.parent, status=self.status)

    def attn(self, mask, num_ctas=0, scale=0.0):
        return tv.attn(self.q, self.k, self.v, self.bt, self.pl, mask, status=self.status, num_ctas=num_ctas,
                       scale=scale)

    def accept(self, mask):
        return tv.accept(self.logits, self.draft, self.parent, mask, status=self.status)


def assert_attn_close(O_gpu, L_gpu, O_ref, L_ref, w, rows=None, o_tol=2e-2, lse_tol=1e-3):
    """O within o_tol absolute (bf16 out vs fp64 oracle), LSE within lse_tol (natural log)."""
    O = bf16_host(O_gpu)
    L = L_gpu.cpu().numpy().astype(np.float64)
    if rows is not None:
        O, L = O[rows], L[rows]
    dO = np.abs(O - O_ref)
    dL = np.abs(L - L_ref)
    assert np.isfinite(O).all() and np.isfinite(L).all(), "non-finite output"
    assert dO.max() <= o_tol, f"max|dO|={dO.max():.3e} at {np.unravel_index(dO.argmax(), dO.shape)}"
    assert dL.max() <= lse_tol, f"max|dLSE|={dL.max():.3e} at {np.unravel_index(dL.argmax(), dL.shape)}"
    return float(dO.max()), float(dL.max())
