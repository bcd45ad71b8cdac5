"""Moving seeded workloads onto the GPU and comparing with the oracle (GPU tests only)."""

from __future__ import annotations

import numpy as np

BF16_OUT_TOL = 2e-2   # max |out - oracle| for a bf16 cache
FP8_OUT_TOL = 5e-2    # max |out - oracle| for an e4m3 cache
LSE_TOL = 1e-3        # max |lse - oracle|


def to_dev(a, dev):
    import torch

    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def kv_of(w, dev):
    import sparse_mla_attention_top_gb300 as S

    return S.KVCache(to_dev(w.kv, dev), w.num_pages, w.page_size, w.kv_dtype)


def out_tol(w) -> float:
    return FP8_OUT_TOL if w.kv_dtype == 1 else BF16_OUT_TOL


def compare(out, lse, ref, ref_lse, tol_out, tol_lse=LSE_TOL, rows=None):
    """Max errors of GPU (out bf16 tensor [T,H,512], lse [T,H]) against oracle fp64 arrays;
    `rows` picks the GPU rows that the oracle computed (sampled checks)."""
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    d_out = float(np.max(np.abs(o - ref))) if o.size else 0.0
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse)), "empty rows differ"
    d_lse = float(np.max(np.abs(np.where(both_inf, 0.0, l - ref_lse)))) if l.size else 0.0
    assert d_out <= tol_out and d_lse <= tol_lse, f"max|out| err {d_out:.3e} (tol {tol_out}), " \
                                                  f"max|lse| err {d_lse:.3e} (tol {tol_lse})"
    return d_out, d_lse
