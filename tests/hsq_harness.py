"""Shared helpers for the library tests: building, uploading a layer,
reading the cache back in the byte layout the oracle understands, and the
near-tie-aware comparisons the acceptance rules ask for."""

from __future__ import annotations

import os
from typing import Dict, Optional

import numpy as np

import oracle as O
import workloads as W


def ensure_built():
    from hierarchical_kv_cache_hsq_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()


def make_ctx(w: W.Workload, beta: Optional[int] = None, max_l1: Optional[int] = None, n_splits: int = 0,
             steps: Optional[int] = None, B: Optional[int] = None):
    import hierarchical_kv_cache_hsq_gb300 as H
    max_pos = w.T + (w.steps if steps is None else steps) + 1
    cfg = H.make_config(w.Hq, w.Hkv, w.N, beta or w.beta, B or w.B, w.T,
                        max(max_l1 if max_l1 is not None else w.l1_size, 1), max_pos, w.theta, n_splits)
    return H.Context(cfg)


def gpu_encode(ctx, w: W.Workload, li: W.LayerInputs, l3_on_host: bool = True):
    import torch
    import hierarchical_kv_cache_hsq_gb300 as H
    B = li.K.shape[0]
    cache = H.allocate_cache(ctx, B, w.T, l3_on_host=l3_on_host)
    H.set_layer_inputs(cache, li.l1_mask, li.signs)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    K = torch.from_numpy(np.ascontiguousarray(li.K, np.float32)).to("cuda").to(dt).contiguous()
    V = torch.from_numpy(np.ascontiguousarray(li.V, np.float32)).to("cuda").to(dt).contiguous()
    H.hsq_encode(ctx, cache, K, V)
    torch.cuda.synchronize()
    return cache


def abi_buffers(cache) -> Dict[str, np.ndarray]:
    """GPU cache buffers as numpy arrays in the oracle's ABI layout."""
    out = {}
    for name in ("l1_kc", "l1_vc", "l1_kn", "l1_vn", "l1_pos", "l1_count", "l2_kc", "l2_vc", "l2_kn",
                 "l2_vn", "l2_cnt", "l3"):
        out[name] = cache.view(name).cpu().numpy()
    return out


def slice_heads(bufs: Dict[str, np.ndarray], h0: int, h1: int) -> Dict[str, np.ndarray]:
    per_head = {"l1_kc", "l1_vc", "l1_kn", "l1_vn", "l2_kc", "l2_vc", "l2_kn", "l2_vn", "l3"}
    return {k: (v[:, h0:h1] if k in per_head else v) for k, v in bufs.items()}


def oracle_view(bufs, li: W.LayerInputs, w: W.Workload) -> O.OracleCache:
    return O.cache_from_abi(bufs, li.l1_mask, li.signs, w.N, w.T, w.theta)


def code_mismatch(gpu_codes: np.ndarray, ora_codes: np.ndarray, y: np.ndarray, bits: int,
                  norms: Optional[np.ndarray] = None):
    """(mismatches outside the near-tie band, near-tie coordinates that differ, near-tie count).

    Zero vectors (norm 0, e.g. empty groups) are encoded by definition, not
    by a boundary decision, so they never count as near-ties."""
    diff = gpu_codes != ora_codes
    tie = O.near_boundary(y, bits)
    if norms is not None:
        tie &= (np.asarray(norms) > 0)[..., None]
    return int(np.sum(diff & ~tie)), int(np.sum(diff & tie)), int(np.sum(tie))


def rel_l2(a: np.ndarray, b: np.ndarray, axis=-1) -> np.ndarray:
    num = np.linalg.norm(np.asarray(a, np.float64) - np.asarray(b, np.float64), axis=axis)
    den = np.maximum(np.linalg.norm(np.asarray(b, np.float64), axis=axis), 1e-30)
    return num / den


def selection_near_ties(scores_row: np.ndarray, beta: int, rel: float = 1e-5) -> np.ndarray:
    """Groups whose fp32 score lies within rel * max(|s_beta|, rms(s)) of the beta-th score."""
    s = scores_row[np.isfinite(scores_row)].astype(np.float64)
    if len(s) <= beta:
        return np.zeros(len(scores_row), bool)
    sb = np.sort(s)[::-1][beta - 1]
    tol = rel * max(abs(sb), float(np.sqrt(np.mean(s * s))))
    out = np.zeros(len(scores_row), bool)
    fin = np.isfinite(scores_row)
    out[fin] = np.abs(scores_row[fin].astype(np.float64) - sb) <= tol
    return out


def sel_mismatch(gpu_sel: np.ndarray, ora_sel: np.ndarray, scores_row: np.ndarray, beta: int):
    """Count selected-set differences that are not explained by near-ties of the beta-th score."""
    a = set(int(g) for g in gpu_sel if g >= 0)
    b = set(int(g) for g in ora_sel if g >= 0)
    ties = selection_near_ties(scores_row, beta)
    bad = [g for g in a ^ b if not ties[g]]
    return len(bad), len(a ^ b)
