"""Seeded generators for K, V, L1 membership, sign vectors and queries.

Every array comes from its own numpy ``SeedSequence`` keyed on
(seed, workload tag, layer, purpose, batch index, head), so any (b, h) slice
can be regenerated on its own and both consumers see identical numbers.

Recipes (stated readings of the workload text):
  * keys, "lognormal": z ~ N(0, 1)^d per token, RMS-normalised, then scaled
    per channel by exp(0.5 * n_c), n_c ~ N(0, 1) drawn once per (layer, head).
  * keys, "student_t": z ~ Student-t(nu=3) per coordinate, 4 seeded channels
    multiplied by 20, then RMS-normalised.
  * keys, "lowrank": A z + 0.1 eps with A in R^{d x 16}, A_ij ~ N(0, 1/16)
    per (layer, head), z ~ N(0, I_16), eps ~ N(0, I_d), then RMS-normalised.
  * values: N(0, 1).
  * storage "bf16": round-to-nearest-even to bfloat16 (values stay float32
    arrays holding exactly representable numbers).
  * L1: sinks [0, sinks) + recent [T - recent, T) + `marked` positions drawn
    without replacement from [sinks, T - recent), per (layer, b).
  * signs: one +-1 vector of length d per layer (shared by K, V, all tiers
    and heads).
  * sketch matrix (TQ-QKV): one [128, d] float32 N(0, 1) matrix per layer.
  * queries: float32 N(0, 1) at position T + s for step s.  With a needle,
    q_s = sqrt(0.8) q_0 + sqrt(0.2) z_s for s >= 1, so the needle stays
    near alignment while the selection still moves from step to step.
  * needle: per (b, h) one seeded group strictly inside [sinks, T - recent)
    whose every token's post-RoPE key is |k_t| (0.9 u + sqrt(0.19) w_t),
    u = normalise(sum of the head's post-RoPE step-0 queries), w_t a random
    unit vector orthogonal to u; the token is stored pre-RoPE.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple, Callable, Optional, Sequence

import numpy as np

from .configs import Workload

_PURPOSE = {
    "keys": 1,
    "values": 2,
    "l1": 3,
    "signs": 4,
    "queries": 5,
    "needle_group": 6,
    "needle_dirs": 7,
    "key_scale": 8,
    "outlier_channels": 9,
    "lowrank_A": 10,
    "qjl_sketch": 11,
}


def _rng(w: Workload, seed: int, layer: int, purpose: str, *extra: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), int(w.seed_tag), int(layer), _PURPOSE[purpose],
                                 *[int(e) for e in extra]])
    return np.random.Generator(np.random.PCG64(ss))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(x.shape)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Bit patterns (uint16) of float32 values that are exact bfloat16 numbers."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not exactly representable in bfloat16")
    return (u >> 16).astype(np.uint16).reshape(x.shape)


def _storage(w: Workload, x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    return round_to_bf16(x) if w.storage == "bf16" else x


def _rms_normalise(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))


def _raw_keys(w: Workload, seed: int, layer: int, b: int, h: int) -> np.ndarray:
    T, d = w.T, w.d
    g = _rng(w, seed, layer, "keys", b, h)
    if w.key_law == "lognormal":
        gamma = np.exp(0.5 * _rng(w, seed, layer, "key_scale", h).standard_normal(d))
        z = g.standard_normal((T, d))
        return gamma * _rms_normalise(z)
    if w.key_law == "student_t":
        ch = _rng(w, seed, layer, "outlier_channels", h).choice(d, size=4, replace=False)
        z = g.standard_t(3.0, size=(T, d))
        z[:, ch] *= 20.0
        return _rms_normalise(z)
    if w.key_law == "lowrank":
        A = _rng(w, seed, layer, "lowrank_A", h).standard_normal((d, 16)) * 0.25
        z = g.standard_normal((T, 16))
        eps = g.standard_normal((T, d))
        return _rms_normalise(z @ A.T + 0.1 * eps)
    raise ValueError(f"unknown key law {w.key_law!r}")


def _l1_mask(w: Workload, seed: int, layer: int, b: int) -> np.ndarray:
    T = w.T
    m = np.zeros(T, dtype=bool)
    m[: min(w.sinks, T)] = True
    if w.recent > 0:
        m[max(T - w.recent, 0):] = True
    lo, hi = w.sinks, T - w.recent
    if w.marked > 0:
        if hi - lo < w.marked:
            raise ValueError("not enough positions for the marked tokens")
        pick = _rng(w, seed, layer, "l1", b).choice(hi - lo, size=w.marked, replace=False)
        m[lo + pick] = True
    return m


def _signs(w: Workload, seed: int, layer: int) -> np.ndarray:
    bits = _rng(w, seed, layer, "signs").integers(0, 2, size=w.d)
    return np.where(bits == 1, 1, -1).astype(np.int8)


def qjl_matrix(w: Workload, layer: int = 0, seed: int = 0, m: int = 128) -> np.ndarray:
    """The [m, d] float32 sketch matrix of a layer, i.i.d. N(0, 1)."""
    return _rng(w, seed, layer, "qjl_sketch").standard_normal((m, w.d)).astype(np.float32)


def layer_meta(w: Workload, layer: int = 0, seed: int = 0,
               batch: Optional[Sequence[int]] = None) -> Tuple[np.ndarray, np.ndarray]:
    """L1 membership [nb, T] and sign vector [d] of one layer, without its K/V."""
    bs = list(range(w.B)) if batch is None else list(batch)
    return np.stack([_l1_mask(w, seed, layer, b) for b in bs]), _signs(w, seed, layer)


def queries(w: Workload, layer: int = 0, steps: Optional[int] = None, seed: int = 0,
            batch: Optional[Sequence[int]] = None):
    """Queries q [steps, nb, Hq, d] float32 and positions pos [steps, nb] int32."""
    steps = w.steps if steps is None else steps
    bs = list(range(w.B)) if batch is None else list(batch)
    q = np.empty((steps, len(bs), w.Hq, w.d), dtype=np.float32)
    for i, b in enumerate(bs):
        g = _rng(w, seed, layer, "queries", b)
        q0 = g.standard_normal((w.Hq, w.d))
        for s in range(steps):
            if s == 0:
                qs = q0
            elif w.needle:
                qs = np.sqrt(0.8) * q0 + np.sqrt(0.2) * g.standard_normal((w.Hq, w.d))
            else:
                qs = g.standard_normal((w.Hq, w.d))
            q[s, i] = qs
    pos = np.broadcast_to((w.T + np.arange(steps, dtype=np.int32))[:, None],
                          (steps, len(bs))).astype(np.int32)
    return q, pos


def needle_groups(w: Workload, l1_mask: np.ndarray, layer: int = 0, seed: int = 0,
                  batch: Optional[Sequence[int]] = None) -> np.ndarray:
    """One seeded group per (b, h), strictly inside [sinks, T - recent), with at
    least one member outside L1."""
    bs = list(range(w.B)) if batch is None else list(batch)
    gmin = -(-w.sinks // w.N)
    gmax = (w.T - w.recent) // w.N  # exclusive
    out = np.empty((len(bs), w.Hkv), dtype=np.int64)
    for i, b in enumerate(bs):
        g = _rng(w, seed, layer, "needle_group", b)
        for h in range(w.Hkv):
            while True:
                cand = int(g.integers(gmin, gmax))
                if not np.all(l1_mask[i, cand * w.N:(cand + 1) * w.N]):
                    break
            out[i, h] = cand
    return out


RopeFn = Callable[[np.ndarray, np.ndarray], np.ndarray]


def plant_needle(w: Workload, K: np.ndarray, groups: np.ndarray, q0: np.ndarray,
                 pos0: np.ndarray, rope: RopeFn, layer: int = 0, seed: int = 0,
                 batch: Optional[Sequence[int]] = None) -> None:
    """Overwrite the needle groups' keys in K (float64, pre-RoPE) in place.

    `rope(x, p)` must apply the rotary embedding at positions p (broadcast
    over the leading axes of x); the caller supplies it.
    """
    bs = list(range(w.B)) if batch is None else list(batch)
    r = w.r
    for i, b in enumerate(bs):
        gdir = _rng(w, seed, layer, "needle_dirs", b)
        for h in range(w.Hkv):
            qh = q0[i, h * r:(h + 1) * r].astype(np.float64)
            u = rope(qh, np.full(r, pos0[i], dtype=np.int64)).sum(axis=0)
            u /= np.linalg.norm(u)
            g0 = int(groups[i, h])
            t = np.arange(g0 * w.N, min((g0 + 1) * w.N, w.T))
            wt = gdir.standard_normal((len(t), w.d))
            wt -= (wt @ u)[:, None] * u[None, :]
            wt /= np.linalg.norm(wt, axis=1, keepdims=True)
            nk = np.linalg.norm(K[i, h, t], axis=1)
            post = nk[:, None] * (0.9 * u[None, :] + np.sqrt(0.19) * wt)
            K[i, h, t] = rope(post, -t)


@dataclass
class LayerInputs:
    K: np.ndarray            # [nb, Hkv, T, d] float32, pre-RoPE, storage-rounded
    V: np.ndarray            # [nb, Hkv, T, d] float32, storage-rounded
    l1_mask: np.ndarray      # [nb, T] bool
    signs: np.ndarray        # [d] int8, +-1
    needle_group: Optional[np.ndarray] = None  # [nb, Hkv]


def layer_inputs(w: Workload, layer: int = 0, seed: int = 0,
                 batch: Optional[Sequence[int]] = None,
                 rope: Optional[RopeFn] = None) -> LayerInputs:
    """K, V, L1 membership and signs for one layer (optionally a subset of sequences)."""
    bs = list(range(w.B)) if batch is None else list(batch)
    nb = len(bs)
    K = np.empty((nb, w.Hkv, w.T, w.d), dtype=np.float64 if w.needle else np.float32)
    V = np.empty((nb, w.Hkv, w.T, w.d), dtype=np.float32)
    mask = np.stack([_l1_mask(w, seed, layer, b) for b in bs])
    for i, b in enumerate(bs):
        for h in range(w.Hkv):
            K[i, h] = _raw_keys(w, seed, layer, b, h)
            V[i, h] = _storage(w, _rng(w, seed, layer, "values", b, h).standard_normal((w.T, w.d)))
    groups = None
    if w.needle:
        if rope is None:
            raise ValueError("a needle workload needs the rotary function to plant its keys")
        groups = needle_groups(w, mask, layer, seed, bs)
        q, pos = queries(w, layer, 1, seed, bs)
        plant_needle(w, K, groups, q[0], pos[0], rope, layer, seed, bs)
    K = _storage(w, K)
    return LayerInputs(K=K, V=V, l1_mask=mask, signs=_signs(w, seed, layer), needle_group=groups)
