"""HSQ (Hierarchical Semantic Quantization, "Tamarin") oracle in plain float64 numpy.

TEST INFRASTRUCTURE ONLY -- see the package docstring.  Slow and direct on
purpose: every step is the definition written out, in the order the pages
give it, with library primitives (matmul, sort, betainc) as the only help.

Sources (page title, then section):
  [HSQ]  "Tamarin (HSQ) - reversible hierarchical KV-cache compression",
         technical summary (gist.science rs-10297225, Korean and Dutch pages):
         section 2 "Method" -- three-tier architecture (L1 focal, L2 summary,
         L3 archive), decode process (1 routing, 2 fetching, 3 attention),
         key components (TurboQuant quantisation).
  [TQ]   "Ablation, Statistical Inference, and Validation for KV-Cache
         Compression", technical summary (gist.science 2607.09683):
         experimental setup, item 1 (TurboQuant = randomised Walsh-Hadamard
         transform followed by a data-oblivious Beta Lloyd-Max codebook).

Readings where the pages are silent (each also listed in the design notes):
  * Codebook law: the exact marginal of one coordinate of a uniform point on
    the unit sphere in d = 128 (Y^2 ~ Beta(1/2, (d-1)/2)); so every vector is
    stored as (fp32 norm, codes of the unit vector).
  * Rotation: Pi = H diag(s) / sqrt(d), H the Sylvester Hadamard matrix, s a
    seeded +-1 vector, one per layer, shared by K, V, all tiers and heads.
  * Quantiser: code = number of boundaries strictly below the coordinate;
    boundaries are midpoints of adjacent centroids.  The decision is taken
    in fp32 (coordinate and boundary both rounded to float32), the precision
    the GPU kernels decide in.  A zero vector stores norm 0 and codes
    2^(b-1) - 1.
  * Packing: code i of a vector occupies bits [b*i, b*i + b) of a
    little-endian bit string (4-bit: low nibble = even index).
  * Tiers: L1 = sinks + recent + marked tokens (a per-sequence set shared by
    heads), stored as TQ4(RoPE(k_t, t)) and TQ4(v_t).  L3 holds TQ4(k_t)
    pre-RoPE and TQ4(v_t) for every token.  Groups are positional blocks
    [gN, gN + N) over the whole context; members are the block's tokens that
    are not in L1; a block with no member is empty and never routed.  The
    summary pair is TQ3(mean of RoPE(k_t, t)) and TQ3(mean of v_t) over the
    members, means taken over the input values.
  * RoPE: rotate-half pairing (i, i + d/2), omega_i = theta^(-2i/d), angle
    p * omega_i evaluated in float64.
  * Routing: per KV head, s_g = sum over the head's query heads j of
    RoPE(q_j, pos) . k_hat_g; the beta largest (fp32 score, ties to the lower
    group index) are selected and listed in ascending group order, padded
    with -1 when fewer groups are non-empty.  Variants: the maximum over
    the query heads instead of the sum, and per-query-head routing (each
    query head selects its own beta groups with its own score and attends
    with that selection: the router's per-head wording taken literally).
  * Attention: for each query head, one softmax (scale 1/sqrt(d)) over L1
    tokens, unselected non-empty summaries (one entry each, no count bias)
    and the selected groups' non-L1 tokens recovered from L3 and rotated to
    their positions.
  * Codec (an ablation on the [TQ] page, "Plain-KV": scalar quantisation
    without the rotation): codec "plain" replaces Pi by the identity in every
    tier and keeps everything else (fp32 norm, the same codebook applied to
    the unrotated unit vector, packing, tiers, routing, attention).
  * TQ-QKV ([TQ] key contributions, item 1: TurboQuant plus a 1-bit QJL
    sketch of the key residual): with a sketch matrix S [m, d] (i.i.d.
    N(0, 1), an input like the signs), every 4-bit key -- L1 and L3 -- keeps
    bits = (S rho >= 0) and |rho| of its residual rho in the frame its logit
    is taken in, rotated by the codec: rho = Pi (RoPE(k_t, t) - RoPE(k^_t, t))
    for L3 (the fetched key is RoPE'd before its logit), rho = Pi (RoPE(k_t,
    t) - k^) for L1.  A token entry's logit gets the unbiased estimate
    sqrt(pi/2) / m |rho| sum_i (S Pi q^r)_i sign_i of q^r . (Pi^T rho) added
    before the 1/sqrt(d) scale; summaries get none.
  * Codec diagnostics ([TQ] metrics: relMSE with the K / V split, and the
    direction error as cosine similarity): relMSE = sum_t |x^_t - x_t|^2 /
    sum_t |x_t|^2 over a set of vectors; cosine = the mean over vectors of
    nonzero norm of x^_t . x_t / (|x^_t| |x_t|).
  * Prefill ([HSQ] section 4, results: the prefill overhead of compressing
    the prompt, 1.2-1.3x at 32K): the prompt's attention is the model's
    ordinary dense causal softmax attention over RoPE'd queries and keys
    (GQA, scale 1/sqrt(d)); HSQ changes only what is kept for decoding, the
    encode of the same K/V.  A fused prefill returns both.
  * Decode-time growth (the pages describe the tiers of a context and leave
    their growth open): a cache grown by appended tokens is, by definition,
    the encode of the longer context under the grown L1 set (grown_l1_mask):
    sinks, the positions marked at encode time, and the recent window at
    the new length.  The oracle therefore grows a cache by encoding again.
"""

from __future__ import annotations

import functools
from dataclasses import dataclass
from typing import Optional, Tuple

import numpy as np
from scipy import special

__all__ = [
    "D",
    "grown_l1_mask",
    "coordinate_pdf",
    "coordinate_cdf",
    "coordinate_cell_mass",
    "coordinate_partial_moment",
    "lloyd_max_codebook",
    "codebook",
    "sylvester_hadamard",
    "rotation_matrix",
    "rope_frequencies",
    "rope",
    "tq_encode",
    "tq_decode",
    "pack_codes",
    "unpack_codes",
    "near_boundary",
    "OracleCache",
    "encode",
    "route",
    "select_top_beta",
    "fetch_dequant",
    "decode_attn",
    "attention_entries",
    "cache_to_abi",
    "cache_from_abi",
    "record_bytes",
    "codec_rotation",
    "Sketch",
    "qjl_sketch",
    "qjl_estimate",
    "entry_sketches",
    "unpack_sketch_words",
    "key_residuals",
    "codec_errors",
    "CODECS",
    "prefill_attn",
    "prefill",
]

D = 128


# ---------------------------------------------------------------------------
# Codebook: Lloyd-Max for the coordinate law of a random unit vector ([TQ]).
# ---------------------------------------------------------------------------

def _log_norm_const(d: int) -> float:
    # C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2))
    return special.gammaln(d / 2.0) - 0.5 * np.log(np.pi) - special.gammaln((d - 1) / 2.0)


def coordinate_pdf(y, d: int = D):
    """Density of one coordinate of a uniform unit vector in R^d on [-1, 1]."""
    y = np.asarray(y, dtype=np.float64)
    inside = np.abs(y) < 1.0
    out = np.zeros_like(y)
    out[inside] = np.exp(_log_norm_const(d) + 0.5 * (d - 3) * np.log1p(-y[inside] ** 2))
    return out


def coordinate_cdf(y, d: int = D):
    """P(Y <= y) via Y^2 ~ Beta(1/2, (d-1)/2) and the symmetry of Y."""
    y = np.clip(np.asarray(y, dtype=np.float64), -1.0, 1.0)
    half = 0.5 * special.betainc(0.5, 0.5 * (d - 1), y * y)
    return np.where(y >= 0, 0.5 + half, 0.5 - half)


def coordinate_cell_mass(lo: float, hi: float, d: int = D) -> float:
    """P(lo < Y <= hi) for 0 <= lo < hi <= 1, without cancellation in the tail."""
    a, b = 0.5, 0.5 * (d - 1)
    return 0.5 * (special.betaincc(a, b, lo * lo) - special.betaincc(a, b, hi * hi))


def coordinate_partial_moment(lo: float, hi: float, d: int = D) -> float:
    """Integral of y f(y) over (lo, hi]; closed form
    C_d / (d - 1) * ((1 - lo^2)^((d-1)/2) - (1 - hi^2)^((d-1)/2))."""
    c = np.exp(_log_norm_const(d)) / (d - 1)
    e = 0.5 * (d - 1)
    return c * ((1.0 - lo * lo) ** e - (1.0 - hi * hi) ** e)


def lloyd_max_codebook(bits: int, d: int = D, tol: float = 1e-15,
                       max_iter: int = 200000) -> Tuple[np.ndarray, np.ndarray]:
    """Lloyd iteration for the symmetric coordinate law.

    Returns (centroids [2^b] ascending, boundaries [2^b - 1] ascending).
    Only the positive half is iterated; the negative half is its mirror, so
    the middle boundary is exactly 0.
    """
    L = 1 << bits
    half = L // 2
    # start: Gaussian quantiles of the cell mid-probabilities, scaled by 1/sqrt(d)
    p = special.ndtri((half + np.arange(half) + 0.5) / L) / np.sqrt(d)
    for _ in range(max_iter):
        edges = np.concatenate([[0.0], 0.5 * (p[:-1] + p[1:]), [1.0]])
        new = np.array([coordinate_partial_moment(edges[i], edges[i + 1], d)
                        / coordinate_cell_mass(edges[i], edges[i + 1], d)
                        for i in range(half)])
        delta = np.max(np.abs(new - p))
        p = new
        if delta < tol:
            break
    centroids = np.concatenate([-p[::-1], p])
    bounds = 0.5 * (centroids[:-1] + centroids[1:])
    bounds[half - 1] = 0.0
    return centroids, bounds


@functools.lru_cache(maxsize=None)
def _codebook_cached(bits: int, d: int):
    c, t = lloyd_max_codebook(bits, d)
    c.setflags(write=False)
    t.setflags(write=False)
    return c, t


def codebook(bits: int, d: int = D) -> Tuple[np.ndarray, np.ndarray]:
    """(centroids, boundaries) in float64 for b bits, cached per process."""
    return _codebook_cached(int(bits), int(d))


# ---------------------------------------------------------------------------
# Rotation ([TQ]: randomised Walsh-Hadamard transform).
# ---------------------------------------------------------------------------

def sylvester_hadamard(d: int = D) -> np.ndarray:
    """H[i, j] = (-1)^popcount(i & j), d a power of two."""
    i = np.arange(d)[:, None]
    j = np.arange(d)[None, :]
    x = i & j
    pc = np.zeros_like(x)
    while np.any(x):
        pc += x & 1
        x >>= 1
    return np.where(pc % 2 == 0, 1.0, -1.0)


def rotation_matrix(signs: np.ndarray) -> np.ndarray:
    """Pi = H diag(s) / sqrt(d) (apply the signs first, then H)."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.shape[0]
    return sylvester_hadamard(d) * s[None, :] / np.sqrt(d)


CODECS = ("tq", "plain")


def codec_rotation(signs: np.ndarray, codec: str = "tq") -> np.ndarray:
    """The codec's rotation: Pi for TurboQuant, the identity for Plain-KV."""
    if codec == "tq":
        return rotation_matrix(signs)
    if codec == "plain":
        return np.eye(len(signs))
    raise ValueError(f"unknown codec {codec!r}")


# ---------------------------------------------------------------------------
# RoPE: the fetched originals are "rotated to their positions" ([HSQ] decode
# process, step 2).  Rotate-half pairing, float64 angles.
# ---------------------------------------------------------------------------

def rope_frequencies(d: int = D, theta: float = 1.0e6) -> np.ndarray:
    return theta ** (-2.0 * np.arange(d // 2) / d)


def rope(x: np.ndarray, pos, theta: float = 1.0e6) -> np.ndarray:
    """Rotate x[..., d] at positions pos (broadcast against x[..., 0])."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_frequencies(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


# ---------------------------------------------------------------------------
# TurboQuant scalar quantiser ([HSQ] key components; [TQ] setup item 1).
# ---------------------------------------------------------------------------

def tq_encode(x: np.ndarray, bits: int, Pi: np.ndarray):
    """x[..., d] -> (codes uint8 [..., d], norms float32 [...], y float64 [..., d]).

    n = ||x|| rounded to float32; y = Pi (x / n); code = #{k : f32(y) > f32(tau_k)}.
    """
    x = np.asarray(x, dtype=np.float64)
    _, tau = codebook(bits, x.shape[-1])
    n32 = np.linalg.norm(x, axis=-1).astype(np.float32)
    n = n32.astype(np.float64)
    safe = np.where(n > 0, n, 1.0)
    y = (x / safe[..., None]) @ Pi.T
    y = np.where((n > 0)[..., None], y, 0.0)
    y32 = y.astype(np.float32)
    tau32 = tau.astype(np.float32)
    codes = (y32[..., None] > tau32).sum(axis=-1).astype(np.uint8)
    return codes, n32, y


def tq_decode(codes: np.ndarray, norms: np.ndarray, bits: int, Pi: np.ndarray) -> np.ndarray:
    """x_hat = n * Pi^T c[codes], float64, original frame."""
    c, _ = codebook(bits, codes.shape[-1])
    return np.asarray(norms, dtype=np.float64)[..., None] * (c[codes.astype(np.int64)] @ Pi)


def near_boundary(y: np.ndarray, bits: int, rel: float = 1e-5) -> np.ndarray:
    """Coordinates within rel * max(|tau_k|, 1/sqrt(d)) of some boundary tau_k."""
    y = np.asarray(y, dtype=np.float64)
    _, tau = codebook(bits, y.shape[-1])
    tol = rel * np.maximum(np.abs(tau), 1.0 / np.sqrt(y.shape[-1]))
    return np.any(np.abs(y[..., None] - tau) <= tol, axis=-1)


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Little-endian bit string: code i occupies bits [b*i, b*i + b)."""
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    bitplanes = (codes[..., :, None] >> np.arange(bits, dtype=np.uint8)) & 1
    flat = bitplanes.reshape(codes.shape[:-1] + (d * bits,))
    return np.packbits(flat, axis=-1, bitorder="little")


def unpack_codes(packed: np.ndarray, bits: int, d: int = D) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    flat = np.unpackbits(packed, axis=-1, bitorder="little")[..., : d * bits]
    planes = flat.reshape(packed.shape[:-1] + (d, bits)).astype(np.uint8)
    return (planes << np.arange(bits, dtype=np.uint8)).sum(axis=-1).astype(np.uint8)


@dataclass
class Sketch:
    """1-bit sketches of key residuals: bits[..., i] = (S rho)_i >= 0, norm = |rho| (fp32)."""
    bits: np.ndarray
    norm: np.ndarray


def qjl_sketch(rho: np.ndarray, S: np.ndarray) -> Sketch:
    """[TQ] TQ-QKV: the 1-bit Johnson-Lindenstrauss sketch of a key's
    quantisation residual rho[..., d] under the sketch matrix S [m, d]."""
    rho = np.asarray(rho, dtype=np.float64)
    return Sketch(bits=(rho @ np.asarray(S, np.float64).T) >= 0.0,
                  norm=np.linalg.norm(rho, axis=-1).astype(np.float32))


def qjl_estimate(Sq: np.ndarray, sk: Sketch) -> np.ndarray:
    """Estimate of q . rho from the sketch: sqrt(pi/2) / m * |rho| * sum_i (S q)_i sign_i,
    sign_i = +1 where the bit is set, else -1.  Sq [..., m] broadcasts against sk."""
    m = sk.bits.shape[-1]
    signs = np.where(sk.bits, 1.0, -1.0)
    return np.sqrt(np.pi / 2.0) / m * sk.norm.astype(np.float64) * np.sum(signs * Sq, axis=-1)


def codec_errors(x: np.ndarray, x_hat: np.ndarray) -> dict:
    """[TQ] metrics over the vectors x[..., d] and their reconstructions:
    relMSE = sum |x^ - x|^2 / sum |x|^2 and the mean cosine similarity over
    vectors where both norms are nonzero (float64)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1, np.shape(x)[-1])
    xh = np.asarray(x_hat, dtype=np.float64).reshape(x.shape)
    den = float(np.sum(x * x))
    rel = float(np.sum((xh - x) ** 2)) / den if den > 0 else 0.0
    nx, nh = np.linalg.norm(x, axis=1), np.linalg.norm(xh, axis=1)
    ok = (nx > 0) & (nh > 0)
    cos = float(np.mean(np.sum(x[ok] * xh[ok], axis=1) / (nx[ok] * nh[ok]))) if ok.any() else 1.0
    return {"relmse": rel, "cosine": cos}


# ---------------------------------------------------------------------------
# Tiers ([HSQ] three-tier architecture).
# ---------------------------------------------------------------------------

@dataclass
class _Store:
    """One set of stored vectors: either TurboQuant codes or exact vectors."""
    bits: int
    codes: Optional[np.ndarray] = None    # uint8 [..., d]
    norms: Optional[np.ndarray] = None    # float32 [...]
    y: Optional[np.ndarray] = None        # float64 [..., d] rotated unit coords (encode only)
    exact: Optional[np.ndarray] = None    # float64 [..., d] when quantisation is off

    def vectors(self, Pi: np.ndarray) -> np.ndarray:
        if self.exact is not None:
            return self.exact
        return tq_decode(self.codes, self.norms, self.bits, Pi)


def _store(x: np.ndarray, bits: int, Pi: np.ndarray, quantize: bool) -> _Store:
    if not quantize:
        return _Store(bits=bits, exact=np.asarray(x, dtype=np.float64).copy())
    codes, norms, y = tq_encode(x, bits, Pi)
    return _Store(bits=bits, codes=codes, norms=norms, y=y)


@dataclass
class OracleCache:
    N: int
    T: int
    theta: float
    signs: np.ndarray          # [d] int8
    l1_mask: np.ndarray        # [B, T] bool
    l1_count: np.ndarray       # [B] int
    l1_pos: np.ndarray         # [B, L1max] int (-1 padded), ascending
    l1_k: _Store               # [B, Hkv, L1max, d] post-RoPE keys
    l1_v: _Store               # [B, Hkv, L1max, d]
    l2_cnt: np.ndarray         # [B, G] members per group
    l2_k: _Store               # [B, Hkv, G, d] summary keys (post-RoPE frame)
    l2_v: _Store               # [B, Hkv, G, d]
    l3_k: _Store               # [B, Hkv, T, d] pre-RoPE keys
    l3_v: _Store               # [B, Hkv, T, d]
    quantized: bool = True
    codec: str = "tq"
    qjl_S: Optional[np.ndarray] = None     # [m, d] sketch matrix (TQ-QKV) or None
    l1_qjl: Optional["Sketch"] = None      # [B, Hkv, L1max] key-residual sketches
    l3_qjl: Optional["Sketch"] = None      # [B, Hkv, T]

    @property
    def Pi(self) -> np.ndarray:
        return codec_rotation(self.signs, self.codec)

    @property
    def G(self) -> int:
        return -(-self.T // self.N)

    @property
    def B(self) -> int:
        return self.l1_mask.shape[0]

    @property
    def Hkv(self) -> int:
        st = self.l3_k
        return (st.codes if st.codes is not None else st.exact).shape[1]


def encode(K: np.ndarray, V: np.ndarray, l1_mask: np.ndarray, signs: np.ndarray, N: int,
           theta: float = 1.0e6, quantize: bool = True, max_l1: Optional[int] = None,
           codec: str = "tq", qjl_S: Optional[np.ndarray] = None) -> OracleCache:
    """Build the three tiers from pre-RoPE K, V [B, Hkv, T, d] at positions 0..T-1."""
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, Hkv, T, d = K.shape
    G = -(-T // N)
    Pi = codec_rotation(signs, codec)
    l1_mask = np.asarray(l1_mask, dtype=bool)
    counts = l1_mask.sum(axis=1)
    L1max = int(counts.max()) if max_l1 is None else int(max_l1)
    if counts.max() > L1max:
        raise ValueError("L1 set larger than max_l1")
    l1_pos = np.full((B, L1max), -1, dtype=np.int64)
    for b in range(B):
        p = np.nonzero(l1_mask[b])[0]
        l1_pos[b, : len(p)] = p

    t_all = np.arange(T)
    K_rope = rope(K, t_all, theta)                               # [B, Hkv, T, d]

    # L1: post-RoPE keys and values of the focal tokens (zero rows beyond the count)
    l1_kx = np.zeros((B, Hkv, L1max, d))
    l1_vx = np.zeros((B, Hkv, L1max, d))
    for b in range(B):
        p = l1_pos[b, : counts[b]]
        l1_kx[b, :, : len(p)] = K_rope[b][:, p]
        l1_vx[b, :, : len(p)] = V[b][:, p]

    # L2: means over each block's non-L1 members
    l2_cnt = np.zeros((B, G), dtype=np.int64)
    l2_kx = np.zeros((B, Hkv, G, d))
    l2_vx = np.zeros((B, Hkv, G, d))
    for b in range(B):
        for g in range(G):
            t = np.arange(g * N, min((g + 1) * N, T))
            m = t[~l1_mask[b, t]]
            l2_cnt[b, g] = len(m)
            if len(m):
                l2_kx[b, :, g] = K_rope[b][:, m].mean(axis=1)
                l2_vx[b, :, g] = V[b][:, m].mean(axis=1)

    cache = OracleCache(
        N=N, T=T, theta=theta, signs=np.asarray(signs, dtype=np.int8), l1_mask=l1_mask,
        l1_count=counts.astype(np.int64), l1_pos=l1_pos,
        l1_k=_store(l1_kx, 4, Pi, quantize), l1_v=_store(l1_vx, 4, Pi, quantize),
        l2_cnt=l2_cnt,
        l2_k=_store(l2_kx, 3, Pi, quantize), l2_v=_store(l2_vx, 3, Pi, quantize),
        l3_k=_store(K, 4, Pi, quantize), l3_v=_store(V, 4, Pi, quantize),
        quantized=quantize, codec=codec,
    )
    if qjl_S is not None:
        if not quantize:
            raise ValueError("the residual sketch needs quantised keys")
        S = np.asarray(qjl_S, dtype=np.float64)
        r3, r1 = key_residuals(cache, K)
        cache.qjl_S, cache.l3_qjl, cache.l1_qjl = S, qjl_sketch(r3, S), qjl_sketch(r1, S)
    return cache


def key_residuals(cache: OracleCache, K: np.ndarray):
    """TQ-QKV: the key residuals of a cache's stored codes against the input
    keys K [B, Hkv, T, d], each in the frame its logit is taken in, rotated by
    the codec: L3 [B, Hkv, T, d] = Pi RoPE(k_t - k^_t, t); L1 [B, Hkv, L1max, d]
    = Pi (RoPE(k_t, t) - k^) for the L1 slots (zero rows past the count)."""
    K = np.asarray(K, dtype=np.float64)
    Pi = cache.Pi
    T = cache.T
    r3 = rope(K - cache.l3_k.vectors(Pi), np.arange(T), cache.theta) @ Pi.T
    k1 = cache.l1_k.vectors(Pi)
    x1 = np.zeros_like(k1)
    for b in range(K.shape[0]):
        c = int(cache.l1_count[b])
        p = cache.l1_pos[b, :c]
        x1[b, :, :c] = rope(K[b][:, p], p, cache.theta)
        k1[b, :, c:] = 0.0
    return r3, (x1 - k1) @ Pi.T


def grown_l1_mask(l1_mask: np.ndarray, T_new: int, sinks: int, recent: int) -> np.ndarray:
    """[HSQ] three-tier architecture, L1 focal tier (attention sinks, an
    optional recent window, reader-marked tokens), after the context grows
    from T = l1_mask.shape[1] to T_new tokens: the sinks [0, sinks), every
    L1 position of the encode-time mask below the encode-time window
    [T - recent, T) (the marked ones), and the window [T_new - recent, T_new)."""
    l1_mask = np.asarray(l1_mask, dtype=bool)
    B, T = l1_mask.shape
    if T_new < T:
        raise ValueError("a cache only grows")
    out = np.zeros((B, T_new), dtype=bool)
    kept = l1_mask.copy()
    kept[:, max(T - recent, 0):] = False          # the old window slides on
    out[:, :T] = kept
    out[:, : min(sinks, T_new)] = True
    out[:, max(T_new - recent, 0):] = True
    return out


# ---------------------------------------------------------------------------
# Decode: routing, fetching, attention ([HSQ] decode process, steps 1-3).
# ---------------------------------------------------------------------------

def _heads(Hq: int, Hkv: int):
    r = Hq // Hkv
    return [list(range(h * r, (h + 1) * r)) for h in range(Hkv)]


def select_top_beta(scores32: np.ndarray, nonempty: np.ndarray, beta: int) -> np.ndarray:
    """Indices of the beta largest scores (ties to the lower index), ascending,
    padded with -1 when fewer than beta entries are non-empty."""
    idx = np.nonzero(nonempty)[0]
    order = np.lexsort((idx, -scores32[idx].astype(np.float64)))
    chosen = np.sort(idx[order[:beta]])
    out = np.full(beta, -1, dtype=np.int64)
    out[: len(chosen)] = chosen
    return out


def route(cache: OracleCache, q: np.ndarray, pos: np.ndarray, beta: int, agg: str = "sum"):
    """Routing scores (float64, -inf for empty groups) and the selection.
    [HSQ] decode process, step 1 (a per-head router scores the summary keys
    against the current query).  agg:
      "sum"  -- per KV head, the sum of its query heads' scores (the reading
                the library defaults to): scores [B, Hkv, G], sel [B, Hkv, beta];
      "max"  -- per KV head, the group's score for its best query head;
      "head" -- per query head, its own score against its KV head's
                summaries: scores [B, Hq, G], sel [B, Hq, beta]."""
    if agg not in ("sum", "max", "head"):
        raise ValueError("agg must be 'sum', 'max' or 'head'")
    B, Hq, d = q.shape
    Hkv = cache.Hkv
    qr = rope(np.asarray(q, dtype=np.float64), np.asarray(pos)[:, None], cache.theta)
    khat = cache.l2_k.vectors(cache.Pi)                              # [B, Hkv, G, d]
    rows = Hq if agg == "head" else Hkv
    scores = np.full((B, rows, cache.G), -np.inf)
    sel = np.full((B, rows, beta), -1, dtype=np.int64)
    for b in range(B):
        ne = cache.l2_cnt[b] > 0
        for h, js in enumerate(_heads(Hq, Hkv)):
            if agg == "head":
                for j in js:
                    scores[b, j] = np.where(ne, khat[b, h] @ qr[b, j], -np.inf)
                    sel[b, j] = select_top_beta(scores[b, j].astype(np.float32), ne, beta)
                continue
            if agg == "sum":
                s = khat[b, h] @ qr[b, js].sum(axis=0)
            else:
                s = (khat[b, h] @ qr[b, js].T).max(axis=1)           # best of the KV head's query heads
            scores[b, h] = np.where(ne, s, -np.inf)
            sel[b, h] = select_top_beta(scores[b, h].astype(np.float32), ne, beta)
    return sel, scores


def fetch_dequant(cache: OracleCache, sel: np.ndarray):
    """Recover the selected groups' originals from L3.

    Returns k [B, Hkv, beta, N, d] (RoPE applied at each token's position,
    original frame), v [same] and valid [B, Hkv, beta, N] (False for -1
    slots, positions >= T and L1 members, which attention already sees).
    """
    B, Hkv, beta = sel.shape
    N, T = cache.N, cache.T
    d = len(cache.signs)
    kx = cache.l3_k.vectors(cache.Pi)
    vx = cache.l3_v.vectors(cache.Pi)
    k = np.zeros((B, Hkv, beta, N, d))
    v = np.zeros((B, Hkv, beta, N, d))
    valid = np.zeros((B, Hkv, beta, N), dtype=bool)
    for b in range(B):
        for h in range(Hkv):
            for i in range(beta):
                g = int(sel[b, h, i])
                if g < 0:
                    continue
                for n in range(N):
                    t = g * N + n
                    if t >= T:
                        continue
                    k[b, h, i, n] = rope(kx[b, h, t], t, cache.theta)
                    v[b, h, i, n] = vx[b, h, t]
                    valid[b, h, i, n] = not cache.l1_mask[b, t]
    return k, v, valid


def attention_entries(cache: OracleCache, sel: np.ndarray, b: int, h: int, kv_head: Optional[int] = None):
    """Keys, values and provenance of the softmax entry set for selection row
    sel[b, h] over the tiers of KV head kv_head (default h).

    provenance rows: (kind, index) with kind 1 = L1 slot, 2 = summary group,
    3 = fetched token position.
    """
    Pi = cache.Pi
    s_row = sel[b, h]
    h = h if kv_head is None else kv_head
    N, T = cache.N, cache.T
    keys, vals, prov = [], [], []
    c = int(cache.l1_count[b])
    if c:
        keys.append(cache.l1_k.vectors(Pi)[b, h, :c])
        vals.append(cache.l1_v.vectors(Pi)[b, h, :c])
        prov += [(1, i) for i in range(c)]
    chosen = set(int(g) for g in s_row if g >= 0)
    groups = [g for g in range(cache.G) if cache.l2_cnt[b, g] > 0 and g not in chosen]
    if groups:
        keys.append(cache.l2_k.vectors(Pi)[b, h, groups])
        vals.append(cache.l2_v.vectors(Pi)[b, h, groups])
        prov += [(2, g) for g in groups]
    toks = [t for g in sorted(chosen) for t in range(g * N, min((g + 1) * N, T))
            if not cache.l1_mask[b, t]]
    if toks:
        toks = np.array(toks)
        kx = cache.l3_k.vectors(Pi)[b, h, toks]
        keys.append(rope(kx, toks, cache.theta))
        vals.append(cache.l3_v.vectors(Pi)[b, h, toks])
        prov += [(3, int(t)) for t in toks]
    d = len(cache.signs)
    if not keys:
        return np.zeros((0, d)), np.zeros((0, d)), prov
    return np.concatenate(keys), np.concatenate(vals), prov


def entry_sketches(cache: OracleCache, sel: np.ndarray, b: int, h: int, kv_head: Optional[int] = None):
    """The residual sketches of attention_entries(...)'s entries (None for a
    cache without them): L1 slots and fetched tokens carry theirs; summaries
    carry a zero norm (no correction)."""
    if cache.qjl_S is None:
        return None
    _, _, prov = attention_entries(cache, sel, b, h, kv_head)
    hb = h if kv_head is None else kv_head
    m = cache.qjl_S.shape[0]
    bits = np.zeros((len(prov), m), bool)
    norm = np.zeros(len(prov), np.float32)
    for e, (kind, idx) in enumerate(prov):
        if kind == 1:
            bits[e], norm[e] = cache.l1_qjl.bits[b, hb, idx], cache.l1_qjl.norm[b, hb, idx]
        elif kind == 3:
            bits[e], norm[e] = cache.l3_qjl.bits[b, hb, idx], cache.l3_qjl.norm[b, hb, idx]
    return Sketch(bits=bits, norm=norm)


def decode_attn(cache: OracleCache, q: np.ndarray, pos: np.ndarray, sel: np.ndarray) -> np.ndarray:
    """out [B, Hq, d] float64: softmax(q_r . k / sqrt(d)) v over the entry set.

    sel [B, Hkv, beta]: one selection per KV head, shared by its query heads;
    sel [B, Hq, beta] with Hq > Hkv: each query head attends with its own."""
    B, Hq, d = q.shape
    Hkv = cache.Hkv
    per_head = sel.shape[1] == Hq and Hq != Hkv
    if sel.shape[1] != (Hq if per_head else Hkv):
        raise ValueError("sel must have Hkv or Hq rows")
    qr = rope(np.asarray(q, dtype=np.float64), np.asarray(pos)[:, None], cache.theta)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h, js in enumerate(_heads(Hq, Hkv)):
            shared = None if per_head else attention_entries(cache, sel, b, h)
            shared_sk = None if per_head else entry_sketches(cache, sel, b, h)
            for j in js:
                keys, vals, _ = attention_entries(cache, sel, b, j, kv_head=h) if per_head else shared
                if len(keys) == 0:
                    continue
                dots = keys @ qr[b, j]
                sk = entry_sketches(cache, sel, b, j, kv_head=h) if per_head else shared_sk
                if sk is not None:  # TQ-QKV: + the sketch estimate of q . residual
                    dots = dots + qjl_estimate(cache.qjl_S @ (cache.Pi @ qr[b, j]), sk)
                logits = dots / np.sqrt(d)
                w = np.exp(logits - logits.max())
                out[b, j] = (w / w.sum()) @ vals
    return out


# ---------------------------------------------------------------------------
# Byte layout shared with the C ABI (a data format both sides must agree on).
# ---------------------------------------------------------------------------

def record_bytes(N: int, d: int = D) -> int:
    """One L3 group record: K codes [N][d/2], V codes [N][d/2], K norms [N] f32, V norms [N] f32."""
    return N * (d // 2) * 2 + N * 4 * 2


def cache_to_abi(cache: OracleCache, max_l1: Optional[int] = None) -> dict:
    """Pack a quantised oracle cache into the library's buffer layout (numpy arrays)."""
    if not cache.quantized:
        raise ValueError("only a quantised cache has a byte layout")
    B, Hkv = cache.l3_k.codes.shape[:2]
    d = len(cache.signs)
    N, T, G = cache.N, cache.T, cache.G
    L1max = cache.l1_pos.shape[1] if max_l1 is None else max_l1
    out = {}
    l1kc = np.zeros((B, Hkv, L1max, d // 2), np.uint8)
    l1vc = np.zeros_like(l1kc)
    l1kn = np.zeros((B, Hkv, L1max), np.float32)
    l1vn = np.zeros_like(l1kn)
    n0 = cache.l1_pos.shape[1]
    l1kc[:, :, :n0] = pack_codes(cache.l1_k.codes, 4)
    l1vc[:, :, :n0] = pack_codes(cache.l1_v.codes, 4)
    l1kn[:, :, :n0] = cache.l1_k.norms
    l1vn[:, :, :n0] = cache.l1_v.norms
    pos = np.full((B, L1max), -1, np.int32)
    pos[:, :n0] = cache.l1_pos
    out.update(l1_kc=l1kc, l1_vc=l1vc, l1_kn=l1kn, l1_vn=l1vn, l1_pos=pos,
               l1_count=cache.l1_count.astype(np.int32))
    out["l2_kc"] = pack_codes(cache.l2_k.codes, 3)
    out["l2_vc"] = pack_codes(cache.l2_v.codes, 3)
    out["l2_kn"] = cache.l2_k.norms.astype(np.float32)
    out["l2_vn"] = cache.l2_v.norms.astype(np.float32)
    out["l2_cnt"] = cache.l2_cnt.astype(np.uint8)
    # L3 records; slots past T hold the zero-vector encoding (norm 0, codes 7)
    zero4 = np.full(d, 7, np.uint8)
    kc = np.broadcast_to(zero4, (B, Hkv, G * N, d)).copy()
    vc = kc.copy()
    kn = np.zeros((B, Hkv, G * N), np.float32)
    vn = np.zeros_like(kn)
    kc[:, :, :T] = cache.l3_k.codes
    vc[:, :, :T] = cache.l3_v.codes
    kn[:, :, :T] = cache.l3_k.norms
    vn[:, :, :T] = cache.l3_v.norms
    rec = np.zeros((B, Hkv, G, record_bytes(N, d)), np.uint8)
    h = d // 2
    rec[..., : N * h] = pack_codes(kc, 4).reshape(B, Hkv, G, N * h)
    rec[..., N * h: 2 * N * h] = pack_codes(vc, 4).reshape(B, Hkv, G, N * h)
    rec[..., 2 * N * h: 2 * N * h + 4 * N] = kn.reshape(B, Hkv, G, N).view(np.uint8).reshape(B, Hkv, G, 4 * N)
    rec[..., 2 * N * h + 4 * N:] = vn.reshape(B, Hkv, G, N).view(np.uint8).reshape(B, Hkv, G, 4 * N)
    out["l3"] = rec
    return out


def unpack_sketch_words(words: np.ndarray, m: int = D) -> np.ndarray:
    """uint32 words [..., m/32] -> bits [..., m]: bit i is bit (i mod 32) of word i // 32."""
    w = np.asarray(words, dtype=np.uint32)
    return ((w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(w.shape[:-1] + (m,))


def cache_from_abi(bufs: dict, l1_mask: np.ndarray, signs: np.ndarray, N: int, T: int,
                   theta: float = 1.0e6, codec: str = "tq", qjl_S: Optional[np.ndarray] = None) -> OracleCache:
    """Read a cache back from the library's buffer layout (numpy copies of the buffers)."""
    rec = np.asarray(bufs["l3"], dtype=np.uint8)
    B, Hkv, G, _ = rec.shape
    d = len(signs)
    h = d // 2
    kc = unpack_codes(rec[..., : N * h].reshape(B, Hkv, G, N, h), 4, d).reshape(B, Hkv, G * N, d)
    vc = unpack_codes(rec[..., N * h: 2 * N * h].reshape(B, Hkv, G, N, h), 4, d).reshape(B, Hkv, G * N, d)
    kn = np.ascontiguousarray(rec[..., 2 * N * h: 2 * N * h + 4 * N]).view(np.float32).reshape(B, Hkv, G * N)
    vn = np.ascontiguousarray(rec[..., 2 * N * h + 4 * N:]).view(np.float32).reshape(B, Hkv, G * N)
    counts = np.asarray(bufs["l1_count"]).astype(np.int64)
    L1max = int(counts.max()) if len(counts) else 0
    pos = np.asarray(bufs["l1_pos"])[:, :L1max].astype(np.int64)
    out = OracleCache(
        N=N, T=T, theta=theta, signs=np.asarray(signs, np.int8),
        l1_mask=np.asarray(l1_mask, bool), l1_count=counts, l1_pos=pos,
        l1_k=_Store(4, codes=unpack_codes(bufs["l1_kc"][:, :, :L1max], 4, d),
                    norms=np.asarray(bufs["l1_kn"])[:, :, :L1max]),
        l1_v=_Store(4, codes=unpack_codes(bufs["l1_vc"][:, :, :L1max], 4, d),
                    norms=np.asarray(bufs["l1_vn"])[:, :, :L1max]),
        l2_cnt=np.asarray(bufs["l2_cnt"]).astype(np.int64),
        l2_k=_Store(3, codes=unpack_codes(bufs["l2_kc"], 3, d), norms=np.asarray(bufs["l2_kn"])),
        l2_v=_Store(3, codes=unpack_codes(bufs["l2_vc"], 3, d), norms=np.asarray(bufs["l2_vn"])),
        l3_k=_Store(4, codes=kc[:, :, :T], norms=kn[:, :, :T]),
        l3_v=_Store(4, codes=vc[:, :, :T], norms=vn[:, :, :T]),
        quantized=True, codec=codec,
    )
    if qjl_S is not None:
        out.qjl_S = np.asarray(qjl_S, np.float64)
        m = out.qjl_S.shape[0]
        out.l1_qjl = Sketch(bits=unpack_sketch_words(np.asarray(bufs["l1_qs"])[:, :, :L1max], m),
                            norm=np.asarray(bufs["l1_qn"])[:, :, :L1max].astype(np.float32))
        out.l3_qjl = Sketch(bits=unpack_sketch_words(np.asarray(bufs["l3_qs"])[:, :, :T], m),
                            norm=np.asarray(bufs["l3_qn"])[:, :, :T].astype(np.float32))
    return out


# ---------------------------------------------------------------------------
# Prefill ([HSQ] section 4, results: prefill overhead at 32K).
# ---------------------------------------------------------------------------

def prefill_attn(Q: np.ndarray, K: np.ndarray, V: np.ndarray, theta: float = 1.0e6,
                 q_start: int = 0) -> np.ndarray:
    """Dense causal attention of a prompt: K, V [B, Hkv, Tk, d] pre-RoPE at
    positions 0..Tk-1 and Q [B, Hq, Tq, d] pre-RoPE at positions q_start ..
    q_start + Tq - 1 (q_start = 0, Tq = Tk: the whole prompt; a later start
    gives those rows of the whole prompt's output); the query at position p of
    head j attends to keys 0..p of KV head j // (Hq / Hkv) with weights
    softmax(RoPE(q, p) . RoPE(k_s, s) / sqrt(d)).  Returns O [B, Hq, Tq, d] in
    float64."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    B, Hq, Tq, d = Q.shape
    Hkv, Tk = K.shape[1], K.shape[2]
    if q_start < 0 or q_start + Tq > Tk:
        raise ValueError("queries must sit at positions covered by the keys")
    tq = q_start + np.arange(Tq)
    tk = np.arange(Tk)
    Qr = rope(Q, tq, theta)
    Kr = rope(K, tk, theta)
    causal = tk[None, :] <= tq[:, None]                  # [query, key]
    O = np.zeros_like(Q)
    for b in range(B):
        for h, js in enumerate(_heads(Hq, Hkv)):
            for j in js:
                logits = (Qr[b, j] @ Kr[b, h].T) / np.sqrt(d)
                logits = np.where(causal, logits, -np.inf)
                w = np.exp(logits - logits.max(axis=1, keepdims=True))
                O[b, j] = (w / w.sum(axis=1, keepdims=True)) @ V[b, h]
    return O


def prefill(Q: np.ndarray, K: np.ndarray, V: np.ndarray, l1_mask: np.ndarray, signs: np.ndarray, N: int,
            theta: float = 1.0e6, **encode_kw):
    """A prompt's prefill with HSQ: the dense causal attention output and the
    three-tier cache of the same K/V (encode)."""
    return prefill_attn(Q, K, V, theta), encode(K, V, l1_mask, signs, N, theta, **encode_kw)
