"""ctypes binding of the HSQ C ABI (``include/hsq.h``).

Argument marshalling only: every step of the compressed-KV path runs in the
CUDA kernels of ``_build/libhsq.so``.  torch supplies device / pinned memory
and stream handles.  If the library has not been built the loader raises --
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Dict, Optional

import numpy as np

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "_build", "libhsq.so")
HEADER = os.path.join(ROOT, "include", "hsq.h")

HSQ_OK, HSQ_ERR_INVALID, HSQ_ERR_CUDA, HSQ_ERR_NOMEM = 0, 1, 2, 3
HSQ_ERR_TIMEOUT, HSQ_ERR_DEVICE_CHECK, HSQ_ERR_UNSUPPORTED = 4, 5, 6
HSQ_DTYPE_F32, HSQ_DTYPE_BF16 = 0, 1
HSQ_ATTN_FROM_STAGING = 1
HSQ_FAULT_ALLOC, HSQ_FAULT_FETCH = 1, 2
HSQ_DEVERR_SEL, HSQ_DEVERR_POS, HSQ_DEVERR_L1_OVER, HSQ_DEVERR_WAIT, HSQ_DEVERR_GROW = 1, 2, 4, 8, 16

BUFFERS = ["l1_kc", "l1_vc", "l1_kn", "l1_vn", "l1_pos", "l1_count", "l2_kc", "l2_vc", "l2_kn",
           "l2_vn", "l2_cnt", "l3", "l1_bitmap", "staging", "win_kv", "gsum", "l1_qs", "l1_qn", "l3_qs", "l3_qn",
           "hot_rec", "hot_tag"]
HSQ_NBUF = len(BUFFERS)
CODECS = {"tq": 0, "plain": 1}  # hsq_codec


class HSQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"hsq status {status}: {msg}")
        self.status = status


class hsq_config(ctypes.Structure):
    _fields_ = [
        ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("group_n", ctypes.c_int), ("beta", ctypes.c_int), ("bits_l1l3", ctypes.c_int),
        ("bits_l2", ctypes.c_int), ("rope_theta", ctypes.c_double), ("max_batch", ctypes.c_int),
        ("max_ctx", ctypes.c_int), ("max_l1", ctypes.c_int), ("max_pos", ctypes.c_int),
        ("n_splits", ctypes.c_int), ("l1_sinks", ctypes.c_int), ("l1_recent", ctypes.c_int),
        ("route_max", ctypes.c_int), ("codec", ctypes.c_int), ("route_per_head", ctypes.c_int),
        ("qjl", ctypes.c_int), ("hot_slots", ctypes.c_int), ("overlap_launch", ctypes.c_int),
    ]


class hsq_cache(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("T", ctypes.c_int),
        ("l1_kc", ctypes.c_void_p), ("l1_vc", ctypes.c_void_p), ("l1_kn", ctypes.c_void_p),
        ("l1_vn", ctypes.c_void_p), ("l1_pos", ctypes.c_void_p), ("l1_count", ctypes.c_void_p),
        ("l2_kc", ctypes.c_void_p), ("l2_vc", ctypes.c_void_p), ("l2_kn", ctypes.c_void_p),
        ("l2_vn", ctypes.c_void_p), ("l2_cnt", ctypes.c_void_p),
        ("l3", ctypes.c_void_p), ("l3_on_host", ctypes.c_int),
        ("l1_bitmap", ctypes.c_void_p), ("signs", ctypes.c_void_p), ("staging", ctypes.c_void_p),
        ("t_cap", ctypes.c_int), ("win_kv", ctypes.c_void_p), ("gsum", ctypes.c_void_p),
        ("qjl_s", ctypes.c_void_p), ("l1_qs", ctypes.c_void_p), ("l1_qn", ctypes.c_void_p),
        ("l3_qs", ctypes.c_void_p), ("l3_qn", ctypes.c_void_p),
        ("hot_rec", ctypes.c_void_p), ("hot_tag", ctypes.c_void_p),
    ]


_lib = None
_vp = ctypes.c_void_p
_SIGS = {
    "hsq_codebook": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _vp, _vp]),
    "hsq_cache_sizes": (ctypes.c_int, [ctypes.POINTER(hsq_config), ctypes.c_int, ctypes.c_int, _vp]),
    "hsq_create": (ctypes.c_int, [ctypes.POINTER(hsq_config), ctypes.POINTER(_vp)]),
    "hsq_destroy": (ctypes.c_int, [_vp]),
    "hsq_encode": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, ctypes.c_int, _vp]),
    "hsq_route": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, _vp, _vp, _vp]),
    "hsq_fetch_dequant": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, _vp, _vp, _vp]),
    "hsq_recover": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]),
    "hsq_decode_attn": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, _vp, _vp, ctypes.c_int, _vp]),
    "hsq_decode_step": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, _vp, _vp, _vp]),
    "hsq_append": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, ctypes.c_int, _vp]),
    "hsq_sync_status": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(ctypes.c_int)]),
    "hsq_route_noalloc": (ctypes.c_int, [ctypes.POINTER(hsq_config), ctypes.POINTER(hsq_cache), _vp, _vp, _vp, _vp]),
    "hsq_prefill_workspace_size": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    "hsq_prefill": (ctypes.c_int, [_vp, ctypes.POINTER(hsq_cache), _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, _vp,
                                   _vp, ctypes.c_size_t, _vp]),
    "hsq_last_error": (ctypes.c_char_p, [_vp]),
    "hsq_debug_set_fault": (ctypes.c_int, [ctypes.c_uint]),
    "hsq_version": (ctypes.c_char_p, []),
}


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libhsq.so (built by ``hierarchical_kv_cache_hsq_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"HSQ CUDA library not built ({p} missing): run "
                           "`python -m hierarchical_kv_cache_hsq_gb300.build` first")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name, None)
        if fn is None:
            continue
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def declared_symbols() -> list:
    """Function names declared in include/hsq.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hsq_[a-z_]+)\s*\(", text)))


def _check(st: int, ctx=None):
    if st != HSQ_OK:
        lib = load_library()
        msg = lib.hsq_last_error(ctx)
        raise HSQError(st, msg.decode() if msg else "")


# -- host-only calls --------------------------------------------------------------

def hsq_codebook(bits: int, dim: int = 128):
    lib = load_library()
    c = np.zeros(1 << bits, np.float64)
    t = np.zeros((1 << bits) - 1, np.float64)
    _check(lib.hsq_codebook(bits, dim, c.ctypes.data, t.ctypes.data))
    return c, t


def make_config(Hq: int, Hkv: int, N: int, beta: int, max_batch: int, max_ctx: int, max_l1: int,
                max_pos: int, theta: float = 1.0e6, n_splits: int = 0, sinks: int = 0,
                recent: int = 0, route_max: bool = False, codec: str = "tq",
                route_per_head: bool = False, qjl: bool = False, hot_slots: int = 0,
                overlap_launch: bool = False) -> hsq_config:
    """recent > 0 makes caches of this context growable (hsq_append) with an
    L1 recent window of that length and `sinks` permanent sink positions;
    route_max scores a group by its best query head instead of their sum;
    codec "plain" quantises the unrotated unit vectors (Plain-KV) instead of
    TurboQuant's rotated ones; route_per_head gives every query head its own
    selection (sel [B, Hq, beta]); qjl adds TQ-QKV's 1-bit sketches of the key
    residuals (set the sketch matrix with set_qjl_matrix); hot_slots > 0 gives
    the fused decode step a device table of that many recently fetched L3
    records per (sequence, KV head); overlap_launch launches the decode kernels
    with programmatic stream serialization (the next layer's launch overlaps
    this one's tail; results unchanged)."""
    if codec not in CODECS:
        raise ValueError(f"codec must be one of {tuple(CODECS)}")
    return hsq_config(n_q_heads=Hq, n_kv_heads=Hkv, head_dim=128, group_n=N, beta=beta,
                      bits_l1l3=4, bits_l2=3, rope_theta=theta, max_batch=max_batch,
                      max_ctx=max_ctx, max_l1=max_l1, max_pos=max_pos, n_splits=n_splits,
                      l1_sinks=sinks, l1_recent=recent, route_max=1 if route_max else 0,
                      codec=CODECS[codec], route_per_head=1 if route_per_head else 0, qjl=1 if qjl else 0,
                      hot_slots=hot_slots, overlap_launch=1 if overlap_launch else 0)


def hsq_cache_sizes(cfg: hsq_config, B: int, T: int) -> Dict[str, int]:
    lib = load_library()
    out = (ctypes.c_size_t * HSQ_NBUF)()
    _check(lib.hsq_cache_sizes(ctypes.byref(cfg), B, T, ctypes.cast(out, _vp)))
    return {name: int(out[i]) for i, name in enumerate(BUFFERS)}


def hsq_debug_set_fault(mask: int):
    _check(load_library().hsq_debug_set_fault(mask))


def hsq_version() -> str:
    return load_library().hsq_version().decode()


# -- context and cache ---------------------------------------------------------------

def _stream_handle(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


class Context:
    """Owns an hsq_ctx (codebooks, RoPE tables, scratch) on the current device."""

    def __init__(self, cfg: hsq_config):
        self.cfg = cfg
        self.lib = load_library()
        h = _vp()
        _check(self.lib.hsq_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.handle = h

    @property
    def r(self) -> int:
        return self.cfg.n_q_heads // self.cfg.n_kv_heads

    def close(self):
        if self.handle:
            self.lib.hsq_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def last_error(self) -> str:
        return self.lib.hsq_last_error(self.handle).decode()


@dataclass
class CacheBuffers:
    """The caller-owned buffers of one layer's cache (torch tensors) and its C view."""
    B: int
    T: int
    N: int
    Hkv: int
    max_l1: int
    beta: int
    tensors: Dict[str, "object"]
    signs: "object"
    l3_on_host: bool
    t_cap: int = 0       # layout capacity in tokens (0: T)
    recent: int = 0      # recent-window length of a growable cache
    sel_heads: int = 0   # selection rows per sequence (Hq under per-query-head routing; 0: Hkv)
    qjl_s: "object" = None  # [128, 128] float32 sketch matrix (TQ-QKV) or None

    @property
    def cap(self) -> int:
        return self.t_cap or self.T

    @property
    def G(self) -> int:
        """Groups of the layout (of the capacity; those past T are empty)."""
        return -(-self.cap // self.N)

    def struct(self) -> hsq_cache:
        t = self.tensors
        c = hsq_cache(B=self.B, T=self.T, l3_on_host=1 if self.l3_on_host else 0, t_cap=self.t_cap)
        for name in BUFFERS:
            setattr(c, name, _ptr(t.get(name)))
        c.signs = _ptr(self.signs)
        c.qjl_s = _ptr(self.qjl_s)
        return c

    # shaped views (for tests and diagnostics)
    def view(self, name: str):
        t = self.tensors[name]
        B, H, L1, G, N = self.B, self.Hkv, self.max_l1, self.G, self.N
        shapes = {
            "l1_kc": (B, H, L1, 64), "l1_vc": (B, H, L1, 64), "l1_kn": (B, H, L1), "l1_vn": (B, H, L1),
            "l1_pos": (B, L1), "l1_count": (B,), "l2_kc": (B, H, G, 48), "l2_vc": (B, H, G, 48),
            "l2_kn": (B, H, G), "l2_vn": (B, H, G), "l2_cnt": (B, G), "l3": (B, H, G, N * 136),
            "l1_bitmap": (B, (self.cap + 31) // 32),
            "staging": (B, self.sel_heads or H, self.beta, N * 136),
            "win_kv": (B, H, self.recent, 2, 128), "gsum": (B, H, 260),
            "l1_qs": (B, H, L1, 4), "l1_qn": (B, H, L1), "l3_qs": (B, H, G * N, 4), "l3_qn": (B, H, G * N),
            "hot_rec": (B, H, -1, N * 136), "hot_tag": (B, H, -1),
        }
        import torch
        dt = {"l1_kn": torch.float32, "l1_vn": torch.float32, "l2_kn": torch.float32,
              "l2_vn": torch.float32, "l1_pos": torch.int32, "l1_count": torch.int32,
              "l1_bitmap": torch.int32, "win_kv": torch.float32, "gsum": torch.float32,
              "l1_qs": torch.int32, "l1_qn": torch.float32, "l3_qs": torch.int32,
              "l3_qn": torch.float32, "hot_tag": torch.int32}.get(name, torch.uint8)
        if name.startswith("hot_"):
            return t.view(dt).view(shapes[name])
        n = int(np.prod(shapes[name]))
        return t.view(dt)[:n].view(shapes[name])


def l1_bitmap_words(mask: np.ndarray) -> np.ndarray:
    """[B, T] bool -> [B, ceil(T/32)] uint32, bit (t & 31) of word t >> 5."""
    mask = np.asarray(mask, dtype=bool)
    B, T = mask.shape
    W = (T + 31) // 32
    padded = np.zeros((B, W * 32), dtype=bool)
    padded[:, :T] = mask
    bits = padded.reshape(B, W, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)
    return bits.sum(axis=2).astype(np.uint32)


def allocate_cache(ctx: Context, B: int, T: int, l3_on_host: bool = True, with_staging: bool = True,
                   device=None, t_cap: Optional[int] = None) -> CacheBuffers:
    """Buffers for B sequences of T tokens, laid out for t_cap tokens (default T;
    a growable cache -- ctx.cfg.l1_recent > 0 -- gets its growth state too)."""
    import torch
    dev = torch.device("cuda") if device is None else torch.device(device)
    cap = T if t_cap is None else t_cap
    sizes = hsq_cache_sizes(ctx.cfg, B, cap)
    t = {}
    for name in BUFFERS:
        n = max(sizes[name], 16)
        if name == "staging" and not with_staging:
            continue
        if name in ("win_kv", "gsum", "l1_qs", "l1_qn", "l3_qs", "l3_qn", "hot_rec", "hot_tag") and sizes[name] == 0:
            continue
        if name == "hot_tag":  # every slot empty (-1)
            t[name] = torch.full((n,), 255, dtype=torch.uint8, device=dev)
        elif name == "l3" and l3_on_host:
            t[name] = torch.zeros(n, dtype=torch.uint8, pin_memory=True)
        else:
            t[name] = torch.zeros(n, dtype=torch.uint8, device=dev)
    signs = torch.ones(128, dtype=torch.int8, device=dev)
    qjl_s = torch.zeros((128, 128), dtype=torch.float32, device=dev) if ctx.cfg.qjl else None
    return CacheBuffers(qjl_s=qjl_s, B=B, T=T, N=ctx.cfg.group_n, Hkv=ctx.cfg.n_kv_heads, max_l1=ctx.cfg.max_l1,
                        beta=ctx.cfg.beta, tensors=t, signs=signs, l3_on_host=l3_on_host,
                        t_cap=0 if cap == T else cap, recent=ctx.cfg.l1_recent,
                        sel_heads=ctx.cfg.n_q_heads if ctx.cfg.route_per_head else ctx.cfg.n_kv_heads)


def set_layer_inputs(cache: CacheBuffers, l1_mask: np.ndarray, signs: np.ndarray):
    """Upload the L1 membership bitmap and the sign vector of a layer."""
    import torch
    words = l1_bitmap_words(l1_mask)
    Wc = (cache.cap + 31) // 32  # one row per sequence at the layout's stride
    if words.shape[1] > Wc:
        raise ValueError("L1 mask longer than the cache capacity")
    rows = np.zeros((words.shape[0], Wc), np.uint32)
    rows[:, : words.shape[1]] = words
    bm = cache.tensors["l1_bitmap"]
    src = torch.from_numpy(rows.view(np.uint8).reshape(-1).copy())
    bm[: src.numel()].copy_(src)
    cache.signs.copy_(torch.from_numpy(np.asarray(signs, np.int8)))


def set_qjl_matrix(cache: CacheBuffers, S: np.ndarray):
    """Upload the [128, 128] sketch matrix of a TQ-QKV cache (before hsq_encode)."""
    import torch
    if cache.qjl_s is None:
        raise ValueError("the cache's context has no key-residual sketches (make_config(qjl=True))")
    cache.qjl_s.copy_(torch.from_numpy(np.ascontiguousarray(S, np.float32)))


# -- the four calls of the path (+ the fused step) ------------------------------------

def hsq_encode(ctx: Context, cache: CacheBuffers, K, V, stream=None):
    import torch
    if K.dtype == torch.bfloat16:
        dt = HSQ_DTYPE_BF16
    elif K.dtype == torch.float32:
        dt = HSQ_DTYPE_F32
    else:
        raise ValueError("K/V must be bfloat16 or float32")
    if not (K.is_contiguous() and V.is_contiguous() and V.dtype == K.dtype):
        raise ValueError("K and V must be contiguous and of one dtype")
    c = cache.struct()
    _check(ctx.lib.hsq_encode(ctx.handle, ctypes.byref(c), K.data_ptr(), V.data_ptr(), dt,
                              _stream_handle(stream)), ctx.handle)


def hsq_append(ctx: Context, cache: CacheBuffers, k, v, stream=None):
    """Append one token per sequence (k, v: [B, Hkv, 128], pre-RoPE) at position
    cache.T; cache.T grows by one."""
    import torch
    if k.dtype == torch.bfloat16:
        dt = HSQ_DTYPE_BF16
    elif k.dtype == torch.float32:
        dt = HSQ_DTYPE_F32
    else:
        raise ValueError("k/v must be bfloat16 or float32")
    if not (k.is_contiguous() and v.is_contiguous() and v.dtype == k.dtype):
        raise ValueError("k and v must be contiguous and of one dtype")
    c = cache.struct()
    _check(ctx.lib.hsq_append(ctx.handle, ctypes.byref(c), k.data_ptr(), v.data_ptr(), dt,
                              _stream_handle(stream)), ctx.handle)
    cache.T = c.T


def hsq_route(ctx: Context, cache: CacheBuffers, q, pos, sel, scores=None, stream=None):
    c = cache.struct()
    _check(ctx.lib.hsq_route(ctx.handle, ctypes.byref(c), q.data_ptr(), pos.data_ptr(), sel.data_ptr(),
                             _ptr(scores), _stream_handle(stream)), ctx.handle)


def hsq_fetch_dequant(ctx: Context, cache: CacheBuffers, sel, k_out=None, v_out=None, valid=None,
                      stream=None):
    c = cache.struct()
    _check(ctx.lib.hsq_fetch_dequant(ctx.handle, ctypes.byref(c), sel.data_ptr(), _ptr(k_out), _ptr(v_out),
                                     _ptr(valid), _stream_handle(stream)), ctx.handle)


def hsq_recover(ctx: Context, cache: CacheBuffers, g0: int, ng: int, k_out=None, v_out=None, stream=None):
    c = cache.struct()
    _check(ctx.lib.hsq_recover(ctx.handle, ctypes.byref(c), int(g0), int(ng), _ptr(k_out), _ptr(v_out),
                               _stream_handle(stream)), ctx.handle)


def hsq_decode_attn(ctx: Context, cache: CacheBuffers, q, pos, sel, out, flags: int = 0, stream=None):
    c = cache.struct()
    _check(ctx.lib.hsq_decode_attn(ctx.handle, ctypes.byref(c), q.data_ptr(), pos.data_ptr(), sel.data_ptr(),
                                   out.data_ptr(), flags, _stream_handle(stream)), ctx.handle)


def hsq_decode_step(ctx: Context, cache: CacheBuffers, q, pos, sel, out, stream=None):
    c = cache.struct()
    _check(ctx.lib.hsq_decode_step(ctx.handle, ctypes.byref(c), q.data_ptr(), pos.data_ptr(), sel.data_ptr(),
                                   out.data_ptr(), _stream_handle(stream)), ctx.handle)


def hsq_prefill_workspace_size(ctx: Context, B: int, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(ctx.lib.hsq_prefill_workspace_size(ctx.handle, B, T, ctypes.byref(n)), ctx.handle)
    return int(n.value)


def hsq_prefill(ctx: Context, cache: Optional[CacheBuffers], Q, K, V, out, workspace, stream=None):
    """Prefill: causal attention of the prompt into out (float32) and, with a
    cache, the encode of K/V (bf16 Q [B, Hq, T, 128], K/V [B, Hkv, T, 128])."""
    import torch
    for x in (Q, K, V):
        if x.dtype != torch.bfloat16 or not x.is_contiguous():
            raise ValueError("Q, K and V must be contiguous bfloat16")
    if out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be contiguous float32")
    B, _, T, _ = Q.shape
    c = ctypes.byref(cache.struct()) if cache is not None else None
    _check(ctx.lib.hsq_prefill(ctx.handle, c, Q.data_ptr(), K.data_ptr(), V.data_ptr(), B, T, out.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               _stream_handle(stream)), ctx.handle)


def hsq_route_noalloc(cfg: hsq_config, cache: CacheBuffers, q, pos, sel, stream=None):
    """Routing through the entry point that allocates no device memory."""
    lib = load_library()
    c = cache.struct()
    _check(lib.hsq_route_noalloc(ctypes.byref(cfg), ctypes.byref(c), q.data_ptr(), pos.data_ptr(),
                                 sel.data_ptr(), _stream_handle(stream)))


def hsq_sync_status(ctx: Context, stream=None) -> int:
    """Synchronise, return the device error word (raises on a CUDA error only)."""
    w = ctypes.c_int(0)
    st = ctx.lib.hsq_sync_status(ctx.handle, _stream_handle(stream), ctypes.byref(w))
    if st not in (HSQ_OK, HSQ_ERR_DEVICE_CHECK):
        _check(st, ctx.handle)
    return int(w.value)
