"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and its host-only parts (codebook, sizes, validation, fault
injection) agree with the oracle and the header.  No GPU is touched."""

import ctypes

import numpy as np
import pytest

import oracle as O
from hsq_harness import ensure_built


@pytest.fixture(scope="module")
def H():
    ensure_built()
    import hierarchical_kv_cache_hsq_gb300 as H
    H.load_library()
    return H


def test_every_declared_symbol_is_exported(H):
    lib = H.load_library()
    names = H.declared_symbols()
    assert {"hsq_encode", "hsq_route", "hsq_fetch_dequant", "hsq_decode_attn"} <= set(names)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_version(H):
    assert H.hsq_version().startswith("hsq-gb300")


@pytest.mark.parametrize("bits", [3, 4])
def test_host_codebook_matches_oracle(H, bits):
    c, t = H.hsq_codebook(bits, 128)
    oc, ot = O.codebook(bits)
    np.testing.assert_allclose(c, oc, rtol=0, atol=1e-12)
    np.testing.assert_allclose(t, ot, rtol=0, atol=1e-12)
    assert t[(1 << bits) // 2 - 1] == 0.0


def test_host_codebook_other_dims_and_errors(H):
    c, _ = H.hsq_codebook(2, 64)
    oc, _ = O.lloyd_max_codebook(2, 64)
    np.testing.assert_allclose(c, oc, atol=1e-12)
    lib = H.load_library()
    buf = np.zeros(512)
    assert lib.hsq_codebook(0, 128, buf.ctypes.data, buf.ctypes.data) == 1
    assert lib.hsq_codebook(3, 2, buf.ctypes.data, buf.ctypes.data) == 1
    assert lib.hsq_codebook(3, 128, None, buf.ctypes.data) == 1


def test_cache_sizes(H):
    cfg = H.make_config(32, 8, 16, 64, 2, 32768, 600, 40000)
    s = H.hsq_cache_sizes(cfg, 2, 32768)
    G = 2048
    assert s["l3"] == 2 * 8 * G * O.record_bytes(16) == 2 * 8 * G * 2176
    assert s["l1_kc"] == 2 * 8 * 600 * 64 and s["l1_kn"] == 2 * 8 * 600 * 4
    assert s["l2_kc"] == 2 * 8 * G * 48 and s["l2_cnt"] == 2 * G
    assert s["l1_bitmap"] == 2 * 1024 * 4
    assert s["staging"] == 2 * 8 * 64 * 2176
    s2 = H.hsq_cache_sizes(cfg, 1, 1000)  # ragged: G = ceil(1000 / 16) = 63
    assert s2["l2_kc"] == 8 * 63 * 48 and s2["l1_bitmap"] == 32 * 4
    assert s["win_kv"] == 0 and s["gsum"] == 0  # not growable: no growth state
    g = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 32768, 600, 40000, sinks=4, recent=256), 2, 32768)
    assert g["win_kv"] == 2 * 8 * 256 * 2 * 128 * 4  # the window's input K and V, float
    assert g["gsum"] == 2 * 8 * 260 * 4              # 128 + 128 sums, the count, padding


@pytest.mark.parametrize("field,value", [
    ("head_dim", 64), ("group_n", 12), ("beta", 0), ("beta", 513), ("bits_l1l3", 8),
    ("bits_l2", 4), ("rope_theta", 0.0), ("max_batch", 0), ("max_pos", 10), ("n_splits", 17),
    ("n_q_heads", 12), ("l1_sinks", -1), ("l1_recent", -1), ("l1_recent", 101),
    ("route_max", 2), ("codec", 2), ("codec", -1), ("route_per_head", 2), ("qjl", 2),
])
def test_invalid_config_rejected(H, field, value):
    cfg = H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000)
    setattr(cfg, field, value)
    lib = H.load_library()
    out = (ctypes.c_size_t * H._binding.HSQ_NBUF)()
    assert lib.hsq_cache_sizes(ctypes.byref(cfg), 1, 4096, ctypes.cast(out, ctypes.c_void_p)) == 1
    h = ctypes.c_void_p()
    assert lib.hsq_create(ctypes.byref(cfg), ctypes.byref(h)) == 1
    assert not h.value
    assert len(lib.hsq_last_error(None)) > 0


def test_cache_sizes_rejects_out_of_range_shapes(H):
    cfg = H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000)
    with pytest.raises(H.HSQError):
        H.hsq_cache_sizes(cfg, 3, 4096)
    with pytest.raises(H.HSQError):
        H.hsq_cache_sizes(cfg, 1, 4097)


def test_injected_allocation_failure_needs_no_gpu(H):
    cfg = H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000)
    H.hsq_debug_set_fault(H.HSQ_FAULT_ALLOC)
    try:
        with pytest.raises(H.HSQError) as ei:
            H.Context(cfg)
        assert ei.value.status == 3
    finally:
        H.hsq_debug_set_fault(0)


def test_unsupported_head_ratio(H):
    cfg = H.make_config(24, 8, 16, 64, 1, 4096, 100, 5000)  # r = 3
    lib = H.load_library()
    h = ctypes.c_void_p()
    assert lib.hsq_create(ctypes.byref(cfg), ctypes.byref(h)) == 6


def test_null_context_calls_fail_cleanly(H):
    lib = H.load_library()
    c = H._binding.hsq_cache()
    assert lib.hsq_encode(None, ctypes.byref(c), None, None, 0, None) == 1
    assert lib.hsq_route(None, ctypes.byref(c), None, None, None, None, None) == 1
    assert lib.hsq_decode_attn(None, ctypes.byref(c), None, None, None, None, 0, None) == 1
    assert lib.hsq_fetch_dequant(None, ctypes.byref(c), None, None, None, None, None) == 1
    assert lib.hsq_append(None, ctypes.byref(c), None, None, 0, None) == 1
    assert lib.hsq_destroy(None) == 0


def test_bitmap_packing_matches_definition(H):
    rng = np.random.default_rng(0)
    mask = rng.random((3, 70)) < 0.3
    words = H.l1_bitmap_words(mask)
    assert words.shape == (3, 3)
    for b in range(3):
        for t in range(70):
            assert bool((int(words[b, t >> 5]) >> (t & 31)) & 1) == mask[b, t]


def test_codec_names(H):
    assert H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000).codec == 0
    assert H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000, codec="plain").codec == 1
    with pytest.raises(ValueError):
        H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000, codec="spectral")
    # the cache layout does not depend on the codec
    a = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000), 2, 4096)
    b = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, codec="plain"), 2, 4096)
    assert a == b


def test_per_head_routing_sizes_and_exclusion(H):
    base = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000), 2, 4096)
    per = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, route_per_head=True), 2, 4096)
    assert per["staging"] == 4 * base["staging"]  # one row per query head (r = 4)
    assert {k: v for k, v in per.items() if k != "staging"} == {k: v for k, v in base.items() if k != "staging"}
    with pytest.raises(H.HSQError):
        H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, route_per_head=True,
                                        route_max=True), 2, 4096)


def test_qjl_sizes_and_codec_requirement(H):
    base = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000), 2, 4096)
    q = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, qjl=True), 2, 4096)
    assert all(base[n] == 0 for n in ("l1_qs", "l1_qn", "l3_qs", "l3_qn"))
    assert q["l3_qs"] == 2 * 8 * 256 * 16 * 16 and q["l3_qn"] == 2 * 8 * 256 * 16 * 4  # 16 B + 4 B per token
    assert q["l1_qs"] == 2 * 8 * 100 * 16 and q["l1_qn"] == 2 * 8 * 100 * 4
    with pytest.raises(H.HSQError):
        H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, codec="plain", qjl=True), 2, 4096)


def test_hot_table_sizes_and_requirements(H):
    base = H.hsq_cache_sizes(H.make_config(40, 8, 16, 256, 4, 32768, 600, 40000), 4, 32768)
    hot = H.hsq_cache_sizes(H.make_config(40, 8, 16, 256, 4, 32768, 600, 40000, hot_slots=1024), 4, 32768)
    assert base["hot_rec"] == 0 and base["hot_tag"] == 0
    assert hot["hot_rec"] == 4 * 8 * 1024 * 16 * 136 and hot["hot_tag"] == 4 * 8 * 1024 * 4
    assert {k: v for k, v in hot.items() if not k.startswith("hot_")} == \
        {k: v for k, v in base.items() if not k.startswith("hot_")}
    for bad in (dict(hot_slots=8), dict(hot_slots=100), dict(hot_slots=2048), dict(hot_slots=-16),
                dict(hot_slots=64, qjl=True), dict(hot_slots=64, codec="plain"),
                dict(hot_slots=64, route_per_head=True)):
        with pytest.raises(H.HSQError):
            H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, **bad), 2, 4096)


def test_overlap_launch_flag_is_checked(H):
    ok = H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000, overlap_launch=True), 2, 4096)
    assert ok == H.hsq_cache_sizes(H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000), 2, 4096)
    cfg = H.make_config(32, 8, 16, 64, 2, 4096, 100, 5000)
    cfg.overlap_launch = 2
    with pytest.raises(H.HSQError):
        H.hsq_cache_sizes(cfg, 2, 4096)


def test_unaligned_l3_rejected_before_any_cuda_call(H):
    # every pointer non-NULL (never dereferenced: validation fails first), l3 off a 16-byte boundary
    cfg = H.make_config(32, 8, 16, 64, 1, 4096, 100, 5000)
    c = H._binding.hsq_cache()
    c.B, c.T = 1, 4096
    fake = 1 << 20
    for name, _ in H._binding.hsq_cache._fields_:
        if name not in ("B", "T", "l3_on_host", "t_cap"):
            setattr(c, name, fake)
    c.l3 = fake + 8
    lib = H.load_library()
    buf = np.zeros(64, dtype=np.int32)
    assert lib.hsq_route_noalloc(ctypes.byref(cfg), ctypes.byref(c), fake, fake, buf.ctypes.data, None) == 1
    assert b"16-byte aligned" in lib.hsq_last_error(None)
