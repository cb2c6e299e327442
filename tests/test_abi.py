"""The C-ABI library loads, exports what include/gc.h declares, and rejects
bad arguments on the host before touching the GPU (CPU only)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gc():
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    gcmod.lib()
    return gcmod


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "gc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gc_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(gc):
    names = _declared_functions()
    assert len(names) >= 10
    L = C.CDLL(gc.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(gc):
    assert gc.status_string(gc.GC_OK) == "ok"
    assert "workspace" in gc.status_string(gc.GC_ERR_WORKSPACE)
    assert gc.version() >= 100


def _host_layout(gc, sizes, k=None):
    off = np.zeros(len(sizes) + 1, np.int64)
    off[1:] = np.cumsum(sizes)
    return gc.Layout(off, k, device="cpu")


def test_workspace_size_scales_with_layout(gc):
    small = _host_layout(gc, [1000, 5000], [10, 50])
    big = _host_layout(gc, [10_000_000, 5000], [10_000, 50])
    s1 = gc.workspace_size(small, gc.GC_OP_TOPK, gc.GC_EF)
    s2 = gc.workspace_size(big, gc.GC_OP_TOPK, gc.GC_EF)
    assert 0 < s1 < s2
    assert gc.workspace_size(big, gc.GC_OP_SIGN) > 0
    assert gc.workspace_size(big, gc.GC_OP_DECOMPRESS) > 0
    # random-k needs no sample buffer
    assert gc.workspace_size(big, gc.GC_OP_TOPK, gc.GC_RANDK) < s2


def test_layout_validation(gc):
    out = C.c_size_t()
    bad_k = _host_layout(gc, [10, 20], [11, 1])           # k > n
    assert gc.lib().gc_workspace_size(bad_k.host(), gc.GC_OP_TOPK, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    lay = _host_layout(gc, [10, 20], [1, 1])
    lay.off[1] = 10; lay.off[2] = 10                         # empty tensor
    assert gc.lib().gc_workspace_size(lay.host(), gc.GC_OP_TOPK, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    huge = _host_layout(gc, [2 ** 31], [1])                  # n >= 2^31
    assert gc.lib().gc_workspace_size(huge.host(), gc.GC_OP_TOPK, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    assert gc.lib().gc_workspace_size(lay.host(), 99, 0, C.byref(out)) == gc.GC_ERR_INVALID_ARG


def test_bucket_layouts_are_accepted_and_sized_like_their_tensors(gc):
    """A bucket (tensors t0..t1-1 of a larger arena, with that arena's
    offsets) validates, and needs the workspace of the same tensors laid
    out from zero; negative offsets are layout errors."""
    sizes, k = [100, 4097, 33, 70_001, 6], [1, 5, 2, 70, 6]
    whole = gc.Layout(np.concatenate([[0], np.cumsum(sizes)]), np.asarray(k, np.int64), device="cpu")
    b = whole.bucket(1, 4)
    assert list(b.off) == [100, 4197, 4230, 74231] and list(b.koff) == [1, 6, 8, 78]
    alone = gc.Layout(np.concatenate([[0], np.cumsum(sizes[1:4])]), np.asarray(k[1:4], np.int64), device="cpu")
    for op, flags in [(gc.GC_OP_TOPK, gc.GC_EF), (gc.GC_OP_TOPK, gc.GC_RANDK), (gc.GC_OP_MOMENTUM, 0),
                      (gc.GC_OP_SIGN, 0), (gc.GC_OP_QUANTIZE, 0), (gc.GC_OP_DECOMPRESS, 0)]:
        assert gc.workspace_size(b, op, flags) == gc.workspace_size(alone, op, flags) > 0
    out = C.c_size_t()
    neg = gc.Layout([-4, 10], np.asarray([1], np.int64), device="cpu")
    assert gc.lib().gc_workspace_size(neg.host(), gc.GC_OP_TOPK, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    assert gc.lib().gc_workspace_size(neg.host(), gc.GC_OP_SIGN, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    negk = gc.Layout([0, 10], np.asarray([1], np.int64), device="cpu", koff0=-1)
    assert gc.lib().gc_workspace_size(negk.host(), gc.GC_OP_TOPK, 0, C.byref(out)) == gc.GC_ERR_LAYOUT
    with pytest.raises(ValueError):
        whole.bucket(3, 3)


def test_bucket_offsets_match_brute_force(gc):
    """Layout.bucket keeps the arena's element and entry offsets; the word
    offsets a caller passes with a bucket are sums over the earlier tensors."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        T = int(rng.integers(1, 12))
        sizes = rng.integers(1, 5000, T)
        k = np.minimum(sizes, rng.integers(0, 300, T))
        L = gc.Layout(np.concatenate([[0], np.cumsum(sizes)]), k.astype(np.int64), device="cpu")
        t0 = int(rng.integers(0, T))
        t1 = int(rng.integers(t0 + 1, T + 1))
        B = L.bucket(t0, t1)
        assert B.T == t1 - t0
        assert list(B.off) == [int(sum(sizes[:t])) for t in range(t0, t1 + 1)]
        assert list(B.koff) == [int(sum(k[:t])) for t in range(t0, t1 + 1)]
        assert list(B.k) == list(k[t0:t1])
        assert L.word_offset(t0) == sum((int(n) + 31) // 32 for n in sizes[:t0])
        assert L.kept_word_offset(t0) == sum((int(x) + 31) // 32 for x in k[:t0])
        assert B.words == sum((int(n) + 31) // 32 for n in sizes[t0:t1])
        assert B.kept_words == sum((int(x) + 31) // 32 for x in k[t0:t1])


def test_argument_errors_return_before_any_launch(gc):
    lay = _host_layout(gc, [100], [5])
    L = gc.lib()
    P = C.c_void_p
    # flags that do not combine, or unknown bits
    for flags in (gc.GC_RANDK | gc.GC_INT8, gc.GC_UNBIASED, gc.GC_RANDK | gc.GC_UNBIASED | gc.GC_EF, 1 << 20):
        st = L.gc_ef_topk_compress(lay.host(), lay.host(), P(16), P(16), P(16), P(16), P(16), P(16),
                                   0, 0, flags, P(256), 1 << 20, None)
        assert st == gc.GC_ERR_INVALID_ARG, flags
    # misaligned gradient pointer
    st = L.gc_ef_topk_compress(lay.host(), lay.host(), P(18), P(16), P(16), P(16), None, None,
                               0, 0, gc.GC_EF, P(256), 1 << 20, None)
    assert st == gc.GC_ERR_ALIGNMENT
    # workspace too small / misaligned
    st = L.gc_ef_topk_compress(lay.host(), lay.host(), P(16), P(16), P(16), P(16), None, None,
                               0, 0, gc.GC_EF, P(256), 8, None)
    assert st == gc.GC_ERR_WORKSPACE
    st = L.gc_ef_topk_compress(lay.host(), lay.host(), P(16), P(16), P(16), P(16), None, None,
                               0, 0, gc.GC_EF, P(260), 1 << 30, None)
    assert st == gc.GC_ERR_WORKSPACE
    # missing payload buffers
    st = L.gc_ef_topk_compress(lay.host(), lay.host(), P(16), P(16), P(16), None, None, None,
                               0, 0, gc.GC_EF, P(256), 1 << 30, None)
    assert st == gc.GC_ERR_INVALID_ARG
    st = L.gc_quantize_stochastic(lay.host(), lay.host(), P(16), None, P(16), P(16), 1, 0, 0, 0,
                                  P(256), 1 << 30, None)
    assert st == gc.GC_ERR_INVALID_ARG                       # QSGD needs s >= 1
    st = L.gc_dense_decompress_accumulate(lay.host(), lay.host(), 1, 7, 16, None, None, P(16),
                                          P(256), 1 << 30, None)
    assert st == gc.GC_ERR_INVALID_ARG


def test_warmup_density_matches_oracle(gc):
    import oracle
    for kind in ("linear", "exponential", "step"):
        for step in (-3, 0, 1, 5, 9, 10, 11, 100):
            a = gc.warmup_density(step, 10, 0.25, 0.001, kind, 4)
            b = oracle.warmup_density(step, 10, 0.25, 0.001, kind)
            assert a == pytest.approx(b, rel=1e-15, abs=0)


def test_powersgd_validation(gc):
    ml = gc.MatrixLayout([0, 100], [10, 5], [10, 7], device="cpu")
    out = C.c_size_t()
    assert gc.lib().gc_powersgd_workspace_size(ml.host(), 4, C.byref(out)) == gc.GC_OK and out.value > 0
    assert gc.lib().gc_powersgd_workspace_size(ml.host(), 3, C.byref(out)) == gc.GC_ERR_INVALID_ARG
    bad = gc.MatrixLayout([0], [0], [5], device="cpu")
    assert gc.lib().gc_powersgd_workspace_size(bad.host(), 1, C.byref(out)) == gc.GC_ERR_LAYOUT
