"""GPU parity: every libgc entry point, called through the C ABI, against the
oracle on the same seeded inputs.

Bit-exact for indices, selected values, residuals, int8/QSGD codes, sign
bits, max-abs scales and scatter-add sums.  Norm-type scales (sign mean-|acc|,
QSGD L2 norm) are reduced in a different order on the two sides and must
agree within 1e-6 relative; the oracle is then re-run with the GPU's scale
and everything downstream of the scale must be bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32 = np.float32
REL_TOL = 1e-6


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _layout(gc, sizes, k=None, rho=None):
    if k is None:
        k = workloads.k_per_tensor(sizes, rho)
    return gc.Layout(workloads.prefix(sizes), np.asarray(k, np.int64), device="cuda")


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _grad(n, seed, kind="t3"):
    gen = torch.Generator().manual_seed(seed)
    if kind == "t3":
        x = torch.empty(n)
        workloads.fill_student_t(x, 3.0, 1e-3, gen)
    elif kind == "ties":
        x = torch.randint(-2, 3, (n,), generator=gen).float() * 1e-3
    elif kind == "zeros":
        x = torch.zeros(n)
        x[::3] = -0.0
    else:
        raise ValueError(kind)
    return x.float()


def _one_launch_expected(gc, L, flags):
    """Whether gc_ef_topk_compress runs as one cooperative launch: Top-k on
    at most 2^22 elements in at most 1024 tensors, unless a flag asks for
    the multi-kernel pipeline (random-k and GC_FORCE_EXACT use it too)."""
    return (not flags & (gc.GC_RANDK | gc.GC_FORCE_EXACT | gc.GC_MULTI_KERNEL) and L.T <= 1024
            and L.numel <= (1 << 22))


def _topk_check(gc, L, g_h, e_h, flags, seed, it, ws=None, expect_exact=None):
    """Runs one GPU call and the oracle; asserts bit-exact payload and residual,
    and that the call took the launch path the layout and flags call for."""
    dev = L.device
    K = L.total_k
    int8 = bool(flags & gc.GC_INT8)
    g = torch.from_numpy(g_h).to(dev)
    e = torch.from_numpy(e_h).to(dev) if e_h is not None else None
    idx = torch.full((max(K, 1),), -1, dtype=torch.int32, device=dev)
    val = torch.empty(max(K, 1), dtype=torch.float32, device=dev)
    q = torch.zeros(max(K, 1), dtype=torch.int8, device=dev) if int8 else None
    sc = torch.zeros(L.T, dtype=torch.float32, device=dev) if int8 else None
    if ws is None:
        ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    gc.ef_topk_compress(L, g, e, idx, val, q, sc, seed, it, flags, ws)
    diag = gc.get_device_status(ws)
    assert diag.error_bits == 0
    assert diag.one_launch == int(_one_launch_expected(gc, L, flags)), (diag.one_launch, flags)
    if expect_exact is not None:
        assert diag.exact_tensors == expect_exact, (diag.exact_tensors, expect_exact)
    gi, gv = idx.cpu().numpy()[:K], val.cpu().numpy()[:K]
    e_ref = e_h.copy() if e_h is not None else None
    randk = bool(flags & gc.GC_RANDK)
    for t in range(L.T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        ka, kb = int(L.koff[t]), int(L.koff[t + 1])
        et = e_ref[a:b] if e_ref is not None else None
        if randk:
            ri, rv = oracle.randk_tensor(g_h[a:b], et, int(L.k[t]), base=a, seed=seed, it=it,
                                         unbiased=bool(flags & gc.GC_UNBIASED))
            rq = rs = None
        else:
            ri, rv, rq, rs = oracle.ef_topk_tensor(g_h[a:b], et, int(L.k[t]), base=a, int8=int8,
                                                   seed=seed, it=it)
        assert np.array_equal(gi[ka:kb], ri), f"tensor {t}: indices differ"
        if int8:
            assert np.array_equal(q.cpu().numpy()[ka:kb], rq), f"tensor {t}: codes differ"
            assert _bits(sc.cpu().numpy()[t:t + 1])[0] == _bits(np.asarray([rs], F32))[0], f"tensor {t}: scale"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"tensor {t}: dequantized values differ"
        else:
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"tensor {t}: values differ"
    if e is not None:
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref)), "residual differs"
    return e_ref, diag


# ----------------------------------------------------------------------------- EF Top-k

LAYOUTS = {
    "single_1": [1],
    "tiny_ragged": [3, 5, 7, 1, 2],
    "misaligned": [4097, 1, 33, 100_003, 6],
    "many_small": [64] * 40 + [513, 4096, 4095],
    "medium": [300_000, 70_001, 12_345],
}


# "one_launch": the default path of these small layouts; "pipeline": the
# multi-kernel pipeline forced with GC_MULTI_KERNEL (GC_FORCE_EXACT implies it)
PATHS = ["one_launch", "pipeline"]


@pytest.mark.parametrize("name", sorted(LAYOUTS))
@pytest.mark.parametrize("flags_name", ["ef", "ef_int8", "noef", "ef_exact", "ef_int8_exact"])
@pytest.mark.parametrize("path", PATHS)
def test_topk_layouts(gc, name, flags_name, path):
    sizes = LAYOUTS[name]
    flags = {"ef": gc.GC_EF, "ef_int8": gc.GC_EF | gc.GC_INT8, "noef": 0,
             "ef_exact": gc.GC_EF | gc.GC_FORCE_EXACT,
             "ef_int8_exact": gc.GC_EF | gc.GC_INT8 | gc.GC_FORCE_EXACT}[flags_name]
    if flags & gc.GC_FORCE_EXACT and path == "one_launch":
        pytest.skip("GC_FORCE_EXACT always runs the pipeline")
    if path == "pipeline":
        flags |= gc.GC_MULTI_KERNEL
    rng = np.random.default_rng(len(sizes))
    k = [int(min(n, max(0, int(rng.integers(0, 3)) if n < 8 else int(np.ceil(0.01 * n))))) for n in sizes]
    if len(sizes) > 2:
        k[0] = sizes[0]               # k = n
        k[-1] = 0                     # k = 0
    L = _layout(gc, sizes, k=k)
    n = L.numel
    g = _grad(n, 3).numpy()
    e = (np.random.default_rng(4).standard_normal(n) * 1e-4).astype(F32) if flags & gc.GC_EF else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(3):
        g = _grad(n, 10 + it).numpy()
        e, _ = _topk_check(gc, L, g, e, flags, seed=5, it=it, ws=ws)


def _kept_quant_check(gc, L, g_h, state, kind, flags, seed, it, ws, momentum=False, beta=0.9, s_levels=16):
    """One GPU call of the Top-k + QSGD / sign entry points against the oracle.
    Protocol: indices bit-exact; each tensor's scale (a norm or mean over the
    kept values, reduced in a different order) within 1e-6 relative; then the
    oracle re-run with the GPU's scale, and codes or bits, decoded values and
    the residual (velocity) bit-exact.  `state` is e, or (u, v) with momentum;
    the oracle's updated state is returned."""
    dev = L.device
    K, T = L.total_k, L.T
    kq = {"qsgd": gc.GC_KEPT_QSGD, "sign": gc.GC_KEPT_SIGN}[kind]
    g = torch.from_numpy(g_h).to(dev)
    idx = torch.full((max(K, 1),), -1, dtype=torch.int32, device=dev)
    val = torch.empty(max(K, 1), dtype=torch.float32, device=dev)
    q = torch.full((max(K, 1),), 99, dtype=torch.int8, device=dev) if kind == "qsgd" else None
    bits = torch.full((max(L.kept_words, 1),), -1, dtype=torch.int32, device=dev) if kind == "sign" else None
    sc = torch.full((T,), -1.0, dtype=torch.float32, device=dev)
    if momentum:
        u_h, v_h = state
        u, v = torch.from_numpy(u_h).to(dev), torch.from_numpy(v_h).to(dev)
        gc.ef_topk_compress_momentum_quantized(L, g, u, v, beta, idx, val, q, bits, sc, kq, s_levels, seed, it,
                                               flags, ws)
    else:
        e = torch.from_numpy(state).to(dev) if state is not None else None
        gc.ef_topk_compress_quantized(L, g, e, idx, val, q, bits, sc, kq, s_levels, seed, it, flags, ws)
    assert gc.get_device_status(ws).error_bits == 0
    gi, gv, gsc = idx.cpu().numpy()[:K], val.cpu().numpy()[:K], sc.cpu().numpy()
    gq = q.cpu().numpy()[:K] if q is not None else None
    gb = bits.cpu().numpy().view(np.uint32) if bits is not None else None
    kw = workloads.prefix((L.k + 31) // 32)
    if momentum:
        u_ref, v_ref = u_h.copy(), v_h.copy()
    else:
        e_ref = state.copy() if state is not None else None
    for t in range(T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        ka, kb, kt = int(L.koff[t]), int(L.koff[t + 1]), int(L.k[t])
        if momentum:
            args = (g_h[a:b], u_ref[a:b].copy(), v_ref[a:b].copy(), kt, beta, kind, s_levels)
            _, _, _, _, s_ref = oracle.momentum_topk_quantized_tensor(*args, base=a, seed=seed, it=it)
        else:
            args = (g_h[a:b], None if e_ref is None else e_ref[a:b].copy(), kt, kind, s_levels)
            _, _, _, _, s_ref = oracle.ef_topk_quantized_tensor(*args, base=a, seed=seed, it=it)
        assert abs(float(gsc[t]) - s_ref) <= REL_TOL * abs(s_ref), f"tensor {t}: scale {gsc[t]} vs {s_ref}"
        # everything downstream of the scale, given the GPU's scale
        if momentum:
            ut, vt = u_ref[a:b], v_ref[a:b]
            ri, rv, rq, rb, _ = oracle.momentum_topk_quantized_tensor(g_h[a:b], ut, vt, kt, beta, kind, s_levels,
                                                                      base=a, seed=seed, it=it,
                                                                      scale_given=float(gsc[t]))
        else:
            et = None if e_ref is None else e_ref[a:b]
            ri, rv, rq, rb, _ = oracle.ef_topk_quantized_tensor(g_h[a:b], et, kt, kind, s_levels, base=a, seed=seed,
                                                                it=it, scale_given=float(gsc[t]))
        assert np.array_equal(gi[ka:kb], ri), f"tensor {t}: indices differ"
        assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"tensor {t}: decoded values differ"
        if kind == "qsgd":
            assert np.array_equal(gq[ka:kb], rq), f"tensor {t}: QSGD codes differ"
        else:
            assert np.array_equal(gb[kw[t]:kw[t + 1]], rb), f"tensor {t}: sign bits differ"
        if kt == 0:
            assert gsc[t] == 0.0
    if momentum:
        assert np.array_equal(_bits(u.cpu().numpy()), _bits(u_ref)), "u differs"
        assert np.array_equal(_bits(v.cpu().numpy()), _bits(v_ref)), "v differs"
        return (u_ref, v_ref)
    if e_ref is not None:
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref)), "residual differs"
    return e_ref


@pytest.mark.parametrize("name", ["tiny_ragged", "misaligned", "many_small", "medium"])
@pytest.mark.parametrize("kind", ["qsgd", "sign"])
@pytest.mark.parametrize("flags_name", ["ef", "noef", "ef_exact"])
def test_topk_kept_quantizers(gc, name, kind, flags_name):
    """EF Top-k + QSGD / sign of the kept values, three chained calls, with
    k = n and k = 0 tensors and ragged, misaligned tensor starts."""
    sizes = LAYOUTS[name]
    flags = {"ef": gc.GC_EF, "noef": 0, "ef_exact": gc.GC_EF | gc.GC_FORCE_EXACT}[flags_name]
    rng = np.random.default_rng(len(sizes) + 7)
    k = [int(min(n, max(0, int(rng.integers(0, 3)) if n < 8 else int(np.ceil(0.01 * n))))) for n in sizes]
    if len(sizes) > 2:
        k[0] = sizes[0]
        k[-1] = 0
    L = _layout(gc, sizes, k=k)
    n = L.numel
    e = (np.random.default_rng(4).standard_normal(n) * 1e-4).astype(F32) if flags & gc.GC_EF else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(3):
        g = _grad(n, 20 + it).numpy()
        e = _kept_quant_check(gc, L, g, e, kind, flags, seed=6, it=it, ws=ws, s_levels=16 if it != 1 else 5)


@pytest.mark.parametrize("kind", ["qsgd", "sign"])
@pytest.mark.parametrize("exact", [False, True])
def test_momentum_kept_quantizers(gc, kind, exact):
    sizes = LAYOUTS["misaligned"] + [70_000]
    L = _layout(gc, sizes, rho=0.005)
    n = L.numel
    flags = gc.GC_FORCE_EXACT if exact else 0
    rng = np.random.default_rng(9)
    state = ((rng.standard_normal(n) * 1e-4).astype(F32), (rng.standard_normal(n) * 1e-4).astype(F32))
    ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM, flags)
    for it in range(3):
        g = _grad(n, 30 + it).numpy()
        state = _kept_quant_check(gc, L, g, state, kind, flags, seed=7, it=it, ws=ws, momentum=True)


@pytest.mark.parametrize("kind", ["qsgd", "sign"])
def test_kept_quantizers_ties_and_extremes(gc, kind):
    """Ties straddling the k-th magnitude (kept ties enter the norm / mean),
    signed zeros, and magnitudes near the fp32 limits."""
    sizes = [10_000, 4096, 333, 70_000]
    L = _layout(gc, sizes, k=[37, 4096, 1, 700])
    n = L.numel
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
    e = np.zeros(n, F32)
    for it, gk in enumerate(["ties", "zeros", "ties"]):
        g = _grad(n, 40 + it, gk).numpy()
        e = _kept_quant_check(gc, L, g, e, kind, gc.GC_EF, seed=8, it=it, ws=ws)
    rng = np.random.default_rng(10)
    # the kept set's L2 norm must stay finite in fp32 (it is the payload's
    # scale): 700 kept values near 4e35 give N near 1e37
    big = (rng.standard_normal(n) * 1e35).astype(F32)
    tiny = (rng.standard_normal(n) * 1e-40).astype(F32)     # subnormal magnitudes
    for it, g in enumerate([big, tiny]):
        _kept_quant_check(gc, L, g, None, kind, 0, seed=9, it=it, ws=ws)


def test_kept_quantizer_arguments(gc):
    L = _layout(gc, [1000, 77], k=[10, 3])
    g = torch.zeros(1077, device="cuda")
    idx = torch.empty(13, dtype=torch.int32, device="cuda")
    q = torch.empty(13, dtype=torch.int8, device="cuda")
    sc = torch.empty(2, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, 0)
    for kind, s_levels, qq, bb, flags in [(gc.GC_KEPT_QSGD, 0, q, None, 0), (gc.GC_KEPT_QSGD, 128, q, None, 0),
                                          (gc.GC_KEPT_QSGD, 16, None, None, 0), (gc.GC_KEPT_SIGN, 0, None, None, 0),
                                          (7, 16, q, None, 0), (gc.GC_KEPT_QSGD, 16, q, None, gc.GC_INT8),
                                          (gc.GC_KEPT_QSGD, 16, q, None, gc.GC_RANDK)]:
        with pytest.raises(gc.GCError) as ei:
            gc.ef_topk_compress_quantized(L, g, None, idx, None, qq, bb, sc, kind, s_levels, 0, 0, flags, ws)
        assert ei.value.status == gc.GC_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", ["ties", "zeros"])
@pytest.mark.parametrize("path", ["one_launch", "pipeline", "pipeline_exact"])
def test_topk_ties(gc, kind, path):
    sizes = [10_000, 4096, 333, 70_000]
    L = _layout(gc, sizes, k=[37, 4096, 1, 700])
    n = L.numel
    exact = path == "pipeline_exact"
    flags = gc.GC_EF | {"one_launch": 0, "pipeline": gc.GC_MULTI_KERNEL,
                        "pipeline_exact": gc.GC_FORCE_EXACT}[path]
    e = np.zeros(n, F32)
    if kind == "zeros":
        e[::5] = -0.0
    g = _grad(n, 1, kind).numpy()
    _, d = _topk_check(gc, L, g, e, flags, seed=1, it=0)
    if kind == "ties" and path == "pipeline":
        # 20% of the 70,000-element tensor ties at the largest magnitude: more
        # candidates than its capacity, so the overflow fallback must have run
        assert d.overflow_tensors >= 1 and d.exact_tensors >= 1


@pytest.mark.parametrize("rho", [0.001, 0.01])
@pytest.mark.parametrize("flags_name", ["ef", "ef_int8"])
@pytest.mark.parametrize("path", PATHS)
def test_topk_boundary_ties(gc, rho, flags_name, path):
    """A group of equal magnitudes straddles the k-th rank (ties kept by lowest
    index); 0.1% gives short candidate chunks per unit, 1% long ones, so both
    candidate walks of the payload write meet a partial tie group."""
    n = 300_000
    flags = gc.GC_EF | (gc.GC_INT8 if flags_name == "ef_int8" else 0) | (gc.GC_MULTI_KERNEL if path == "pipeline" else 0)
    L = _layout(gc, [n, 4099], rho=rho)
    g = _grad(L.numel, 21).numpy()
    k0 = int(L.k[0])
    mag = np.sort(np.abs(g[:n]))[::-1]
    v = mag[k0 - 40]
    rng = np.random.default_rng(22)
    pos = rng.choice(n, 120, replace=False)
    g[pos] = np.where(rng.random(120) < 0.5, -v, v).astype(F32)
    e = np.zeros(L.numel, F32)
    _, d = _topk_check(gc, L, g, e, flags, seed=9, it=0, expect_exact=0)
    assert d.overflow_tensors == 0


@pytest.mark.parametrize("path", PATHS)
def test_topk_flat_2p20_ten_iterations(gc, path):
    """One flat fp32 gradient of 2^20 elements at 0.1% (k = 1049), EF, 10 fresh gradients."""
    lay = workloads.flat_layout(1 << 20)
    L = _layout(gc, lay.sizes, rho=0.001)
    assert L.total_k == 1049
    flags = gc.GC_EF | (gc.GC_MULTI_KERNEL if path == "pipeline" else 0)
    e = np.zeros(L.numel, F32)
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(10):
        g = workloads.make_grad(1, lay, it).numpy()
        e, d = _topk_check(gc, L, g, e, flags, seed=0, it=it, ws=ws, expect_exact=0)


@pytest.mark.parametrize("n", [1 << 22, (1 << 22) + 1])
def test_one_launch_size_boundary(gc, n):
    """2^22 elements is the largest arena the one-launch path takes; one more
    element and the call runs the pipeline (the check inside _topk_check)."""
    sizes = [n - 3000, 1000, 2000]
    L = _layout(gc, sizes, rho=0.001)
    e = np.zeros(L.numel, F32)
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF | gc.GC_INT8)
    for it in range(2):
        g = _grad(L.numel, 50 + it).numpy()
        e, _ = _topk_check(gc, L, g, e, gc.GC_EF | gc.GC_INT8, seed=4, it=it, ws=ws)


def test_topk_resnet50_and_randk(gc):
    """ResNet-50 (25.6M elements, above the one-launch path's 2^22): the pipeline."""
    lay = workloads.resnet50_layout()
    L = _layout(gc, lay.sizes, rho=0.01)
    assert L.total_k == 255_658
    flags = gc.GC_EF
    e = np.zeros(L.numel, F32)
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(3):
        g = workloads.make_grad(2, lay, it).numpy()
        e, d = _topk_check(gc, L, g, e, flags, seed=2, it=it, ws=ws)
        assert d.exact_tensors <= 3      # only degenerate tensors may need full passes
    e = np.zeros(L.numel, F32)
    for it in range(2):
        g = workloads.make_grad(2, lay, 100 + it).numpy()
        e, _ = _topk_check(gc, L, g, e, gc.GC_EF | gc.GC_RANDK, seed=3, it=it)


@pytest.mark.parametrize("flags_name", ["ef", "plain", "unbiased", "ef_exact"])
def test_randk_layouts(gc, flags_name):
    flags = {"ef": gc.GC_EF | gc.GC_RANDK, "plain": gc.GC_RANDK, "unbiased": gc.GC_RANDK | gc.GC_UNBIASED,
             "ef_exact": gc.GC_EF | gc.GC_RANDK | gc.GC_FORCE_EXACT}[flags_name]
    sizes = [4097, 1, 33, 100_003, 6, 64, 250_000]
    L = _layout(gc, sizes, k=[41, 1, 33, 1000, 0, 3, 2500])
    n = L.numel
    e = np.zeros(n, F32) if flags & gc.GC_EF else None
    for it in range(2):
        g = _grad(n, 20 + it).numpy()
        e, _ = _topk_check(gc, L, g, e, flags, seed=9, it=it)


# ----------------------------------------------------------------------------- momentum

def _momentum_check(gc, L, beta, flags, iters, seed=4, gen=None):
    dev = L.device
    n, K = L.numel, L.total_k
    int8 = bool(flags & gc.GC_INT8)
    u_h = np.zeros(n, F32)
    v_h = np.zeros(n, F32)
    u, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    idx = torch.empty(max(K, 1), dtype=torch.int32, device=dev)
    val = torch.empty(max(K, 1), dtype=torch.float32, device=dev)
    q = torch.empty(max(K, 1), dtype=torch.int8, device=dev) if int8 else None
    sc = torch.empty(L.T, dtype=torch.float32, device=dev) if int8 else None
    ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM, flags)
    for it in range(iters):
        g_h = gen(it) if gen else _grad(n, 40 + it).numpy()
        gc.ef_topk_compress_momentum(L, torch.from_numpy(g_h).to(dev), u, v, beta, idx, val, q, sc, seed, it,
                                     flags, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gi, gv = idx.cpu().numpy()[:K], val.cpu().numpy()[:K]
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            ri, rv, rq, rs = oracle.momentum_topk_tensor(g_h[a:b], u_h[a:b], v_h[a:b], int(L.k[t]), beta,
                                                         masking=not (flags & gc.GC_NO_MASK), base=a,
                                                         int8=int8, seed=seed, it=it)
            assert np.array_equal(gi[ka:kb], ri), f"it {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"it {it} tensor {t}: values"
            if int8:
                assert np.array_equal(q.cpu().numpy()[ka:kb], rq)
                assert sc.cpu().numpy()[t] == rs
        assert np.array_equal(_bits(u.cpu().numpy()), _bits(u_h)), f"it {it}: u"
        assert np.array_equal(_bits(v.cpu().numpy()), _bits(v_h)), f"it {it}: v"


@pytest.mark.parametrize("flags_name", ["mask", "nomask", "int8", "exact"])
def test_momentum_layouts(gc, flags_name):
    flags = {"mask": 0, "nomask": gc.GC_NO_MASK, "int8": gc.GC_INT8, "exact": gc.GC_FORCE_EXACT}[flags_name]
    sizes = [4097, 1, 33, 100_003, 64, 70_000]
    L = _layout(gc, sizes, rho=0.005)
    _momentum_check(gc, L, 0.9, flags, iters=3)


# ----------------------------------------------------------------------------- sign / quantize

def _sign_check(gc, L, g_h, e_h):
    dev = L.device
    g = torch.from_numpy(g_h).to(dev)
    e = torch.from_numpy(e_h).to(dev) if e_h is not None else None
    bits = torch.zeros(L.words, dtype=torch.int32, device=dev)
    mu = torch.zeros(L.T, dtype=torch.float32, device=dev)
    ws = gc.alloc_workspace(L, gc.GC_OP_SIGN)
    gc.sign_compress(L, g, e, bits, mu, ws)
    assert gc.get_device_status(ws).error_bits == 0
    gb, gm = bits.cpu().numpy().view(np.uint32), mu.cpu().numpy()
    ge = e.cpu().numpy() if e is not None else None
    n = np.diff(L.off)
    woff = workloads.prefix((n + 31) // 32)
    e_ref = e_h.copy() if e_h is not None else None
    for t in range(L.T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        et = e_ref[a:b] if e_ref is not None else None
        _, mu_ref = oracle.sign_tensor(g_h[a:b], None if et is None else et.copy())
        assert abs(float(gm[t]) - mu_ref) <= REL_TOL * abs(mu_ref), f"tensor {t}: mean |acc|"
        rb, _ = oracle.sign_tensor(g_h[a:b], et, mu_given=float(gm[t]))
        assert np.array_equal(gb[woff[t]:woff[t + 1]], rb), f"tensor {t}: sign bits"
    if ge is not None:
        assert np.array_equal(_bits(ge), _bits(e_ref)), "residual"
    return e_ref


@pytest.mark.parametrize("ef", [True, False])
def test_sign_layouts(gc, ef):
    sizes = [4097, 1, 33, 100_003, 6, 64, 31, 32, 250_000]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n = L.numel
    e = np.zeros(n, F32) if ef else None
    for it in range(3):
        g = _grad(n, 60 + it).numpy()
        g[::17] = -0.0
        e = _sign_check(gc, L, g, e)


def _quant_check(gc, L, g_h, e_h, mode, s, seed, it):
    dev = L.device
    g = torch.from_numpy(g_h).to(dev)
    e = torch.from_numpy(e_h).to(dev) if e_h is not None else None
    codes = torch.zeros(L.numel, dtype=torch.int8, device=dev)
    sc = torch.zeros(L.T, dtype=torch.float32, device=dev)
    ws = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE)
    gc.quantize_stochastic(L, g, e, codes, sc, gc.GC_Q_INT8 if mode == "int8" else gc.GC_Q_QSGD, s, seed, it, ws)
    assert gc.get_device_status(ws).error_bits == 0
    gcodes, gsc = codes.cpu().numpy(), sc.cpu().numpy()
    e_ref = e_h.copy() if e_h is not None else None
    for t in range(L.T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        et = e_ref[a:b] if e_ref is not None else None
        _, ref_sc = oracle.quantize_tensor(g_h[a:b], None if et is None else et.copy(), mode, s, base=a,
                                           seed=seed, it=it)
        if mode == "int8":
            assert gsc[t] == F32(ref_sc), f"tensor {t}: int8 scale must be exact"
        else:
            assert abs(float(gsc[t]) - ref_sc) <= REL_TOL * abs(ref_sc), f"tensor {t}: norm"
        rc, _ = oracle.quantize_tensor(g_h[a:b], et, mode, s, base=a, seed=seed, it=it,
                                       scale_given=float(gsc[t]))
        assert np.array_equal(gcodes[a:b], rc), f"tensor {t}: codes"
    if e is not None:
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref)), "residual"
    return e_ref


@pytest.mark.parametrize("mode,s", [("int8", 0), ("qsgd", 16), ("qsgd", 1), ("qsgd", 127)])
@pytest.mark.parametrize("ef", [False, True])
def test_quantize_layouts(gc, mode, s, ef):
    sizes = [4097, 1, 33, 100_003, 6, 64, 250_000]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n = L.numel
    e = (np.random.default_rng(1).standard_normal(n) * 1e-5).astype(F32) if ef else None
    for it in range(2):
        g = _grad(n, 80 + it).numpy()
        g[5] = 0.0
        e = _quant_check(gc, L, g, e, mode, s, seed=11, it=it)


@pytest.mark.parametrize("mode,s,ef", [("int8", 0, True), ("qsgd", 16, False), ("qsgd", 16, True)])
def test_quantize_large_and_ragged_tensors(gc, mode, s, ef):
    """A tensor of 2^23 + 3 elements among one-element, misaligned and
    ragged ones (unit tails of 1023 and 1 elements)."""
    sizes = [1, (1 << 23) + 3, 4097, 33, 1024, 1023, 100_003, 6, 2_000_001]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n = L.numel
    e = (np.random.default_rng(2).standard_normal(n) * 1e-5).astype(F32) if ef else None
    for it in range(2):
        e = _quant_check(gc, L, _grad(n, 90 + it).numpy(), e, mode, s, seed=12, it=it)


def test_sign_large_and_ragged_tensors(gc):
    sizes = [1, (1 << 23) + 3, 4097, 33, 1024, 1023, 100_003, 6, 2_000_001]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n = L.numel
    e = np.zeros(n, F32)
    for it in range(2):
        e = _sign_check(gc, L, _grad(n, 95 + it).numpy(), e)


def test_quantize_zero_tensor(gc):
    L = _layout(gc, [100, 37], k=[0, 0])
    for mode, s in (("int8", 0), ("qsgd", 16)):
        _quant_check(gc, L, np.zeros(137, F32), None, mode, s, seed=0, it=0)


def _extreme_tensors():
    """Tensors whose squares (or sums) leave the fp32 range, or whose
    quotients by the scale are tiny: huge values (norm above 2^125), values
    near the subnormal range, values spread over 2^-149 .. 2^10, values
    whose squares underflow fp32, zeros of both signs."""
    rng = np.random.default_rng(123)

    def signed(x):
        return np.where(rng.random(x.size) < 0.5, -x, x).astype(F32)
    parts = [
        signed(1e36 * rng.uniform(0.5, 1.0, 5001)),             # ||g|| ~ 5e37 > 2^125
        signed(1e-40 * rng.uniform(0.5, 1.0, 3000)),            # subnormal values, norm < 2^-125
        signed(np.exp2(rng.uniform(-149, 10, 20000))),          # quotients down to the subnormal range
        signed(1e-25 * rng.uniform(0.5, 1.0, 7000)),            # squares underflow fp32
        np.zeros(1, F32),
        np.concatenate([np.asarray([0.0, -0.0, 1e-45, -1e-45], F32), signed(rng.uniform(0, 1, 29))]),
        signed(1e30 * rng.standard_t(3, 4100)),                 # heavy tail, squares overflow fp32
    ]
    return [p.size for p in parts], np.concatenate(parts).astype(F32)


def test_dense_extreme_magnitudes(gc):
    """Scales and codes stay exact-to-the-oracle where fp32 squares or sums
    of the values would overflow or underflow, and where the quotient by the
    scale leaves the range of the fast division."""
    sizes, g = _extreme_tensors()
    L = _layout(gc, sizes, k=[0] * len(sizes))
    for mode, s in (("qsgd", 16), ("int8", 0), ("qsgd", 1)):
        _quant_check(gc, L, g, None, mode, s, seed=13, it=0)
    _quant_check(gc, L, g, np.zeros_like(g), "qsgd", 16, seed=13, it=1)
    _sign_check(gc, L, g, np.zeros_like(g))
    # single-pass sign: the same mean |acc| and bits
    ws = gc.alloc_workspace(L, gc.GC_OP_SIGN)
    bits = torch.empty(L.words, dtype=torch.int32, device="cuda")
    mu = torch.empty(L.T, dtype=torch.float32, device="cuda")
    gc.sign_compress_lazy(L, torch.from_numpy(g).cuda(), torch.zeros(L.numel, device="cuda"), None, bits, mu, ws)
    gb, gm = bits.cpu().numpy().view(np.uint32), mu.cpu().numpy()
    woff = workloads.prefix((np.diff(L.off) + 31) // 32)
    for t in range(L.T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        _, mu_ref = oracle.sign_tensor(g[a:b], np.zeros(b - a, F32))
        assert abs(float(gm[t]) - mu_ref) <= REL_TOL * abs(mu_ref), f"lazy sign tensor {t}: mean |acc|"
        rb, _ = oracle.sign_tensor(g[a:b], np.zeros(b - a, F32), mu_given=float(gm[t]))
        assert np.array_equal(gb[woff[t]:woff[t + 1]], rb), f"lazy sign tensor {t}: bits"


def test_int8_rounding_boundaries(gc):
    """Dense int8 with max |x| = 127, so the scale is exactly 1 and |x| / s is
    |x| itself: integers, values just above and below them, fractions that
    are small multiples of 2^-32, subnormals; codes bit-exact against the
    oracle (the random words decide against exactly these fractions)."""
    rng = np.random.default_rng(77)
    k = rng.integers(0, 127, 2000).astype(np.float64)
    parts = [np.asarray([127.0]), k, k + 2.0 ** -20, k + 0.5, k + (1 - 2.0 ** -17), k + 2.0 ** -23 * 3,
             2.0 ** -32 * rng.integers(1, 4096, 1000), np.exp2(rng.uniform(-149, -126, 500)),
             rng.uniform(0, 127, 3000)]
    g = np.concatenate(parts).astype(F32)
    g = np.where(rng.random(g.size) < 0.5, -g, g).astype(F32)
    g[0] = 127.0
    L = _layout(gc, [g.size], k=[0])
    for it in range(3):
        _quant_check(gc, L, g, None, "int8", 0, seed=21, it=it)


def test_clipping_extreme_magnitudes(gc):
    sizes, g_h = _extreme_tensors()
    L = _layout(gc, sizes, rho=0.01)
    n, K, T = L.numel, L.total_k, L.T
    e_ref = np.zeros(n, F32)
    e = torch.zeros(n, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
    idx = torch.empty(K, dtype=torch.int32, device="cuda")
    val = torch.empty(K, device="cuda")
    norm = torch.empty(T, device="cuda")
    gn = [float(np.linalg.norm(g_h[int(L.off[t]):int(L.off[t + 1])].astype(np.float64))) for t in range(T)]
    cap = np.asarray([0.5 * x for x in gn], F32)
    gc.ef_topk_compress_clipped(L, torch.from_numpy(g_h).cuda(), e, torch.from_numpy(cap).cuda(), norm,
                                idx, val, None, None, 8, 0, gc.GC_EF, ws)
    assert gc.get_device_status(ws).error_bits == 0
    gi, gv, gno = idx.cpu().numpy(), val.cpu().numpy(), norm.cpu().numpy()
    for t in range(T):
        a, b = int(L.off[t]), int(L.off[t + 1])
        ka, kb = int(L.koff[t]), int(L.koff[t + 1])
        _, _, _, _, nref = oracle.clip_topk_tensor(g_h[a:b], e_ref[a:b].copy(), int(L.k[t]), float(cap[t]),
                                                   base=a, int8=False, seed=8, it=0)
        assert abs(float(gno[t]) - nref) <= 1e-6 * nref, f"tensor {t}: norm"
        ri, rv, _, _, _ = oracle.clip_topk_tensor(g_h[a:b], e_ref[a:b], int(L.k[t]), float(cap[t]), base=a,
                                                  int8=False, seed=8, it=0, norm_given=float(gno[t]))
        assert np.array_equal(gi[ka:kb], ri), f"tensor {t}: indices"
        assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"tensor {t}: values"
    assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref)), "residual"


# ----------------------------------------------------------------------------- receivers

@pytest.mark.parametrize("int8", [False, True])
def test_sparse_decompress(gc, int8):
    sizes = [4097, 1, 33, 100_003, 6, 64, 250_000]
    k = [41, 1, 33, 1000, 0, 3, 2500]
    lay = workloads.Layout("t", sizes)
    L = _layout(gc, sizes, k=k)
    W = 5
    kk = np.asarray(k, np.int64)
    payloads = [workloads.make_sparse_payload(lay, kk, w, device="cpu", cfg=0, int8=int8) for w in range(W)]
    base = _grad(L.numel, 7).numpy()
    out = torch.from_numpy(base).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    idx = [p[0].cuda() for p in payloads]
    if int8:
        gc.sparse_decompress_accumulate(L, idx, None, [p[2].cuda() for p in payloads],
                                        [p[3].cuda() for p in payloads], out, ws)
    else:
        gc.sparse_decompress_accumulate(L, idx, [p[1].cuda() for p in payloads], None, None, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    ref = base.copy()
    if int8:
        oracle.sparse_accumulate(L.off, L.koff, [p[0].numpy() for p in payloads], None,
                                 [p[2].numpy() for p in payloads], [p[3].numpy() for p in payloads], ref)
    else:
        oracle.sparse_accumulate(L.off, L.koff, [p[0].numpy() for p in payloads],
                                 [p[1].numpy() for p in payloads], None, None, ref)
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref))


def _receiver_ref(L, kind, pays, base, s_levels=16):
    ref = base.copy()
    idx = [p["idx"].cpu().numpy() for p in pays]
    if kind == "f32":
        oracle.sparse_accumulate(L.off, L.koff, idx, [p["val"].cpu().numpy() for p in pays], None, None, ref)
    else:
        oracle.sparse_accumulate_quantized(L.off, L.koff, kind, idx,
                                           [p["q"].cpu().numpy() for p in pays] if kind != "sign" else None,
                                           [p["bits"].cpu().numpy().view(np.uint32) for p in pays]
                                           if kind == "sign" else None,
                                           [p["scale"].cpu().numpy() for p in pays], ref, s_levels)
    return ref


def _receiver_run(gc, L, kind, pays, out, ws, s_levels=16):
    idx = [p["idx"] for p in pays]
    if kind == "f32":
        gc.sparse_decompress_accumulate(L, idx, [p["val"] for p in pays], None, None, out, ws)
    else:
        k = {"int8": gc.GC_KEPT_INT8, "qsgd": gc.GC_KEPT_QSGD, "sign": gc.GC_KEPT_SIGN}[kind]
        gc.sparse_decompress_accumulate_quantized(L, k, s_levels, idx,
                                                  [p["q"] for p in pays] if kind != "sign" else None,
                                                  [p["bits"] for p in pays] if kind == "sign" else None,
                                                  [p["scale"] for p in pays], out, ws)


def _random_payload(L, rng, kind, clustered=False):
    """One worker's payload: ascending distinct local indices per tensor (a
    uniform subset, or the first k_t indices when clustered), values of the
    given kind."""
    idx = []
    for t in range(L.T):
        n, k = int(L.off[t + 1] - L.off[t]), int(L.k[t])
        sel = np.arange(k) if clustered else np.sort(rng.choice(n, size=k, replace=False))
        idx.append(sel.astype(np.int32))
    p = {"idx": torch.from_numpy(np.concatenate(idx)).cuda()}
    K = L.total_k
    p["val"] = torch.from_numpy((rng.standard_normal(K) * 1e-3).astype(F32)).cuda()
    p["q"] = torch.from_numpy(rng.integers(-16 if kind == "qsgd" else -127, 17 if kind == "qsgd" else 128,
                                           K).astype(np.int8)).cuda()
    p["bits"] = torch.from_numpy(rng.integers(0, 2 ** 32, max(L.kept_words, 1), dtype=np.uint64)
                                 .astype(np.uint32).view(np.int32)).cuda()
    p["scale"] = torch.from_numpy(rng.uniform(1e-4, 1e-2, L.T).astype(F32)).cuda()
    return p


@pytest.mark.parametrize("kind", ["f32", "int8", "qsgd", "sign"])
@pytest.mark.parametrize("W", [1, 3, 8, 11])
def test_sparse_receiver_merged_windows(gc, kind, W):
    """Workers merged per window (W = 11 takes two launch groups), densities
    from one entry per tensor to k = n, tensors with k = 0, misaligned
    starts; bit-exact against the oracle's sequential worker loop."""
    sizes = [4097, 1, 33, 100_003, 6, 64, 250_000, 5000]
    k = [41, 1, 33, 1000, 0, 64, 2500, 5000]
    L = _layout(gc, sizes, k=k)
    rng = np.random.default_rng(100 + W)
    pays = [_random_payload(L, rng, kind) for _ in range(W)]
    base = _grad(L.numel, 7).numpy()
    out = torch.from_numpy(base).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    _receiver_run(gc, L, kind, pays, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(_receiver_ref(L, kind, pays, base)))


@pytest.mark.parametrize("kind", ["f32", "sign"])
def test_sparse_receiver_clustered_indices(gc, kind):
    """Every worker sends the same first k_t indices: a few windows hold all
    entries, and every element gets W contributions, which must still be
    added in worker order."""
    sizes = [300_000, 20_000]
    L = _layout(gc, sizes, k=[3000, 200])
    rng = np.random.default_rng(5)
    pays = [_random_payload(L, rng, kind, clustered=True) for _ in range(8)]
    base = _grad(L.numel, 9).numpy()
    out = torch.from_numpy(base).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    _receiver_run(gc, L, kind, pays, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(_receiver_ref(L, kind, pays, base)))


def test_sparse_receiver_subnormal_sums_are_ieee(gc):
    """The window pass adds with L2 atomics, whose hardware add flushes
    subnormals; sums with subnormal operands or results must still equal the
    IEEE sums of the oracle (base values, addends and cancelling pairs in the
    subnormal range)."""
    n = 4096
    L = _layout(gc, [n], k=[n])
    rng = np.random.default_rng(12)
    tiny = np.float32(2.0 ** -140)
    base = (rng.integers(-1000, 1000, n) * tiny).astype(F32)          # subnormal or zero
    base[::5] = (rng.standard_normal(base[::5].size) * 1e-38).astype(F32)
    idx = torch.arange(n, dtype=torch.int32, device="cuda")
    v0 = (rng.integers(-1000, 1000, n) * tiny).astype(F32)            # subnormal addends
    v1 = (-base.astype(np.float64) - v0.astype(np.float64) + rng.integers(-3, 4, n) * 2.0 ** -149).astype(F32)
    v2 = (rng.standard_normal(n) * 1e-3).astype(F32)                  # normal
    vals = [torch.from_numpy(v).cuda() for v in (v0, v1, v2)]
    out = torch.from_numpy(base.copy()).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    gc.sparse_decompress_accumulate(L, [idx, idx, idx], vals, None, None, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    ref = base.copy()
    oracle.sparse_accumulate(L.off, L.koff, [np.arange(n, dtype=np.int32)] * 3, [v0, v1, v2], None, None, ref)
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref))


def test_sparse_receiver_flags_unsorted_indices(gc):
    """Indices out of ascending order are reported; entries inside their
    tensor's window are still added (here the tensor is one window)."""
    L = _layout(gc, [4096], k=[4])
    idx = torch.tensor([7, 3, 900, 5], dtype=torch.int32, device="cuda")     # one window, not ascending
    val = torch.tensor([1.0, 2.0, 4.0, 8.0], device="cuda")
    out = torch.zeros(4096, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    gc.sparse_decompress_accumulate(L, [idx, idx], [val, val], None, None, out, ws)
    d = gc.get_device_status(ws, raise_on_error=False)
    assert d.error_bits & gc.GC_DIAG_INDEX_ORDER and not d.error_bits & gc.GC_DIAG_INDEX_RANGE
    o = out.cpu().numpy()
    assert o[7] == 2.0 and o[3] == 4.0 and o[900] == 8.0 and o[5] == 16.0 and o.sum() == 30.0


def test_sparse_decompress_flags_bad_index(gc):
    L = _layout(gc, [10, 20], k=[1, 1])
    out = torch.zeros(30, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    idx = torch.tensor([3, 25], dtype=torch.int32, device="cuda")        # 25 >= n_1 = 20
    val = torch.tensor([1.0, 2.0], device="cuda")
    gc.sparse_decompress_accumulate(L, [idx], [val], None, None, out, ws)
    d = gc.get_device_status(ws, raise_on_error=False)
    assert d.error_bits & gc.GC_DIAG_INDEX_RANGE
    o = out.cpu().numpy()
    assert o[3] == 1.0 and o.sum() == 1.0


@pytest.mark.parametrize("kind", ["sign", "int8", "qsgd"])
def test_dense_decompress(gc, kind):
    sizes = [4097, 1, 33, 100_003, 6, 64, 31]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n, W, s = L.numel, 3, 16
    rng = np.random.default_rng(2)
    base = _grad(n, 8).numpy()
    out = torch.from_numpy(base).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    datas, scales = [], []
    for w in range(W):
        if kind == "sign":
            datas.append(rng.integers(0, 2 ** 32, L.words, dtype=np.uint64).astype(np.uint32))
        elif kind == "int8":
            datas.append(rng.integers(-127, 128, n).astype(np.int8))
        else:
            datas.append(rng.integers(-s, s + 1, n).astype(np.int8))
        scales.append(rng.uniform(1e-4, 1e-2, L.T).astype(F32))
    kd = {"sign": gc.GC_DENSE_SIGN, "int8": gc.GC_DENSE_INT8, "qsgd": gc.GC_DENSE_QSGD}[kind]
    dd = [torch.from_numpy(d.view(np.int32) if kind == "sign" else d).cuda() for d in datas]
    gc.dense_decompress_accumulate(L, kd, s, dd, [torch.from_numpy(x).cuda() for x in scales], out, ws)
    ref = base.copy()
    woff = workloads.prefix((np.diff(L.off) + 31) // 32)
    for w in range(W):
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            if kind == "sign":
                oracle.sign_decode_accumulate(datas[w][woff[t]:woff[t + 1]], scales[w][t], ref[a:b])
            else:
                oracle.codes_decode_accumulate(datas[w][a:b], scales[w][t], kind, ref[a:b], s)
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref))


@pytest.mark.parametrize("path", PATHS)
def test_layout_mismatch_is_reported_not_run(gc, path):
    flags = gc.GC_EF | (gc.GC_MULTI_KERNEL if path == "pipeline" else 0)
    sizes = [1000, 2000]
    L = _layout(gc, sizes, k=[10, 20])
    bad = _layout(gc, [1000, 3000], k=[10, 20])          # device copy disagrees with the host mirror
    L._dev_off.copy_(bad._dev_off)
    g = torch.zeros(3000, device="cuda")
    e = torch.zeros(3000, device="cuda")
    idx = torch.full((30,), -7, dtype=torch.int32, device="cuda")
    val = torch.zeros(30, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    gc.ef_topk_compress(L, g, e, idx, val, None, None, 0, 0, flags, ws)
    d = gc.get_device_status(ws, raise_on_error=False)
    assert d.error_bits & gc.GC_DIAG_LAYOUT_MISMATCH
    assert (idx.cpu() == -7).all() and not bool(e.any())


# ----------------------------------------------------------------------------- lazy residual

@pytest.mark.parametrize("name", ["misaligned", "many_small", "medium", "flat"])
@pytest.mark.parametrize("flags_name", ["ef", "ef_int8", "ef_int8_exact"])
def test_topk_lazy_residual(gc, name, flags_name):
    """Payloads of gc_ef_topk_compress_lazy equal the oracle's at every step, and
    materializing a copy of (e, rd) gives the oracle's residual at every step."""
    sizes = [1 << 20] if name == "flat" else LAYOUTS[name]
    flags = {"ef": 0, "ef_int8": gc.GC_INT8, "ef_int8_exact": gc.GC_INT8 | gc.GC_FORCE_EXACT}[flags_name]
    k = workloads.k_per_tensor(sizes, 0.01)
    if len(sizes) > 2:
        k[0] = sizes[0]
        k[-1] = 0
    L = _layout(gc, sizes, k=k)
    n, K = L.numel, L.total_k
    int8 = bool(flags & gc.GC_INT8)
    e_ref = (np.random.default_rng(4).standard_normal(n) * 1e-4).astype(F32)
    e = torch.from_numpy(e_ref).cuda()
    rd = gc.alloc_residual_desc(L)
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF | flags)
    idx = torch.empty(K, dtype=torch.int32, device="cuda")
    val = torch.empty(K, dtype=torch.float32, device="cuda")
    q = torch.empty(K, dtype=torch.int8, device="cuda") if int8 else None
    sc = torch.empty(L.T, dtype=torch.float32, device="cuda") if int8 else None
    for it in range(4):
        g_h = _grad(n, 200 + it).numpy()
        gc.ef_topk_compress_lazy(L, torch.from_numpy(g_h).cuda(), e, rd, idx, val, q, sc, 3, it, flags, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gi, gv = idx.cpu().numpy(), val.cpu().numpy()
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            ri, rv, rq, rs = oracle.ef_topk_tensor(g_h[a:b], e_ref[a:b], int(L.k[t]), base=a, int8=int8,
                                                   seed=3, it=it)
            assert np.array_equal(gi[ka:kb], ri), f"it {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"it {it} tensor {t}: values"
            if int8:
                assert np.array_equal(q.cpu().numpy()[ka:kb], rq), f"it {it} tensor {t}: codes"
                assert sc.cpu().numpy()[t] == rs
        e_copy, rd_copy = e.clone(), rd.clone()
        gc.ef_residual_materialize(L, e_copy, rd_copy)
        assert np.array_equal(_bits(e_copy.cpu().numpy()), _bits(e_ref)), f"it {it}: materialized residual"
        assert int(rd_copy.sum()) == 0
    # switching back to the eager entry point after materializing continues the same sequence
    gc.ef_residual_materialize(L, e, rd)
    g_h = _grad(n, 300).numpy()
    assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref))
    _topk_check(gc, L, g_h, e_ref, gc.GC_EF | flags, seed=3, it=9)


@pytest.mark.parametrize("name", ["misaligned_sign", "many_small", "medium"])
def test_sign_lazy_residual(gc, name):
    """Single-pass sign compression: bits and mean |acc| as the oracle's at every
    step, and the materialized pending residual equals the oracle's residual."""
    sizes = {"misaligned_sign": [4097, 1, 33, 100_003, 6, 64, 31, 32, 250_000]}.get(name) or LAYOUTS[name]
    L = _layout(gc, sizes, k=[0] * len(sizes))
    n = L.numel
    woff = workloads.prefix((np.diff(L.off) + 31) // 32)
    e_ref = (np.random.default_rng(6).standard_normal(n) * 1e-4).astype(F32)
    e = torch.from_numpy(e_ref).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_SIGN)
    bits = torch.empty(L.words, dtype=torch.int32, device="cuda")
    mu = torch.empty(L.T, dtype=torch.float32, device="cuda")
    prev = None
    for it in range(3):
        g_h = _grad(n, 400 + it).numpy()
        g_h[::13] = -0.0
        gc.sign_compress_lazy(L, torch.from_numpy(g_h).cuda(), e, prev, bits, mu, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gb, gm = bits.cpu().numpy().view(np.uint32), mu.cpu().numpy()
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            _, mu_ref = oracle.sign_tensor(g_h[a:b], e_ref[a:b].copy())
            assert abs(float(gm[t]) - mu_ref) <= REL_TOL * abs(mu_ref), f"it {it} tensor {t}: mean |acc|"
            rb, _ = oracle.sign_tensor(g_h[a:b], e_ref[a:b], mu_given=float(gm[t]))
            assert np.array_equal(gb[woff[t]:woff[t + 1]], rb), f"it {it} tensor {t}: bits"
        e_copy = e.clone()
        gc.sign_residual_materialize(L, e_copy, mu)
        assert np.array_equal(_bits(e_copy.cpu().numpy()), _bits(e_ref)), f"it {it}: residual"
        prev = mu.clone()


# ----------------------------------------------------------------------------- threshold

@pytest.mark.parametrize("flags_name", ["ef", "ef_int8", "noef", "ef_exact"])
def test_threshold_layouts(gc, flags_name):
    flags = {"ef": gc.GC_EF, "ef_int8": gc.GC_EF | gc.GC_INT8, "noef": 0,
             "ef_exact": gc.GC_EF | gc.GC_FORCE_EXACT}[flags_name]
    sizes = [4097, 1, 33, 100_003, 6, 70_000, 300_000, 500_000]
    kmax = [60, 1, 33, 500, 3, 2000, 3000, 500]
    L = _layout(gc, sizes, k=kmax)
    n, K, T = L.numel, L.total_k, L.T
    int8 = bool(flags & gc.GC_INT8)
    # thresholds: some tensors pass fewer than k_t, some more, tau = 0 and tau = inf
    tau_h = np.asarray([2e-3, 0.0, np.inf, 2e-2, 0.0, 3e-3, 1e-2, 1e-3], F32)   # last: ~40% pass, cap 0.1%
    tau = torch.from_numpy(tau_h).cuda()
    e_ref = (np.random.default_rng(9).standard_normal(n) * 1e-4).astype(F32) if flags & gc.GC_EF else None
    e = torch.from_numpy(e_ref).cuda() if e_ref is not None else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    cnt = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    idx = torch.full((K,), -1, dtype=torch.int32, device="cuda")
    val = torch.zeros(K, device="cuda")
    q = torch.zeros(K, dtype=torch.int8, device="cuda") if int8 else None
    sc = torch.zeros(T, device="cuda") if int8 else None
    counts_seen = set()
    for it in range(2):
        g_h = _grad(n, 500 + it).numpy()
        gc.ef_threshold_compress(L, torch.from_numpy(g_h).cuda(), e, tau, cnt, idx, val, q, sc, 7, it, flags, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gcnt, gi, gv = cnt.cpu().numpy(), idx.cpu().numpy(), val.cpu().numpy()
        for t in range(T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka = int(L.koff[t])
            et = e_ref[a:b] if e_ref is not None else None
            ri, rv, rq, rs, c = oracle.threshold_tensor(g_h[a:b], et, int(kmax[t]), float(tau_h[t]), base=a,
                                                        int8=int8, seed=7, it=it)
            assert gcnt[t] == c, f"it {it} tensor {t}: count {gcnt[t]} vs {c}"
            counts_seen.add((t, c < kmax[t]))
            assert np.array_equal(gi[ka:ka + c], ri), f"it {it} tensor {t}: indices"
            if int8:
                assert np.array_equal(q.cpu().numpy()[ka:ka + c], rq)
                assert sc.cpu().numpy()[t] == (rs if c else 0.0)
            assert np.array_equal(_bits(gv[ka:ka + c]), _bits(rv)), f"it {it} tensor {t}: values"
        if e is not None:
            assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref))
    assert {c for _, c in counts_seen} == {True, False}     # both regimes exercised


def test_threshold_rejects_negative_tau(gc):
    L = _layout(gc, [100, 200], k=[5, 5])
    tau = torch.tensor([-1.0, 1e-3], device="cuda")
    cnt = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    idx = torch.zeros(10, dtype=torch.int32, device="cuda")
    val = torch.zeros(10, device="cuda")
    g = torch.from_numpy(_grad(300, 1).numpy()).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, 0)
    gc.ef_threshold_compress(L, g, None, tau, cnt, idx, val, None, None, 0, 0, 0, ws)
    d = gc.get_device_status(ws, raise_on_error=False)
    assert d.error_bits & gc.GC_DIAG_BAD_THRESHOLD
    assert int(cnt[0]) == 0


# ----------------------------------------------------------------------------- local clipping

@pytest.mark.parametrize("flags_name", ["ef", "ef_int8", "ef_exact"])
def test_clipped_topk_layouts(gc, flags_name):
    flags = {"ef": gc.GC_EF, "ef_int8": gc.GC_EF | gc.GC_INT8, "ef_exact": gc.GC_EF | gc.GC_FORCE_EXACT}[flags_name]
    sizes = [4097, 1, 33, 100_003, 6, 70_000, 300_000]
    L = _layout(gc, sizes, rho=0.01)
    n, K, T = L.numel, L.total_k, L.T
    int8 = bool(flags & gc.GC_INT8)
    e_ref = (np.random.default_rng(10).standard_normal(n) * 1e-4).astype(F32)
    e = torch.from_numpy(e_ref).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    idx = torch.empty(K, dtype=torch.int32, device="cuda")
    val = torch.empty(K, device="cuda")
    q = torch.empty(K, dtype=torch.int8, device="cuda") if int8 else None
    sc = torch.empty(T, device="cuda") if int8 else None
    norm = torch.empty(T, device="cuda")
    for it in range(2):
        g_h = _grad(n, 600 + it).numpy()
        gn = [float(np.linalg.norm(g_h[int(L.off[t]):int(L.off[t + 1])].astype(np.float64))) for t in range(T)]
        # clip some tensors hard, some mildly, one to zero, leave others alone
        cap = np.asarray([0.5 * gn[0], 10 * gn[1], 0.0, 0.9 * gn[3], np.inf, 0.1 * gn[5], 2 * gn[6]], F32)
        gc.ef_topk_compress_clipped(L, torch.from_numpy(g_h).cuda(), e, torch.from_numpy(cap).cuda(), norm,
                                    idx, val, q, sc, 8, it, flags, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gi, gv, gno = idx.cpu().numpy(), val.cpu().numpy(), norm.cpu().numpy()
        for t in range(T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            _, _, _, _, nref = oracle.clip_topk_tensor(g_h[a:b], e_ref[a:b].copy(), int(L.k[t]), float(cap[t]),
                                                       base=a, int8=int8, seed=8, it=it)
            assert abs(float(gno[t]) - nref) <= 1e-6 * nref, f"it {it} tensor {t}: norm"
            ri, rv, rq, rs, _ = oracle.clip_topk_tensor(g_h[a:b], e_ref[a:b], int(L.k[t]), float(cap[t]), base=a,
                                                        int8=int8, seed=8, it=it, norm_given=float(gno[t]))
            assert np.array_equal(gi[ka:kb], ri), f"it {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"it {it} tensor {t}: values"
            if int8:
                assert np.array_equal(q.cpu().numpy()[ka:kb], rq) and sc.cpu().numpy()[t] == rs
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_ref)), f"it {it}: residual"


# ----------------------------------------------------------------------------- PowerSGD

PS_SHAPES = [(1, 1), (3, 5), (17, 33), (64, 4096), (300, 1024), (1024, 1000), (2000, 257)]


@pytest.mark.parametrize("rank", [1, 2, 4])
def test_powersgd_steps(gc, rank):
    """Fixed-order reductions on the GPU vs fp64 in the oracle: P_raw = MQ and
    Q = M^T P within 2e-6 of sum |M||.| (compensated fp32 partials), the
    orthonormalized P within a Gram-Schmidt error bound given the GPU's
    P_raw (see _check_orthonormalized), and the residual
    E = M - P Q^T bit-exact given the GPU's P and Q; three warm-started calls."""
    _powersgd_check(gc, rank, PS_SHAPES, 40 + rank, iters=3)


@pytest.mark.parametrize("rank", [1, 2, 4])
def test_powersgd_lazy_matches_eager(gc, rank):
    """The pending-residual entry point against gc_powersgd_compress on the
    same inputs, four chained calls: P and Q bit-identical every call, and
    the materialized residual (on a copy) bit-identical to the eager one.
    The eager path is checked against the oracle by the tests above."""
    shapes = [(1, 1), (17, 33), (300, 1024), (2000, 257), (9000, 16)]
    rng = np.random.default_rng(70 + rank)
    starts, pos = [], 0
    for i, (m, n) in enumerate(shapes):
        pos += 3 * (i % 2)
        starts.append(pos)
        pos += m * n
    N = pos
    ml = gc.MatrixLayout(starts, [a for a, _ in shapes], [b for _, b in shapes], device="cuda")
    Msum, Nsum = int(ml.poff[-1]), int(ml.qoff[-1])
    e0 = torch.from_numpy((0.1 * rng.standard_normal(N)).astype(F32)).cuda()
    q0 = torch.from_numpy(rng.standard_normal(Nsum * rank).astype(F32)).cuda()
    e_eager, q_eager = e0.clone(), q0.clone()
    e_lazy, q_lazy = e0.clone(), q0.clone()
    p_eager = torch.empty(Msum * rank, device="cuda")
    p_lazy = [torch.empty(Msum * rank, device="cuda") for _ in range(2)]
    ws = gc.powersgd_workspace(ml, rank)
    for it in range(4):
        g = torch.from_numpy(rng.standard_normal(N).astype(F32)).cuda()
        gc.powersgd_compress(ml, rank, g, e_eager, q_eager, p_eager, None, ws)
        cur, prev = p_lazy[it % 2], (p_lazy[(it - 1) % 2] if it else None)
        gc.powersgd_compress_lazy(ml, rank, g, e_lazy, q_lazy, cur, prev, None, ws)
        assert gc.get_device_status(ws).error_bits == 0
        assert torch.equal(cur.view(torch.int32), p_eager.view(torch.int32)), f"call {it}: P"
        assert torch.equal(q_lazy.view(torch.int32), q_eager.view(torch.int32)), f"call {it}: Q"
        e_mat = e_lazy.clone()
        gc.powersgd_residual_materialize(ml, rank, e_mat, cur, q_lazy, ws)
        assert torch.equal(e_mat.view(torch.int32), e_eager.view(torch.int32)), f"call {it}: residual"
    with pytest.raises(gc.GCError):
        gc.powersgd_compress_lazy(ml, rank, g, e_lazy, q_lazy, cur, cur, None, ws)


@pytest.mark.parametrize("rank", [1, 4])
def test_powersgd_tall_matrices(gc, rank):
    """Matrices taller than 8192 rows (Gram-Schmidt on a cluster of CTAs),
    between small ones, one with a misaligned start."""
    _powersgd_check(gc, rank, [(5, 7), (9000, 16), (16385, 5), (30522, 12), (100, 3)], 60 + rank, iters=2)


U32 = 2.0 ** -24      # unit roundoff of fp32


def _check_orthonormalized(p_gpu, p_ref, p_raw, what):
    """Modified Gram-Schmidt of the same P_raw on both sides.  The dot products
    and norms agree to about one fp32 ulp (compensated sums on the GPU, fp64 in
    the oracle) and the element updates are the same fp32 operations, so column
    k differs by a few ulps of its elements, amplified by the cancellation of
    each projection step: rho_j = ||P_raw_j|| / |R_jj|, with R_jj the part of
    column j outside the span of the columns before it (numpy's QR).  The bound
    is 32 (k + 1) u sum_{j <= k} rho_j on the 2-norm of column k's difference
    (columns have unit norm), u = 2^-24; and the GPU's columns are orthonormal
    to 32 r u kappa(P_raw), the loss of orthogonality of modified
    Gram-Schmidt.  Rank-deficient P_raw (R_jj = 0) has no stable direction
    from column j on; those columns are not compared."""
    m, r = p_raw.shape
    raw = p_raw.astype(np.float64)
    rdiag = np.abs(np.diag(np.linalg.qr(raw, mode="r"))) if m >= 1 else np.zeros(r)
    rdiag = np.concatenate([rdiag, np.zeros(r - rdiag.size)])
    cnorm = np.linalg.norm(raw, axis=0)
    ok_cols = 0
    rho_sum = 0.0
    for k in range(r):
        if rdiag[k] <= 1e-6 * max(cnorm[k], 1e-300):
            break                      # column k is (nearly) in the span of the previous ones
        rho_sum += cnorm[k] / rdiag[k]
        diff = np.linalg.norm(p_gpu[:, k].astype(np.float64) - p_ref[:, k].astype(np.float64))
        bound = 32 * (k + 1) * U32 * rho_sum
        assert diff <= bound, f"{what}: orthonormalized column {k} differs by {diff:.3g} > {bound:.3g}"
        ok_cols += 1
    if ok_cols:
        sv = np.linalg.svd(raw[:, :ok_cols], compute_uv=False)
        kappa = sv[0] / sv[-1]
        pk = p_gpu[:, :ok_cols].astype(np.float64)
        gram = pk.T @ pk - np.eye(ok_cols)
        assert np.abs(gram).max() <= 32 * r * U32 * kappa, f"{what}: P^T P - I = {np.abs(gram).max():.3g}"


def _powersgd_check(gc, rank, shapes, seed, iters):
    PS_SHAPES = shapes
    rng = np.random.default_rng(seed)
    starts, pos = [], 0
    for i, (m, n) in enumerate(PS_SHAPES):
        pos += 3 * (i % 2)                      # gaps: some matrices start misaligned
        starts.append(pos)
        pos += m * n
    N = pos
    ml = gc.MatrixLayout(starts, [s[0] for s in PS_SHAPES], [s[1] for s in PS_SHAPES], device="cuda")
    Msum, Nsum = int(ml.poff[-1]), int(ml.qoff[-1])
    e_h = (0.1 * rng.standard_normal(N)).astype(F32)
    q_h = rng.standard_normal(Nsum * rank).astype(F32)
    e, q = torch.from_numpy(e_h).cuda(), torch.from_numpy(q_h).cuda()
    p = torch.empty(Msum * rank, device="cuda")
    p_raw = torch.empty(Msum * rank, device="cuda")
    ws = gc.powersgd_workspace(ml, rank)
    for it in range(iters):
        g_h = rng.standard_normal(N).astype(F32)
        gc.powersgd_compress(ml, rank, torch.from_numpy(g_h).cuda(), e, q, p, p_raw, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gp, gpr, gq, ge = p.cpu().numpy(), p_raw.cpu().numpy(), q.cpu().numpy(), e.cpu().numpy()
        for t, (m, n) in enumerate(PS_SHAPES):
            a = starts[t]
            sl = slice(a, a + m * n)
            ps_ = slice(int(ml.poff[t]) * rank, int(ml.poff[t + 1]) * rank)
            qs_ = slice(int(ml.qoff[t]) * rank, int(ml.qoff[t + 1]) * rank)
            Mh = (g_h[sl] + e_h[sl]).reshape(m, n)
            q_in = q_h[qs_].reshape(n, rank)
            # step 1: P_raw
            e1, q1 = e_h[sl].reshape(m, n).copy(), q_in.copy()
            _, pr_ref = oracle.powersgd_tensor(g_h[sl].reshape(m, n), e1, q1, rank)
            bound = 2e-6 * (np.abs(Mh).astype(np.float64) @ np.abs(q_in).astype(np.float64)) + 1e-30
            assert np.all(np.abs(gpr[ps_].reshape(m, rank) - pr_ref) <= bound), f"it {it} matrix {t}: P = MQ"
            # step 2: Gram-Schmidt given the GPU's P_raw
            e2, q2 = e_h[sl].reshape(m, n).copy(), q_in.copy()
            p_ref, _ = oracle.powersgd_tensor(g_h[sl].reshape(m, n), e2, q2, rank,
                                              p_raw_given=gpr[ps_].reshape(m, rank))
            _check_orthonormalized(gp[ps_].reshape(m, rank), p_ref, gpr[ps_].reshape(m, rank), f"it {it} matrix {t}")
            # step 3: Q given the GPU's P
            e3, q3 = e_h[sl].reshape(m, n).copy(), q_in.copy()
            oracle.powersgd_tensor(g_h[sl].reshape(m, n), e3, q3, rank, p_given=gp[ps_].reshape(m, rank))
            bound = 2e-6 * (np.abs(Mh).T.astype(np.float64) @ np.abs(gp[ps_].reshape(m, rank)).astype(np.float64)) + 1e-30
            assert np.all(np.abs(gq[qs_].reshape(n, rank) - q3) <= bound), f"it {it} matrix {t}: Q = M^T P"
            # step 4: residual given the GPU's P and Q, bit-exact
            e4, q4 = e_h[sl].reshape(m, n).copy(), q_in.copy()
            oracle.powersgd_tensor(g_h[sl].reshape(m, n), e4, q4, rank, p_given=gp[ps_].reshape(m, rank),
                                   q_given=gq[qs_].reshape(n, rank))
            assert np.array_equal(_bits(ge[sl]), _bits(e4.ravel())), f"it {it} matrix {t}: residual"
        e_h = ge.copy()           # both sides continue from the same state
        q_h = gq.copy()
    # receiver: out += P Q^T, bit-exact
    base = rng.standard_normal(N).astype(F32)
    out = torch.from_numpy(base).cuda()
    gc.powersgd_decompress_accumulate(ml, rank, p, q, out, ws)
    ref = base.copy()
    for t, (m, n) in enumerate(PS_SHAPES):
        sl = slice(starts[t], starts[t] + m * n)
        blk = ref[sl].reshape(m, n).copy()
        oracle.powersgd_decode_accumulate(gp[int(ml.poff[t]) * rank:int(ml.poff[t + 1]) * rank].reshape(m, rank),
                                          gq[int(ml.qoff[t]) * rank:int(ml.qoff[t + 1]) * rank].reshape(n, rank), blk)
        ref[sl] = blk.ravel()
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(ref))
