"""Randomized parity: seeded random layouts (1 to 40 tensors, sizes from 1
to ~400K elements, k from 0 to n), mixed value distributions and every
selection flag, GPU against the oracle, EF state carried over two
iterations; the quantizers of the kept values and the sparse receiver over
the same kind of layouts.  Complements the fixed cases of
test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import (F32, _bits, _kept_quant_check, _random_payload, _receiver_ref, _receiver_run,
                             _topk_check)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _random_case(seed, max_total=1_500_000):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.integers(1, 41))
    sizes = np.maximum(1, np.exp(rng.uniform(0, np.log(400_000), T)).astype(np.int64))
    while sizes.sum() > max_total:
        sizes = np.maximum(1, sizes // 2)
    k = []
    for n in sizes:
        c = rng.integers(0, 7)
        if c == 0:
            k.append(0)
        elif c == 1:
            k.append(min(int(n), 1))
        elif c == 2:
            k.append(int(n))
        else:
            rho = [1e-3, 1e-2, 0.1, 0.5][c - 3]
            k.append(int(min(n, np.ceil(rho * n))))
    n_tot = int(sizes.sum())
    kind = ["t3", "mixed", "ties", "heavy"][seed % 4]
    gen = torch.Generator().manual_seed(seed)

    def grad(it):
        g = torch.empty(n_tot)
        workloads.fill_student_t(g, 3.0, 1e-3, torch.Generator().manual_seed(seed * 100 + it))
        if kind == "ties":
            g = torch.round(g * 2e3) / 2e3
        elif kind == "mixed":
            # tensors at very different scales, some exact zeros
            scales = np.exp(rng.uniform(np.log(1e-20), np.log(1e20), T))
            off = workloads.prefix(sizes)
            for t in range(T):
                g[int(off[t]):int(off[t + 1])] *= float(scales[t])
            g[::97] = 0.0
        elif kind == "heavy":
            g = g * torch.exp(torch.randn(n_tot, generator=gen) * 3.0)
        return g.float().numpy()
    return sizes, np.asarray(k, np.int64), grad


@pytest.mark.parametrize("seed", list(range(8)))
def test_topk_random_layouts(gc, seed):
    sizes, k, grad = _random_case(seed)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    flags = [gc.GC_EF, gc.GC_EF | gc.GC_INT8, 0, gc.GC_EF | gc.GC_FORCE_EXACT,
             gc.GC_EF | gc.GC_INT8 | gc.GC_FORCE_EXACT][seed % 5]
    if seed % 2:
        flags |= gc.GC_MULTI_KERNEL  # odd seeds: the pipeline; even seeds mostly the one-launch path
    e = np.zeros(L.numel, F32) if flags & gc.GC_EF else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(2):
        e, _ = _topk_check(gc, L, grad(it), e, flags, seed=seed, it=it, ws=ws)


@pytest.mark.parametrize("seed", list(range(4)))
def test_randk_random_layouts(gc, seed):
    sizes, k, grad = _random_case(seed + 50)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    flags = [gc.GC_EF | gc.GC_RANDK, gc.GC_RANDK | gc.GC_UNBIASED, gc.GC_RANDK, gc.GC_EF | gc.GC_RANDK][seed]
    e = np.zeros(L.numel, F32) if flags & gc.GC_EF else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(2):
        e, _ = _topk_check(gc, L, grad(it), e, flags, seed=seed, it=it, ws=ws)


@pytest.mark.parametrize("seed", list(range(4)))
def test_momentum_random_layouts(gc, seed):
    sizes, k, grad = _random_case(seed + 80)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    N, K = L.numel, L.total_k
    flags = [0, gc.GC_NO_MASK, gc.GC_INT8, gc.GC_FORCE_EXACT][seed]
    int8 = bool(flags & gc.GC_INT8)
    beta = [0.9, 0.5, 0.99, 0.0][seed]
    u = torch.zeros(N, device="cuda")
    v = torch.zeros(N, device="cuda")
    u_h, v_h = np.zeros(N, F32), np.zeros(N, F32)
    idx = torch.empty(max(K, 1), dtype=torch.int32, device="cuda")
    val = torch.empty(max(K, 1), device="cuda")
    q = torch.empty(max(K, 1), dtype=torch.int8, device="cuda") if int8 else None
    sc = torch.empty(L.T, device="cuda") if int8 else None
    ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM, flags)
    for it in range(2):
        g_h = grad(it)
        gc.ef_topk_compress_momentum(L, torch.from_numpy(g_h).cuda(), u, v, beta, idx, val, q, sc, seed, it,
                                     flags, ws)
        assert gc.get_device_status(ws).error_bits == 0
        gi, gv = idx.cpu().numpy(), val.cpu().numpy()
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            ri, rv, rq, rs = oracle.momentum_topk_tensor(g_h[a:b], u_h[a:b], v_h[a:b], int(L.k[t]), beta,
                                                         base=a, seed=seed, it=it, int8=int8,
                                                         masking=not (flags & gc.GC_NO_MASK))
            assert np.array_equal(gi[ka:kb], ri), f"it {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"it {it} tensor {t}: values"
            if int8:
                assert np.array_equal(q.cpu().numpy()[ka:kb], rq), f"it {it} tensor {t}: codes"
        assert np.array_equal(_bits(u.cpu().numpy()), _bits(u_h)), f"it {it}: u"
        assert np.array_equal(_bits(v.cpu().numpy()), _bits(v_h)), f"it {it}: v"


@pytest.mark.parametrize("seed", list(range(6)))
def test_kept_quantizers_random_layouts(gc, seed):
    sizes, k, grad = _random_case(seed + 120)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    kind = ["qsgd", "sign"][seed % 2]
    flags = [gc.GC_EF, 0, gc.GC_EF | gc.GC_FORCE_EXACT][seed % 3]
    e = np.zeros(L.numel, F32) if flags & gc.GC_EF else None
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    for it in range(2):
        e = _kept_quant_check(gc, L, grad(it), e, kind, flags, seed=seed, it=it, ws=ws,
                              s_levels=[16, 1, 127, 7][seed % 4])


@pytest.mark.parametrize("seed", list(range(4)))
def test_receiver_random_layouts(gc, seed):
    sizes, k, _ = _random_case(seed + 160)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    rng = np.random.default_rng(seed + 170)
    kind = ["f32", "int8", "qsgd", "sign"][seed]
    W = int(rng.integers(1, 11))
    pays = [_random_payload(L, rng, kind) for _ in range(W)]
    base = (rng.standard_normal(L.numel) * 1e-3).astype(F32)
    out = torch.from_numpy(base).cuda()
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    _receiver_run(gc, L, kind, pays, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    assert np.array_equal(_bits(out.cpu().numpy()), _bits(_receiver_ref(L, kind, pays, base)))
