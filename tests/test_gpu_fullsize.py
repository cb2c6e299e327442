"""Parity at the benchmark sizes and iteration counts, through the C ABI, in
the launch configuration bench.py times.

- BERT-large (335,141,888 elements): EF Top-k 0.1% + int8, and + QSGD or
  sign of the kept values, ten iterations with the residual carried, every
  tensor against the oracle every iteration.
- GPT-2-medium (354,823,168 elements): sign + EF, QSGD s = 16 and momentum
  correction Top-k 0.5%, ten iterations each with their state carried, every
  tensor against the oracle every iteration.
- Llama-3-8B (8,030,261,248 elements, 64 GB of g + e): EF Top-k 0.1% + int8,
  ten iterations.  Every iteration, for the whole arena: each tensor's kept
  set is its Top-k (every kept |acc| at least every unkept |acc|, and ties at
  the k-th magnitude kept from the lowest index up), payload order, code
  range, and the EF identity e' = acc off the kept set, e' = acc - q * s on
  it; sampled tensors (the smallest, a k/v projection, a q projection, an MLP
  matrix and the 525M-element embedding) bit-exact against the oracle.  Then
  the receiver with W = 8 workers' payloads: the whole arena against the
  workers' payloads added one worker after another by torch's indexed
  accumulate, and the sampled tensors against the oracle.

The oracle runs on the host cores, one tensor per thread (its C calls
release the interpreter lock).
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32 = np.float32


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _pool_map(fn, items):
    with cf.ThreadPoolExecutor(max_workers=max(1, min(os.cpu_count() or 1, 32))) as ex:
        return list(ex.map(fn, items))


def _check_topk_tensor(L, t, g_h, e_h, gi, gq, gsc, ge, seed, it, int8=True):
    """One tensor's GPU payload (gi, gq, gsc) and residual (ge) against the oracle."""
    a = int(L.off[t])
    e_ref = e_h.copy()
    ri, rv, rq, rs = oracle.ef_topk_tensor(g_h, e_ref, int(L.k[t]), base=a, int8=int8, seed=seed, it=it)
    assert np.array_equal(gi, ri), f"tensor {t}: indices"
    if int8:
        assert np.array_equal(gq, rq), f"tensor {t}: codes"
        assert _bits(np.asarray([gsc], F32))[0] == _bits(np.asarray([rs], F32))[0], f"tensor {t}: scale"
    assert np.array_equal(_bits(ge), _bits(e_ref)), f"tensor {t}: residual"
    return e_ref


def test_bert_large_topk_int8_full(gc):
    lay = workloads.bert_large_layout()
    k = workloads.k_per_tensor(lay.sizes, 0.001)
    L = gc.Layout(lay.off, k, device="cuda")
    T = lay.num_tensors
    flags = gc.GC_EF | gc.GC_INT8
    comp = gc.TopkCompressor(L, flags)
    e = torch.zeros(L.numel, device="cuda")
    e_ref = np.zeros(L.numel, F32)
    for it in range(10):
        g = workloads.make_grad(3, lay, it, device="cuda")
        comp(g, e, seed=3, it=it)
        d = gc.get_device_status(comp.workspace)
        assert d.error_bits == 0
        g_h = g.cpu().numpy()
        gi, gq, gs = comp.idx.cpu().numpy(), comp.q.cpu().numpy(), comp.scale.cpu().numpy()
        ge = e.cpu().numpy()

        def one(t):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            e_ref[a:b] = _check_topk_tensor(L, t, g_h[a:b], e_ref[a:b], gi[ka:kb], gq[ka:kb], float(gs[t]),
                                            ge[a:b], 3, it)
        _pool_map(one, range(T))


def test_gpt2_medium_dense_and_momentum_full(gc):
    lay = workloads.gpt2_medium_layout()
    T, N = lay.num_tensors, lay.numel
    L = gc.Layout(lay.off, workloads.k_per_tensor(lay.sizes, 0.005), device="cuda")
    off = L.off
    woff = workloads.prefix((np.diff(off) + 31) // 32)
    # sign + EF, ten iterations (e starts at zero, carried)
    e = torch.zeros(N, device="cuda")
    e_ref = np.zeros(N, F32)
    bits = torch.empty(L.words, dtype=torch.int32, device="cuda")
    mu = torch.empty(T, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_SIGN)
    for it in range(10):
        g = workloads.make_grad(4, lay, it, device="cuda")
        gc.sign_compress(L, g, e, bits, mu, ws)
        g_h = g.cpu().numpy()
        gb, gm, ge = bits.cpu().numpy().view(np.uint32), mu.cpu().numpy(), e.cpu().numpy()

        def sign_one(t):
            a, b = int(off[t]), int(off[t + 1])
            _, mref = oracle.sign_tensor(g_h[a:b], e_ref[a:b].copy())
            assert abs(float(gm[t]) - mref) <= 1e-6 * mref, f"it {it} sign tensor {t}: mean |acc|"
            et = e_ref[a:b].copy()
            rb, _ = oracle.sign_tensor(g_h[a:b], et, mu_given=float(gm[t]))
            assert np.array_equal(gb[woff[t]:woff[t + 1]], rb), f"it {it} sign tensor {t}: bits"
            assert np.array_equal(_bits(ge[a:b]), _bits(et)), f"it {it} sign tensor {t}: residual"
            e_ref[a:b] = et
        _pool_map(sign_one, range(T))
    # QSGD s = 16, no EF, ten iterations (fresh draws each)
    codes = torch.empty(N, dtype=torch.int8, device="cuda")
    norm = torch.empty(T, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE)
    for it in range(10):
        g = workloads.make_grad(4, lay, it, device="cuda")
        gc.quantize_stochastic(L, g, None, codes, norm, gc.GC_Q_QSGD, 16, 11, it, ws)
        g_h = g.cpu().numpy()
        gcod, gn = codes.cpu().numpy(), norm.cpu().numpy()

        def qsgd_one(t):
            a, b = int(off[t]), int(off[t + 1])
            _, nref = oracle.quantize_tensor(g_h[a:b], None, "qsgd", 16, base=a, seed=11, it=it)
            assert abs(float(gn[t]) - nref) <= 1e-6 * nref, f"it {it} qsgd tensor {t}: norm"
            rc, _ = oracle.quantize_tensor(g_h[a:b], None, "qsgd", 16, base=a, seed=11, it=it,
                                           scale_given=float(gn[t]))
            assert np.array_equal(gcod[a:b], rc), f"it {it} qsgd tensor {t}: codes"
        _pool_map(qsgd_one, range(T))
    # momentum correction Top-k 0.5%, beta 0.9, ten iterations
    u = torch.zeros(N, device="cuda")
    v = torch.zeros(N, device="cuda")
    u_h, v_h = np.zeros(N, F32), np.zeros(N, F32)
    K = L.total_k
    idx = torch.empty(K, dtype=torch.int32, device="cuda")
    val = torch.empty(K, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM)
    for it in range(10):
        g = workloads.make_grad(4, lay, it, device="cuda")
        g_h = g.cpu().numpy()
        gc.ef_topk_compress_momentum(L, g, u, v, 0.9, idx, val, None, None, 4, it, 0, ws)
        gi, gv = idx.cpu().numpy(), val.cpu().numpy()

        def mom_one(t):
            a, b = int(off[t]), int(off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            ri, rv, _, _ = oracle.momentum_topk_tensor(g_h[a:b], u_h[a:b], v_h[a:b], int(L.k[t]), 0.9,
                                                       base=a, seed=4, it=it)
            assert np.array_equal(gi[ka:kb], ri) and np.array_equal(_bits(gv[ka:kb]), _bits(rv)), \
                f"it {it} momentum tensor {t}"
        _pool_map(mom_one, range(T))
        assert np.array_equal(_bits(u.cpu().numpy()), _bits(u_h)), f"it {it}: u"
        assert np.array_equal(_bits(v.cpu().numpy()), _bits(v_h)), f"it {it}: v"


def _assert_kept_is_topk(acc, kept, off, k):
    """For every tensor: the kept set is the Top-k of |acc| with ties to the
    lower index (checked on the GPU): the smallest kept magnitude is at least
    the largest unkept one, and where they are equal every kept element of
    that magnitude precedes every unkept one."""
    for t in range(len(k)):
        a, b = int(off[t]), int(off[t + 1])
        if k[t] == 0 or k[t] == b - a:
            continue
        m = acc[a:b].abs()
        kt = kept[a:b]
        kmin = float(m[kt].min())
        umax = float(m.masked_fill(kt, -1.0).max())
        assert kmin >= umax, f"tensor {t}: a dropped |acc| {umax} exceeds a kept one {kmin}"
        if kmin == umax:
            tie = m == kmin
            last_kept = int(torch.nonzero(tie & kt).max())
            first_dropped = int(torch.nonzero(tie & ~kt).min())
            assert last_kept < first_dropped, f"tensor {t}: ties at the k-th magnitude not kept from the lowest index"


def test_llama3_8b_topk_int8_and_decompress_full(gc):
    lay = workloads.llama3_8b_layout()
    k = workloads.k_per_tensor(lay.sizes, 0.001)
    L = gc.Layout(lay.off, k, device="cuda")
    T, N, K = lay.num_tensors, lay.numel, L.total_k
    flags = gc.GC_EF | gc.GC_INT8
    comp = gc.TopkCompressor(L, flags)
    sizes = np.diff(L.off)
    sample = [int(np.argmin(sizes)), 2, 1, 5, 0]          # norm, k_proj, q_proj, gate_proj, embedding
    e = torch.zeros(N, device="cuda")
    e_prev = {t: np.zeros(int(sizes[t]), F32) for t in sample}
    g = torch.empty(N, device="cuda")
    owner = torch.repeat_interleave(torch.arange(T, device="cuda"), torch.from_numpy(k).cuda())
    base = torch.from_numpy(L.off[:-1]).cuda()[owner]
    for it in range(10):
        workloads.make_grad(5, lay, it, device="cuda", out=g)
        acc = g + e                                         # fp32 RNE add (torch), for the properties
        comp(g, e, seed=5, it=it)
        d = gc.get_device_status(comp.workspace)
        assert d.error_bits == 0 and d.exact_tensors == 0
        idx_all, q_all, sc_all = comp.idx[:K], comp.q[:K], comp.scale
        # properties over the whole arena
        assert int(idx_all.min()) >= 0 and bool((idx_all.long() < torch.from_numpy(sizes).cuda()[owner]).all())
        same = owner[1:] == owner[:-1]
        assert bool((idx_all[1:][same] > idx_all[:-1][same]).all()), "indices ascending within each tensor"
        assert int(q_all.abs().max()) <= 127
        gidx = base + idx_all.long()
        expect = acc.clone()
        expect[gidx] = acc[gidx] - q_all.float() * sc_all[owner]
        assert torch.equal(e.view(torch.int32), expect.view(torch.int32)), f"it {it}: EF identity over the arena"
        del expect
        kept = torch.zeros(N, dtype=torch.bool, device="cuda")
        kept[gidx] = True
        _assert_kept_is_topk(acc, kept, L.off, k)
        del kept, acc
        # sampled tensors against the oracle (the host checks run in parallel)
        host = {}
        for t in sample:
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            host[t] = (g[a:b].cpu().numpy(), comp.idx[ka:kb].cpu().numpy(), comp.q[ka:kb].cpu().numpy(),
                       float(comp.scale[t]), e[a:b].cpu().numpy())

        def one(t):
            g_h, gi, gq, gs, ge = host[t]
            e_prev[t] = _check_topk_tensor(L, t, g_h, e_prev[t], gi, gq, gs, ge, 5, it)
        _pool_map(one, sample)
        del host
    del e, g
    torch.cuda.empty_cache()
    # receiver: W = 8 workers' seeded fp32 payloads into one dense arena
    W = 8
    pays = [workloads.make_sparse_payload(lay, k, w, device="cuda", cfg=5) for w in range(W)]
    out = torch.zeros(N, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_DECOMPRESS)
    gc.sparse_decompress_accumulate(L, [p[0] for p in pays], [p[1] for p in pays], None, None, out, ws)
    assert gc.get_device_status(ws).error_bits == 0
    # whole arena: the workers added one after another (indices are distinct
    # within a worker, so each call adds once per element, in worker order)
    ref = torch.zeros(N, device="cuda")
    for p in pays:
        ref.index_put_((base + p[0].long(),), p[1], accumulate=True)
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), "receiver over the whole arena"
    del ref
    for t in sample:
        a, b = int(L.off[t]), int(L.off[t + 1])
        ka, kb = int(L.koff[t]), int(L.koff[t + 1])
        ref = np.zeros(b - a, F32)
        oracle.sparse_accumulate(np.asarray([0, b - a]), np.asarray([0, kb - ka]),
                                 [p[0][ka:kb].cpu().numpy() for p in pays], [p[1][ka:kb].cpu().numpy() for p in pays],
                                 None, None, ref)
        assert np.array_equal(_bits(out[a:b].cpu().numpy()), _bits(ref)), f"decompress tensor {t}"


@pytest.mark.parametrize("kind", ["qsgd", "sign"])
def test_bert_large_topk_kept_quantizers_full(gc, kind):
    """EF Top-k 0.1% + QSGD s = 16 or sign of the kept values on the BERT-large
    arena, ten iterations with the residual carried: indices, codes or bits,
    decoded values and residual bit-exact against the oracle given the GPU's
    per-tensor scale, which must be within 1e-6 of the oracle's."""
    lay = workloads.bert_large_layout()
    k = workloads.k_per_tensor(lay.sizes, 0.001)
    L = gc.Layout(lay.off, k, device="cuda")
    T, N, K = lay.num_tensors, lay.numel, L.total_k
    kq = {"qsgd": gc.GC_KEPT_QSGD, "sign": gc.GC_KEPT_SIGN}[kind]
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
    idx = torch.empty(K, dtype=torch.int32, device="cuda")
    val = torch.empty(K, device="cuda")
    q = torch.empty(K, dtype=torch.int8, device="cuda") if kind == "qsgd" else None
    bits = torch.empty(L.kept_words, dtype=torch.int32, device="cuda") if kind == "sign" else None
    sc = torch.empty(T, device="cuda")
    e = torch.zeros(N, device="cuda")
    e_ref = np.zeros(N, F32)
    kw = workloads.prefix((L.k + 31) // 32)
    for it in range(10):
        g = workloads.make_grad(3, lay, it, device="cuda")
        gc.ef_topk_compress_quantized(L, g, e, idx, val, q, bits, sc, kq, 16, 7, it, gc.GC_EF, ws)
        assert gc.get_device_status(ws).error_bits == 0
        g_h, gi, gv, gsc, ge = g.cpu().numpy(), idx.cpu().numpy(), val.cpu().numpy(), sc.cpu().numpy(), e.cpu().numpy()
        gq = q.cpu().numpy() if q is not None else None
        gb = bits.cpu().numpy().view(np.uint32) if bits is not None else None

        def one(t):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            _, _, _, _, s_ref = oracle.ef_topk_quantized_tensor(g_h[a:b], e_ref[a:b].copy(), int(L.k[t]), kind, 16,
                                                                base=a, seed=7, it=it)
            assert abs(float(gsc[t]) - s_ref) <= 1e-6 * abs(s_ref), f"it {it} tensor {t}: scale"
            et = e_ref[a:b].copy()
            ri, rv, rq, rb, _ = oracle.ef_topk_quantized_tensor(g_h[a:b], et, int(L.k[t]), kind, 16, base=a, seed=7,
                                                                it=it, scale_given=float(gsc[t]))
            assert np.array_equal(gi[ka:kb], ri), f"it {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"it {it} tensor {t}: decoded values"
            if kind == "qsgd":
                assert np.array_equal(gq[ka:kb], rq), f"it {it} tensor {t}: codes"
            else:
                assert np.array_equal(gb[kw[t]:kw[t + 1]], rb), f"it {it} tensor {t}: bits"
            assert np.array_equal(_bits(ge[a:b]), _bits(et)), f"it {it} tensor {t}: residual"
            e_ref[a:b] = et
        _pool_map(one, range(T))
