"""Bucketed compression: a layout made of tensors t0..t1-1 of a larger arena,
with that arena's element and entry offsets (Layout.bucket), gives exactly
the whole-arena call's outputs when the buckets run one by one or at once on
several streams, each with its own workspace.  The Top-k and random-k
buckets are also checked against the oracle directly (random draws at arena
indices), the other entry points against the whole-arena call, whose own
parity with the oracle the other GPU tests cover."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32 = np.float32

# more than 2^22 elements in all, so the whole call runs the multi-kernel
# pipeline while each bucket (at most 2^22) may take the one-launch path
SIZES = [100_003, 4097, 64, 300_000, 1, 33, 2_100_000, 513, 65_536, 1_000_001, 7, 16_385, 2_400_000]
BUCKETS = [(0, 4), (4, 7), (7, 13)]


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _same(a, b, what):
    a, b = a.cpu().numpy(), b.cpu().numpy()
    if a.dtype == np.float32:
        a, b = _bits(a), _bits(b)
    assert np.array_equal(a, b), what


def _layout(gc, rho):
    return gc.Layout(workloads.prefix(SIZES), workloads.k_per_tensor(SIZES, rho), device="cuda")


def _grad(n, seed):
    gen = torch.Generator().manual_seed(seed)
    x = torch.empty(n)
    workloads.fill_student_t(x, 3.0, 1e-3, gen)
    return x.cuda()


def _run_buckets(gc, L, op, flags, call, concurrent):
    """call(B, t0, t1, ws, stream) for every bucket; on one stream each when
    concurrent, else in order on the current stream."""
    cur = torch.cuda.current_stream()
    streams = [torch.cuda.Stream() for _ in BUCKETS] if concurrent else [cur] * len(BUCKETS)
    wss = []
    for (t0, t1), s in zip(BUCKETS, streams):
        B = L.bucket(t0, t1)
        ws = gc.alloc_workspace(B, op, flags)
        wss.append(ws)
        s.wait_stream(cur)
        call(B, t0, t1, ws, s)
    for s in streams:
        cur.wait_stream(s)
    torch.cuda.synchronize()
    for ws in wss:
        assert gc.get_device_status(ws).error_bits == 0


@pytest.mark.parametrize("flags_name", ["ef", "ef_int8", "ef_int8_pipeline", "randk_ef"])
@pytest.mark.parametrize("concurrent", [False, True])
def test_topk_buckets_equal_the_oracle(gc, flags_name, concurrent):
    flags = {"ef": gc.GC_EF, "ef_int8": gc.GC_EF | gc.GC_INT8,
             "ef_int8_pipeline": gc.GC_EF | gc.GC_INT8 | gc.GC_MULTI_KERNEL,
             "randk_ef": gc.GC_EF | gc.GC_RANDK}[flags_name]
    int8, randk = bool(flags & gc.GC_INT8), bool(flags & gc.GC_RANDK)
    L = _layout(gc, 0.01)
    N, K = L.numel, L.total_k
    seed = 77
    e_h = np.zeros(N, F32)
    e = torch.zeros(N, device="cuda")
    for it in range(2):
        g = _grad(N, 500 + it)
        g_h = g.cpu().numpy()
        idx = torch.full((K,), -1, dtype=torch.int32, device="cuda")
        val = torch.full((K,), -1.0, device="cuda")
        q = torch.zeros(K, dtype=torch.int8, device="cuda") if int8 else None
        sc = torch.zeros(L.T, device="cuda") if int8 else None

        def call(B, t0, t1, ws, s):
            gc.ef_topk_compress(B, g, e, idx, val, q, None if sc is None else sc[t0:t1], seed, it, flags, ws, s)

        _run_buckets(gc, L, gc.GC_OP_TOPK, flags, call, concurrent)
        gi, gv = idx.cpu().numpy(), val.cpu().numpy()
        for t in range(L.T):
            a, b = int(L.off[t]), int(L.off[t + 1])
            ka, kb = int(L.koff[t]), int(L.koff[t + 1])
            if randk:
                ri, rv = oracle.randk_tensor(g_h[a:b], e_h[a:b], int(L.k[t]), base=a, seed=seed, it=it,
                                             unbiased=False)
            else:
                ri, rv, rq, rs = oracle.ef_topk_tensor(g_h[a:b], e_h[a:b], int(L.k[t]), base=a, int8=int8,
                                                       seed=seed, it=it)
                if int8:
                    assert np.array_equal(q.cpu().numpy()[ka:kb], rq), f"tensor {t}: codes"
                    assert _bits(sc.cpu().numpy()[t:t + 1])[0] == _bits(np.asarray([rs], F32))[0], f"tensor {t}"
            assert np.array_equal(gi[ka:kb], ri), f"iteration {it} tensor {t}: indices"
            assert np.array_equal(_bits(gv[ka:kb]), _bits(rv)), f"iteration {it} tensor {t}: values"
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(e_h)), f"iteration {it}: residual"


def _whole_and_buckets(gc, L, op, flags, make, call, concurrent=True):
    """Runs `call` once on the whole layout and once bucket by bucket, each
    on fresh buffers from make(); returns both buffer dicts."""
    whole, parts = make(), make()
    ws = gc.alloc_workspace(L, op, flags)
    call(L, 0, L.T, ws, None, whole)
    torch.cuda.synchronize()
    assert gc.get_device_status(ws).error_bits == 0
    _run_buckets(gc, L, op, flags, lambda B, t0, t1, w, s: call(B, t0, t1, w, s, parts), concurrent)
    return whole, parts


@pytest.mark.parametrize("kind_name", ["qsgd", "sign"])
def test_kept_quantizer_buckets_equal_the_whole_call(gc, kind_name):
    kind = {"qsgd": gc.GC_KEPT_QSGD, "sign": gc.GC_KEPT_SIGN}[kind_name]
    L = _layout(gc, 0.01)
    N, K = L.numel, L.total_k
    g = _grad(N, 610)
    e0 = _grad(N, 611) * 0.5

    def make():
        return {"e": e0.clone(), "idx": torch.full((K,), -1, dtype=torch.int32, device="cuda"),
                "q": torch.zeros(K, dtype=torch.int8, device="cuda"),
                "bits": torch.zeros(L.kept_words, dtype=torch.int32, device="cuda"),
                "scale": torch.zeros(L.T, device="cuda")}

    def call(B, t0, t1, ws, s, d):
        w0 = L.kept_word_offset(t0)
        gc.ef_topk_compress_quantized(B, g, d["e"], d["idx"], None, d["q"] if kind == gc.GC_KEPT_QSGD else None,
                                      d["bits"][w0:] if kind == gc.GC_KEPT_SIGN else None, d["scale"][t0:t1],
                                      kind, 16, 9, 3, gc.GC_EF, ws, s)

    whole, parts = _whole_and_buckets(gc, L, gc.GC_OP_TOPK, gc.GC_EF, make, call)
    for name in whole:
        _same(whole[name], parts[name], name)


def test_momentum_buckets_equal_the_whole_call(gc):
    L = _layout(gc, 0.005)
    N, K = L.numel, L.total_k
    g = _grad(N, 620)
    u0, v0 = _grad(N, 621), _grad(N, 622)

    def make():
        return {"u": u0.clone(), "v": v0.clone(), "idx": torch.full((K,), -1, dtype=torch.int32, device="cuda"),
                "val": torch.zeros(K, device="cuda")}

    def call(B, t0, t1, ws, s, d):
        gc.ef_topk_compress_momentum(B, g, d["u"], d["v"], 0.9, d["idx"], d["val"], None, None, 5, 1, 0, ws, s)

    whole, parts = _whole_and_buckets(gc, L, gc.GC_OP_MOMENTUM, 0, make, call)
    for name in whole:
        _same(whole[name], parts[name], name)


@pytest.mark.parametrize("mode_name", ["int8_ef", "qsgd", "sign_ef"])
def test_dense_buckets_equal_the_whole_call(gc, mode_name):
    L = _layout(gc, 0.01)
    N = L.numel
    g = _grad(N, 630)
    e0 = _grad(N, 631) * 0.25
    ef = mode_name.endswith("_ef")

    def make():
        d = {"e": e0.clone() if ef else None, "scale": torch.zeros(L.T, device="cuda")}
        if mode_name == "sign_ef":
            d["bits"] = torch.zeros(L.words, dtype=torch.int32, device="cuda")
        else:
            d["codes"] = torch.zeros(N, dtype=torch.int8, device="cuda")
        return d

    def call(B, t0, t1, ws, s, d):
        if mode_name == "sign_ef":
            gc.sign_compress(B, g, d["e"], d["bits"][L.word_offset(t0):], d["scale"][t0:t1], ws, s)
        else:
            mode = gc.GC_Q_INT8 if mode_name == "int8_ef" else gc.GC_Q_QSGD
            gc.quantize_stochastic(B, g, d["e"], d["codes"], d["scale"][t0:t1], mode, 16, 21, 4, ws, s)

    op = gc.GC_OP_SIGN if mode_name == "sign_ef" else gc.GC_OP_QUANTIZE
    whole, parts = _whole_and_buckets(gc, L, op, 0, make, call)
    for name in whole:
        if whole[name] is not None:
            _same(whole[name], parts[name], name)


@pytest.mark.parametrize("int8", [False, True])
def test_receiver_buckets_equal_the_whole_call(gc, int8):
    L = _layout(gc, 0.01)
    N, K = L.numel, L.total_k
    W = 3
    pays = []
    for w in range(W):
        g = _grad(N, 640 + w)
        idx = torch.empty(K, dtype=torch.int32, device="cuda")
        val = torch.empty(K, device="cuda")
        q = torch.empty(K, dtype=torch.int8, device="cuda") if int8 else None
        sc = torch.empty(L.T, device="cuda") if int8 else None
        ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_INT8 if int8 else 0)
        gc.ef_topk_compress(L, g, None, idx, val, q, sc, 1, w, gc.GC_INT8 if int8 else 0, ws)
        pays.append((idx, val, q, sc))
    base = _grad(N, 650)

    def make():
        return {"out": base.clone()}

    def call(B, t0, t1, ws, s, d):
        gc.sparse_decompress_accumulate(B, [p[0] for p in pays], None if int8 else [p[1] for p in pays],
                                        [p[2] for p in pays] if int8 else None,
                                        [p[3][t0:t1] for p in pays] if int8 else None, d["out"], ws, s)

    whole, parts = _whole_and_buckets(gc, L, gc.GC_OP_DECOMPRESS, 0, make, call)
    _same(whole["out"], parts["out"], "receiver sums")
