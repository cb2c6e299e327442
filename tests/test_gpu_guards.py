"""Guard words and resumption.

Guard words: every output, in/out and workspace buffer handed to the
library is a view into a larger allocation filled with a sentinel; after the
call the sentinel regions before and after each view must be untouched (no
out-of-bounds write by any kernel).  Resumption: the compression state is
the residual e (u and v for momentum) plus (seed, iteration); a run stopped
after two steps, copied to the host and restored into fresh buffers must
continue bit-identically to an uninterrupted run."""
import numpy as np
import pytest
import torch

import workloads
from test_gpu_parity import F32, _bits

pytestmark = pytest.mark.gpu

GUARD_BYTES = 256            # guard bytes on each side (keeps the views 256-byte aligned)
SENT_F = -7.25e30
SENT_I = -123456789


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


class Guarded:
    """n elements of dtype, preceded and followed by GUARD_BYTES of sentinel."""

    def __init__(self, n, dtype, init=None):
        self.n, self.dtype = n, dtype
        self.pad = GUARD_BYTES // torch.empty(0, dtype=dtype).element_size()
        fill = SENT_F if dtype.is_floating_point else (SENT_I if dtype == torch.int32 else -77)
        if dtype == torch.uint8:
            fill = 0xA5
        self.buf = torch.full((n + 2 * self.pad,), fill, dtype=dtype, device="cuda")
        self.fill = fill
        if init is not None:
            self.view.copy_(init)

    @property
    def view(self):
        return self.buf[self.pad:self.pad + self.n]

    def check(self, name):
        b = self.buf.cpu()
        head, tail = b[:self.pad], b[self.pad + self.n:]
        assert bool((head == self.fill).all()) and bool((tail == self.fill).all()), f"{name}: guard words overwritten"


def _layout(gc, sizes, rho):
    k = workloads.k_per_tensor(np.asarray(sizes), rho)
    return gc.Layout(workloads.prefix(np.asarray(sizes)), k, device="cuda")


SIZES = [4097, 1, 33, 100_003, 6, 70_000, 300_001]


@pytest.mark.parametrize("flags_name", ["ef_int8", "ef", "noef", "randk", "ef_exact", "ef_int8_pipeline", "ef_pipeline"])
def test_topk_writes_stay_in_bounds(gc, flags_name):
    # this layout runs as one cooperative launch unless a flag asks for the pipeline
    flags = {"ef_int8": gc.GC_EF | gc.GC_INT8, "ef": gc.GC_EF, "noef": 0, "randk": gc.GC_EF | gc.GC_RANDK,
             "ef_exact": gc.GC_EF | gc.GC_FORCE_EXACT, "ef_int8_pipeline": gc.GC_EF | gc.GC_INT8 | gc.GC_MULTI_KERNEL,
             "ef_pipeline": gc.GC_EF | gc.GC_MULTI_KERNEL}[flags_name]
    L = _layout(gc, SIZES, 0.01)
    N, K, T = L.numel, L.total_k, L.T
    int8 = bool(flags & gc.GC_INT8)
    g = Guarded(N, torch.float32, torch.randn(N) * 1e-3)
    e = Guarded(N, torch.float32, torch.randn(N) * 1e-4)
    idx = Guarded(K, torch.int32)
    val = Guarded(K, torch.float32)
    q = Guarded(K, torch.int8) if int8 else None
    sc = Guarded(T, torch.float32) if int8 else None
    ws0 = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    ws = Guarded(ws0.numel(), torch.uint8)
    for it in range(2):
        gc.ef_topk_compress(L, g.view, e.view, idx.view, val.view, q.view if q else None, sc.view if sc else None,
                            3, it, flags, ws.view)
        assert gc.get_device_status(ws.view).error_bits == 0
    for name, b in (("g", g), ("e", e), ("idx", idx), ("val", val), ("q", q), ("scale", sc), ("workspace", ws)):
        if b is not None:
            b.check(name)


def test_momentum_writes_stay_in_bounds(gc):
    L = _layout(gc, SIZES, 0.005)
    N, K = L.numel, L.total_k
    g = Guarded(N, torch.float32, torch.randn(N) * 1e-3)
    u, v = Guarded(N, torch.float32, torch.zeros(N)), Guarded(N, torch.float32, torch.zeros(N))
    idx, val = Guarded(K, torch.int32), Guarded(K, torch.float32)
    ws0 = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM)
    ws = Guarded(ws0.numel(), torch.uint8)
    for it in range(2):
        gc.ef_topk_compress_momentum(L, g.view, u.view, v.view, 0.9, idx.view, val.view, None, None, 1, it, 0,
                                     ws.view)
        assert gc.get_device_status(ws.view).error_bits == 0
    for name, b in (("g", g), ("u", u), ("v", v), ("idx", idx), ("val", val), ("workspace", ws)):
        b.check(name)


@pytest.mark.parametrize("op", ["sign", "qsgd", "int8"])
def test_dense_writes_stay_in_bounds(gc, op):
    L = _layout(gc, SIZES, 0.0)
    N, T = L.numel, L.T
    g = Guarded(N, torch.float32, torch.randn(N) * 1e-3)
    e = Guarded(N, torch.float32, torch.randn(N) * 1e-4)
    sc = Guarded(T, torch.float32)
    if op == "sign":
        bits = Guarded(L.words, torch.int32)
        ws0 = gc.alloc_workspace(L, gc.GC_OP_SIGN)
        ws = Guarded(ws0.numel(), torch.uint8)
        gc.sign_compress(L, g.view, e.view, bits.view, sc.view, ws.view)
        outs = (("bits", bits),)
    else:
        codes = Guarded(N, torch.int8)
        ws0 = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE)
        ws = Guarded(ws0.numel(), torch.uint8)
        mode = gc.GC_Q_QSGD if op == "qsgd" else gc.GC_Q_INT8
        gc.quantize_stochastic(L, g.view, e.view, codes.view, sc.view, mode, 16 if op == "qsgd" else 0, 2, 0,
                               ws.view)
        outs = (("codes", codes),)
    assert gc.get_device_status(ws.view).error_bits == 0
    for name, b in (("g", g), ("e", e), ("scale", sc), ("workspace", ws)) + outs:
        b.check(name)


def test_powersgd_writes_stay_in_bounds(gc):
    shapes = [(5, 7), (300, 1024), (9000, 16), (64, 4096)]
    starts, pos = [], 0
    for m, n in shapes:
        starts.append(pos)
        pos += m * n
    ml = gc.MatrixLayout(starts, [s[0] for s in shapes], [s[1] for s in shapes], device="cuda")
    R = 4
    Msum, Nsum = int(ml.poff[-1]), int(ml.qoff[-1])
    g = Guarded(pos, torch.float32, torch.randn(pos))
    e = Guarded(pos, torch.float32, torch.zeros(pos))
    q = Guarded(Nsum * R, torch.float32, torch.randn(Nsum * R))
    p = Guarded(Msum * R, torch.float32)
    praw = Guarded(Msum * R, torch.float32)
    ws0 = gc.powersgd_workspace(ml, R)
    ws = Guarded(ws0.numel(), torch.uint8)
    gc.powersgd_compress(ml, R, g.view, e.view, q.view, p.view, praw.view, ws.view)
    out = Guarded(pos, torch.float32, torch.zeros(pos))
    gc.powersgd_decompress_accumulate(ml, R, p.view, q.view, out.view, ws.view)
    assert gc.get_device_status(ws.view).error_bits == 0
    for name, b in (("g", g), ("e", e), ("q", q), ("p", p), ("p_raw", praw), ("out", out), ("workspace", ws)):
        b.check(name)


@pytest.mark.parametrize("mode", ["topk_int8", "momentum_int8"])
def test_resume_from_host_copy_is_bit_identical(gc, mode):
    lay = workloads.bert_large_layout()
    sizes = lay.sizes[:40]
    L = gc.Layout(workloads.prefix(sizes), workloads.k_per_tensor(sizes, 0.01), device="cuda")
    N, K, T = L.numel, L.total_k, L.T
    grads = [torch.randn(N, generator=torch.Generator().manual_seed(70 + i)).cuda() * 1e-3 for i in range(4)]

    def run(state, its):
        outs = []
        if mode == "topk_int8":
            flags = gc.GC_EF | gc.GC_INT8
            ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
            idx = torch.empty(K, dtype=torch.int32, device="cuda")
            q = torch.empty(K, dtype=torch.int8, device="cuda")
            sc = torch.empty(T, device="cuda")
            for it in its:
                gc.ef_topk_compress(L, grads[it], state[0], idx, None, q, sc, 11, it, flags, ws)
                outs.append((idx.clone(), q.clone(), sc.clone()))
        else:
            flags = gc.GC_INT8
            ws = gc.alloc_workspace(L, gc.GC_OP_MOMENTUM, flags)
            idx = torch.empty(K, dtype=torch.int32, device="cuda")
            q = torch.empty(K, dtype=torch.int8, device="cuda")
            sc = torch.empty(T, device="cuda")
            for it in its:
                gc.ef_topk_compress_momentum(L, grads[it], state[0], state[1], 0.9, idx, None, q, sc, 11, it,
                                             flags, ws)
                outs.append((idx.clone(), q.clone(), sc.clone()))
        return outs

    nstate = 1 if mode == "topk_int8" else 2
    straight = [torch.zeros(N, device="cuda") for _ in range(nstate)]
    ref = run(straight, range(4))
    first = [torch.zeros(N, device="cuda") for _ in range(nstate)]
    run(first, range(2))
    checkpoint = [s.cpu().numpy().copy() for s in first]          # the state a caller saves
    del first
    resumed = [torch.from_numpy(c).cuda() for c in checkpoint]     # fresh buffers, fresh workspace
    tail = run(resumed, range(2, 4))
    for (ri, rq, rs), (ti, tq, ts) in zip(ref[2:], tail):
        assert torch.equal(ri, ti) and torch.equal(rq, tq) and torch.equal(rs.view(torch.int32), ts.view(torch.int32))
    for a, b in zip(straight, resumed):
        assert np.array_equal(_bits(a.cpu().numpy()), _bits(b.cpu().numpy())), "state after resuming"
