"""CUDA-graph capture of the device-counter entry points: one captured call,
replayed for several steps with fresh gradients copied into its input
buffer, must give bit-identical payloads, codes and residuals to direct
calls of the plain entry points with iter = 0, 1, 2, ... (random-k keys and
stochastic rounding depend on the iteration), and the counter must advance
by one per replay."""
import numpy as np
import pytest
import torch

import workloads
from test_gpu_parity import _bits

pytestmark = pytest.mark.gpu

SIZES = [4097, 1, 33, 100_003, 6, 70_000, 300_001]
STEPS = 4


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _grads(n):
    return [torch.randn(n, generator=torch.Generator().manual_seed(900 + i)).cuda() * 1e-3 for i in range(STEPS)]


@pytest.mark.parametrize("flags_name", ["randk_ef", "topk_int8", "topk_int8_pipeline"])
def test_topk_graph_replay_matches_direct_calls(gc, flags_name):
    # topk_int8 captures the one-launch path (a cooperative kernel node)
    flags = {"randk_ef": gc.GC_EF | gc.GC_RANDK, "topk_int8": gc.GC_EF | gc.GC_INT8,
             "topk_int8_pipeline": gc.GC_EF | gc.GC_INT8 | gc.GC_MULTI_KERNEL}[flags_name]
    int8 = bool(flags & gc.GC_INT8)
    sizes = np.asarray(SIZES)
    L = gc.Layout(workloads.prefix(sizes), workloads.k_per_tensor(sizes, 0.01), device="cuda")
    N, K, T = L.numel, L.total_k, L.T
    grads = _grads(N)

    def bufs():
        return (torch.empty(K, dtype=torch.int32, device="cuda"),
                None if int8 else torch.empty(K, device="cuda"),
                torch.empty(K, dtype=torch.int8, device="cuda") if int8 else None,
                torch.empty(T, device="cuda") if int8 else None)

    # direct calls
    e_ref = torch.zeros(N, device="cuda")
    ws_ref = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    idx, val, q, sc = bufs()
    ref = []
    for it in range(STEPS):
        gc.ef_topk_compress(L, grads[it], e_ref, idx, val, q, sc, 7, 10 + it, flags, ws_ref)
        ref.append([x.clone() if x is not None else None for x in (idx, val, q, sc)] + [e_ref.clone()])
    # one capture, replayed
    g_in = torch.empty(N, device="cuda")
    e = torch.zeros(N, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)
    gi, gv, gq, gs = bufs()
    it_dev = torch.full((1,), 10, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gc.ef_topk_compress_dev_iter(L, g_in, e, gi, gv, gq, gs, 7, it_dev, flags, ws)
    torch.cuda.synchronize()
    # capturing ran nothing: state and counter untouched
    assert int(it_dev.item()) == 10 and not bool(e.any())
    for it in range(STEPS):
        g_in.copy_(grads[it])
        graph.replay()
        torch.cuda.synchronize()
        assert int(it_dev.item()) == 11 + it
        assert gc.get_device_status(ws).error_bits == 0
        r = ref[it]
        assert torch.equal(gi, r[0]), f"step {it}: indices"
        if int8:
            assert torch.equal(gq, r[2]) and torch.equal(gs.view(torch.int32), r[3].view(torch.int32)), f"step {it}: codes"
        else:
            assert torch.equal(gv.view(torch.int32), r[1].view(torch.int32)), f"step {it}: values"
        assert np.array_equal(_bits(e.cpu().numpy()), _bits(r[4].cpu().numpy())), f"step {it}: residual"


def test_qsgd_graph_replay_matches_direct_calls(gc):
    sizes = np.asarray(SIZES)
    L = gc.Layout(workloads.prefix(sizes), np.zeros(len(sizes), np.int64), device="cuda")
    N, T = L.numel, L.T
    grads = _grads(N)
    ws_ref = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE)
    codes = torch.empty(N, dtype=torch.int8, device="cuda")
    norm = torch.empty(T, device="cuda")
    ref = []
    for it in range(STEPS):
        gc.quantize_stochastic(L, grads[it], None, codes, norm, gc.GC_Q_QSGD, 16, 3, it, ws_ref)
        ref.append((codes.clone(), norm.clone()))
    g_in = torch.empty(N, device="cuda")
    gcod = torch.empty(N, dtype=torch.int8, device="cuda")
    gn = torch.empty(T, device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_QUANTIZE)
    it_dev = torch.zeros(1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            gc.quantize_stochastic_dev_iter(L, g_in, None, gcod, gn, gc.GC_Q_QSGD, 16, 3, it_dev, ws)
    for it in range(STEPS):
        g_in.copy_(grads[it])
        graph.replay()
        torch.cuda.synchronize()
        assert int(it_dev.item()) == it + 1
        assert torch.equal(gcod, ref[it][0]) and torch.equal(gn.view(torch.int32), ref[it][1].view(torch.int32))


def test_dev_iter_rejects_a_misaligned_counter(gc):
    sizes = np.asarray([100, 200])
    L = gc.Layout(workloads.prefix(sizes), np.asarray([1, 2]), device="cuda")
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, gc.GC_EF)
    base = torch.zeros(4, dtype=torch.int64, device="cuda")
    bad = base.data_ptr() + 4
    with pytest.raises(gc.GCError):
        gc.ef_topk_compress_dev_iter(L, torch.zeros(300, device="cuda"), torch.zeros(300, device="cuda"),
                                     torch.empty(3, dtype=torch.int32, device="cuda"),
                                     torch.empty(3, device="cuda"), None, None, 0, bad, gc.GC_EF, ws)
