"""gc_ef_topk_compress_noalloc: the compression entry point for callers that
cannot allocate device memory where they compress (their memory manager owns
the GPU's memory, or a cudaMalloc there would stall the device).  It uses a
fixed scratch array inside libgc instead of a caller workspace.

Checked through the C ABI against gc_ef_topk_compress (caller workspace) on
two calls in a row, with the residual carried from the first call to the
second: indices, values, int8 codes, scales and residuals must be identical
(bit-exact, the tolerance of all selection and residual checks here).
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gc(cuda_device):
    from gradient_compression_gb300 import build
    build.build()
    import gradient_compression_gb300 as gcmod
    return gcmod


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("case", ["flat_2p20_int8", "ragged_ef", "randk_ef"])
def test_noalloc_matches_workspace_entry_on_two_calls(gc, case):
    if case == "flat_2p20_int8":
        sizes, rho, flags = [1 << 20], 0.001, gc.GC_EF | gc.GC_INT8
    elif case == "ragged_ef":
        sizes, rho, flags = [4097, 1, 33, 100_003, 6, 70_000], 0.01, gc.GC_EF
    else:
        sizes, rho, flags = [4097, 1, 33, 100_003, 6, 70_000], 0.01, gc.GC_EF | gc.GC_RANDK
    k = workloads.k_per_tensor(sizes, rho)
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    assert gc.workspace_size(L, gc.GC_OP_TOPK, flags) <= gc.GC_NOALLOC_MAX_WORKSPACE_BYTES
    n, K = L.numel, L.total_k
    int8 = bool(flags & gc.GC_INT8)
    gen = torch.Generator().manual_seed(17)
    e0 = (torch.randn(n, generator=gen) * 1e-4).float().cuda()
    e_ws, e_na = e0.clone(), e0.clone()
    ws = gc.alloc_workspace(L, gc.GC_OP_TOPK, flags)

    def outs():
        return (torch.empty(K, dtype=torch.int32, device="cuda"),
                torch.empty(K, dtype=torch.float32, device="cuda"),
                torch.empty(K, dtype=torch.int8, device="cuda") if int8 else None,
                torch.empty(L.T, dtype=torch.float32, device="cuda") if int8 else None)

    for it in range(2):
        g_h = torch.empty(n)
        workloads.fill_student_t(g_h, 3.0, 1e-3, torch.Generator().manual_seed(100 + it))
        g = g_h.cuda()
        a, b = outs(), outs()
        gc.ef_topk_compress(L, g, e_ws, *a, 5, it, flags, ws)
        gc.ef_topk_compress_noalloc(L, g, e_na, *b, 5, it, flags)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]), f"call {it}: indices"
        assert np.array_equal(_bits(a[1]), _bits(b[1])), f"call {it}: values"
        if int8:
            assert torch.equal(a[2], b[2]), f"call {it}: int8 codes"
            assert np.array_equal(_bits(a[3]), _bits(b[3])), f"call {it}: scales"
        assert np.array_equal(_bits(e_ws), _bits(e_na)), f"call {it}: residual"
        # the built-in scratch's diagnostics are this call's, and match the workspace's
        d_ws, d_na = gc.get_device_status(ws), gc.noalloc_device_status()
        assert d_na.error_bits == 0
        assert (d_na.exact_tensors, d_na.overflow_tensors) == (d_ws.exact_tensors, d_ws.overflow_tensors)


def test_noalloc_rejects_layout_beyond_its_scratch(gc):
    lay = workloads.bert_large_layout()
    k = workloads.k_per_tensor(lay.sizes, 0.001)
    L = gc.Layout(lay.off, k, device="cuda")
    assert gc.workspace_size(L, gc.GC_OP_TOPK, gc.GC_EF) > gc.GC_NOALLOC_MAX_WORKSPACE_BYTES
    with pytest.raises(gc.GCError) as ei:
        gc.ef_topk_compress_noalloc(L, None, None, None, None, None, None, 0, 0, gc.GC_EF)
    assert ei.value.status in (gc.GC_ERR_WORKSPACE, gc.GC_ERR_INVALID_ARG)
    # with valid pointers the only objection left is the size
    g = torch.zeros(16, device="cuda")
    st = gc.lib().gc_ef_topk_compress_noalloc(L.dev(), L.host(), g.data_ptr(), g.data_ptr(), g.data_ptr(),
                                              g.data_ptr(), None, None, 0, 0, gc.GC_EF, None)
    assert st == gc.GC_ERR_WORKSPACE


def test_noalloc_status_reports_layout_mismatch_then_clears(gc):
    """A noalloc call whose device layout disagrees with the host mirror does
    nothing and says so through gc_ef_topk_compress_noalloc_status, like a
    workspace call through gc_get_device_status; the next good call's status
    is clean, and with GC_FORCE_EXACT it counts every selecting tensor."""
    sizes = [1000, 2000]
    k = [10, 20]
    L = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    bad = gc.Layout(workloads.prefix([1000, 3000]), k, device="cuda")
    L._dev_off.copy_(bad._dev_off)                 # device copy disagrees with the host mirror
    g = torch.zeros(3000, device="cuda")
    e = torch.zeros(3000, device="cuda")
    idx = torch.full((30,), -7, dtype=torch.int32, device="cuda")
    val = torch.zeros(30, device="cuda")
    gc.ef_topk_compress_noalloc(L, g, e, idx, val, None, None, 0, 0, gc.GC_EF)
    d = gc.noalloc_device_status(raise_on_error=False)
    assert d.error_bits & gc.GC_DIAG_LAYOUT_MISMATCH
    with pytest.raises(gc.GCError) as ei:
        gc.noalloc_device_status()
    assert ei.value.status == gc.GC_ERR_DEVICE
    assert (idx.cpu() == -7).all()
    good = gc.Layout(workloads.prefix(sizes), k, device="cuda")
    g = torch.randn(3000, device="cuda")
    gc.ef_topk_compress_noalloc(good, g, e, idx, val, None, None, 0, 1, gc.GC_EF | gc.GC_FORCE_EXACT)
    d = gc.noalloc_device_status()
    assert d.error_bits == 0 and d.exact_tensors == 2 and d.overflow_tensors == 0
    assert (idx.cpu() >= 0).all()
