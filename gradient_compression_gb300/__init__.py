"""Python binding of libgc (EF gradient compression on GB300).

Argument marshalling only: every step of the compression path runs in the
CUDA kernels of libgc.so, called through its C ABI (include/gc.h).  PyTorch
provides device memory and the current stream.  There is no CPU fallback:
if the library is not built, importing the binding raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgc.so")

GC_OK, GC_ERR_INVALID_ARG, GC_ERR_LAYOUT, GC_ERR_WORKSPACE, GC_ERR_ALIGNMENT, GC_ERR_CUDA, GC_ERR_DEVICE = range(7)
GC_EF, GC_INT8, GC_RANDK, GC_UNBIASED, GC_NO_MASK, GC_FORCE_EXACT = 0x1, 0x2, 0x4, 0x8, 0x10, 0x100
GC_MULTI_KERNEL = 0x200
GC_OP_TOPK, GC_OP_MOMENTUM, GC_OP_SIGN, GC_OP_QUANTIZE, GC_OP_DECOMPRESS = range(5)
GC_Q_INT8, GC_Q_QSGD = 0, 1
GC_DENSE_SIGN, GC_DENSE_INT8, GC_DENSE_QSGD = 0, 1, 2
GC_KEPT_INT8, GC_KEPT_QSGD, GC_KEPT_SIGN = 1, 2, 3
GC_DIAG_LAYOUT_MISMATCH, GC_DIAG_SELECT, GC_DIAG_INDEX_RANGE, GC_DIAG_BAD_THRESHOLD = 0x1, 0x2, 0x4, 0x8
GC_DIAG_INDEX_ORDER, GC_DIAG_TIMEOUT = 0x10, 0x20
GC_NOALLOC_MAX_WORKSPACE_BYTES = 32 << 20


class gc_layout(C.Structure):
    _fields_ = [("num_tensors", C.c_int32), ("off", C.c_void_p), ("k", C.c_void_p), ("koff", C.c_void_p)]


class gc_matrix_layout(C.Structure):
    _fields_ = [("num_tensors", C.c_int32), ("start", C.c_void_p), ("rows", C.c_void_p), ("cols", C.c_void_p)]


class gc_diag(C.Structure):
    _fields_ = [("error_bits", C.c_uint32), ("exact_tensors", C.c_uint32),
                ("overflow_tensors", C.c_uint32), ("one_launch", C.c_uint32)]


class GCError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib() -> C.CDLL:
    """The loaded libgc.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgc.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                               "or python gradient_compression_gb300/build.py")
        L = C.CDLL(LIB_PATH)
        P, I32, I64, U32, U64, F, SZ = (C.c_void_p, C.c_int32, C.c_int64, C.c_uint32, C.c_uint64,
                                        C.c_float, C.c_size_t)
        LP = C.POINTER(gc_layout)
        L.gc_workspace_size.argtypes = [LP, I32, U32, C.POINTER(SZ)]
        L.gc_ef_topk_compress.argtypes = [LP, LP, P, P, P, P, P, P, U64, U64, U32, P, SZ, P]
        L.gc_ef_topk_compress_profiled.argtypes = [LP, LP, P, P, P, P, P, P, U64, U64, U32, P, SZ, P, P, I32]
        L.gc_ef_topk_compress_lazy.argtypes = [LP, LP, P, P, P, P, P, P, P, U64, U64, U32, P, SZ, P]
        L.gc_ef_residual_materialize.argtypes = [LP, LP, P, P, P]
        L.gc_sign_compress_lazy.argtypes = [LP, LP, P, P, P, P, P, P, SZ, P]
        L.gc_sign_residual_materialize.argtypes = [LP, LP, P, P, P]
        MLP = C.POINTER(gc_matrix_layout)
        L.gc_powersgd_workspace_size.argtypes = [MLP, I32, C.POINTER(SZ)]
        L.gc_powersgd_compress.argtypes = [MLP, MLP, I32, P, P, P, P, P, P, SZ, P]
        L.gc_powersgd_decompress_accumulate.argtypes = [MLP, MLP, I32, P, P, P, P, SZ, P]
        L.gc_powersgd_compress_lazy.argtypes = [MLP, MLP, I32, P, P, P, P, P, P, P, SZ, P]
        L.gc_powersgd_residual_materialize.argtypes = [MLP, MLP, I32, P, P, P, P, SZ, P]
        L.gc_ef_topk_compress_clipped.argtypes = [LP, LP, P, P, P, P, P, P, P, P, U64, U64, U32, P, SZ, P]
        L.gc_ef_threshold_compress.argtypes = [LP, LP, P, P, P, P, P, P, P, P, U64, U64, U32, P, SZ, P]
        L.gc_warmup_density.argtypes = [I64, I64, C.c_double, C.c_double, I32, I32]
        L.gc_warmup_density.restype = C.c_double
        L.gc_ef_topk_compress_noalloc.argtypes = [LP, LP, P, P, P, P, P, P, U64, U64, U32, P]
        L.gc_ef_topk_compress_noalloc_status.argtypes = [P, C.POINTER(gc_diag)]
        L.gc_ef_topk_compress_momentum.argtypes = [LP, LP, P, P, P, F, P, P, P, P, U64, U64, U32, P, SZ, P]
        L.gc_ef_topk_compress_quantized.argtypes = [LP, LP, P, P, P, P, P, P, P, I32, I32, U64, U64, U32, P, SZ, P]
        L.gc_ef_topk_compress_momentum_quantized.argtypes = [LP, LP, P, P, P, F, P, P, P, P, P, I32, I32, U64, U64,
                                                             U32, P, SZ, P]
        L.gc_sign_compress.argtypes = [LP, LP, P, P, P, P, P, SZ, P]
        L.gc_quantize_stochastic.argtypes = [LP, LP, P, P, P, P, I32, I32, U64, U64, P, SZ, P]
        L.gc_quantize_stochastic_dev_iter.argtypes = [LP, LP, P, P, P, P, I32, I32, U64, P, P, SZ, P]
        L.gc_ef_topk_compress_dev_iter.argtypes = [LP, LP, P, P, P, P, P, P, U64, P, U32, P, SZ, P]
        L.gc_sparse_decompress_accumulate.argtypes = [LP, LP, I32, P, P, P, P, P, P, SZ, P]
        L.gc_sparse_decompress_accumulate_quantized.argtypes = [LP, LP, I32, I32, I32, P, P, P, P, P, P, SZ, P]
        L.gc_dense_decompress_accumulate.argtypes = [LP, LP, I32, I32, I32, P, P, P, P, SZ, P]
        L.gc_get_device_status.argtypes = [P, SZ, P, C.POINTER(gc_diag)]
        L.gc_status_string.argtypes = [I32]
        L.gc_status_string.restype = C.c_char_p
        L.gc_version.restype = I32
        for name in ("gc_workspace_size", "gc_ef_topk_compress", "gc_ef_topk_compress_profiled",
                     "gc_ef_topk_compress_noalloc", "gc_ef_topk_compress_noalloc_status",
                     "gc_ef_topk_compress_lazy", "gc_ef_residual_materialize",
                     "gc_sign_compress_lazy", "gc_sign_residual_materialize", "gc_ef_threshold_compress",
                     "gc_ef_topk_compress_clipped", "gc_powersgd_workspace_size", "gc_powersgd_compress",
                     "gc_powersgd_decompress_accumulate", "gc_powersgd_compress_lazy",
                     "gc_powersgd_residual_materialize",
                     "gc_ef_topk_compress_momentum", "gc_ef_topk_compress_quantized",
                     "gc_ef_topk_compress_momentum_quantized",
                     "gc_sign_compress", "gc_quantize_stochastic", "gc_sparse_decompress_accumulate",
                     "gc_sparse_decompress_accumulate_quantized",
                     "gc_dense_decompress_accumulate", "gc_get_device_status",
                     "gc_ef_topk_compress_dev_iter", "gc_quantize_stochastic_dev_iter"):
            getattr(L, name).restype = I32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gc_status_string(int(status)).decode()


def version() -> int:
    return int(lib().gc_version())


def _check(status: int, what: str) -> None:
    if status != GC_OK:
        raise GCError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Layout:
    """A flat-arena layout: host arrays (validation, sizing) + device copies.

    off[t]..off[t+1] are tensor t's elements; k (optional) kept entries per
    tensor; koff their running sum from koff0 (0 for a whole arena; a
    bucket, made by Layout.bucket, keeps its arena's offsets).
    """

    def __init__(self, off, k=None, device="cuda", koff0=0):
        self.off = np.ascontiguousarray(off, dtype=np.int64)
        self.T = int(self.off.size - 1)
        if k is not None:
            self.k = np.ascontiguousarray(k, dtype=np.int64)
            self.koff = np.full(self.T + 1, int(koff0), np.int64)
            self.koff[1:] += np.cumsum(self.k)
        else:
            self.k = self.koff = None
        self.device = torch.device(device)
        self._host = gc_layout(self.T, self.off.ctypes.data, None if self.k is None else self.k.ctypes.data,
                               None if self.koff is None else self.koff.ctypes.data)
        self._dev_off = self._dev_k = self._dev_koff = None
        self._dev = None
        if self.device.type == "cuda":
            self._dev_off = torch.from_numpy(self.off).to(self.device)
            if self.k is not None:
                self._dev_k = torch.from_numpy(self.k).to(self.device)
                self._dev_koff = torch.from_numpy(self.koff).to(self.device)
            self._dev = gc_layout(self.T, _ptr(self._dev_off), _ptr(self._dev_k), _ptr(self._dev_koff))

    def bucket(self, t0: int, t1: int) -> "Layout":
        """Tensors t0 .. t1-1 as a layout of their own with this arena's
        element and entry offsets: calls on it read and write the whole
        arena's element and payload arrays at those offsets, and the
        per-tensor arrays and sign-bit words passed offset to tensor t0
        (word_offset / kept_word_offset)."""
        if not 0 <= t0 < t1 <= self.T:
            raise ValueError(f"bucket [{t0}, {t1}) outside 0..{self.T}")
        k = None if self.k is None else self.k[t0:t1]
        return Layout(self.off[t0:t1 + 1], k, device=self.device,
                      koff0=0 if self.koff is None else int(self.koff[t0]))

    @property
    def numel(self) -> int:
        """Elements the arena's arrays must hold (the end of the last tensor)."""
        return int(self.off[-1])

    @property
    def total_k(self) -> int:
        """Entries the payload arrays must hold (the end of the last tensor's)."""
        return int(self.koff[-1]) if self.koff is not None else 0

    def word_offset(self, t: int) -> int:
        """First sign-bit word of tensor t (dense sign compressor)."""
        n = np.diff(self.off[:t + 1])
        return int(((n + 31) // 32).sum())

    def kept_word_offset(self, t: int) -> int:
        """First word of tensor t's kept-value sign bits."""
        return int(((self.k[:t] + 31) // 32).sum())

    @property
    def kept_words(self) -> int:
        """uint32 words of the kept-value sign bits: sum of ceil(k_t / 32)."""
        return int(((self.k + 31) // 32).sum())

    @property
    def words(self) -> int:
        n = np.diff(self.off)
        return int(((n + 31) // 32).sum())

    def host(self):
        return C.byref(self._host)

    def dev(self):
        if self._dev is None:
            raise RuntimeError("layout has no device copy")
        return C.byref(self._dev)


class MatrixLayout:
    """Matrices of an arena for PowerSGD: host arrays + device copies."""

    def __init__(self, start, rows, cols, device="cuda"):
        self.start = np.ascontiguousarray(start, dtype=np.int64)
        self.rows = np.ascontiguousarray(rows, dtype=np.int64)
        self.cols = np.ascontiguousarray(cols, dtype=np.int64)
        self.T = int(self.start.size)
        self.device = torch.device(device)
        self._host = gc_matrix_layout(self.T, self.start.ctypes.data, self.rows.ctypes.data, self.cols.ctypes.data)
        self._dev = None
        if self.device.type == "cuda":
            self._d = [torch.from_numpy(a).to(self.device) for a in (self.start, self.rows, self.cols)]
            self._dev = gc_matrix_layout(self.T, *[_ptr(x) for x in self._d])
        self.poff = np.zeros(self.T + 1, np.int64); self.poff[1:] = np.cumsum(self.rows)
        self.qoff = np.zeros(self.T + 1, np.int64); self.qoff[1:] = np.cumsum(self.cols)

    def host(self):
        return C.byref(self._host)

    def dev(self):
        return C.byref(self._dev)


def powersgd_workspace(ml: MatrixLayout, rank: int, device=None) -> torch.Tensor:
    out = C.c_size_t(0)
    _check(lib().gc_powersgd_workspace_size(ml.host(), int(rank), C.byref(out)), "gc_powersgd_workspace_size")
    return torch.empty(max(int(out.value), 256), dtype=torch.uint8, device=device or ml.device)


def powersgd_compress(ml, rank, g, e, q, p, p_raw, workspace, stream=None):
    _check(lib().gc_powersgd_compress(ml.dev(), ml.host(), int(rank), _ptr(g), _ptr(e), _ptr(q), _ptr(p),
                                      _ptr(p_raw), _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_powersgd_compress")


def powersgd_compress_lazy(ml, rank, g, e, q, p, p_prev, p_raw, workspace, stream=None):
    """powersgd_compress with the residual kept pending (e holds M; p_prev is
    the previous call's p, or None when e is a plain residual)."""
    _check(lib().gc_powersgd_compress_lazy(ml.dev(), ml.host(), int(rank), _ptr(g), _ptr(e), _ptr(q), _ptr(p),
                                           _ptr(p_prev), _ptr(p_raw), _ptr(workspace), workspace.numel(),
                                           _stream(stream)), "gc_powersgd_compress_lazy")


def powersgd_residual_materialize(ml, rank, e, p, q, workspace, stream=None):
    _check(lib().gc_powersgd_residual_materialize(ml.dev(), ml.host(), int(rank), _ptr(e), _ptr(p), _ptr(q),
                                                  _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_powersgd_residual_materialize")


def powersgd_decompress_accumulate(ml, rank, p, q, out, workspace, stream=None):
    _check(lib().gc_powersgd_decompress_accumulate(ml.dev(), ml.host(), int(rank), _ptr(p), _ptr(q), _ptr(out),
                                                   _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_powersgd_decompress_accumulate")


def workspace_size(layout: Layout, op: int, flags: int = 0) -> int:
    out = C.c_size_t(0)
    _check(lib().gc_workspace_size(layout.host(), op, flags, C.byref(out)), "gc_workspace_size")
    return int(out.value)


def alloc_workspace(layout: Layout, op: int, flags: int = 0, device=None) -> torch.Tensor:
    """A workspace tensor (uint8) of the size the operation needs."""
    n = workspace_size(layout, op, flags)
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or layout.device)


def ef_topk_compress(layout, g, e, idx, val, q, scale, seed, it, flags, workspace, stream=None):
    _check(lib().gc_ef_topk_compress(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(idx), _ptr(val),
                                     _ptr(q), _ptr(scale), int(seed), int(it), int(flags), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "gc_ef_topk_compress")


RESIDUAL_DESC_BYTES = 32


def alloc_residual_desc(layout: Layout, device=None) -> torch.Tensor:
    """Zeroed gc_residual_desc[T] for gc_ef_topk_compress_lazy (no pending selection)."""
    return torch.zeros(layout.T * RESIDUAL_DESC_BYTES, dtype=torch.uint8, device=device or layout.device)


def ef_topk_compress_lazy(layout, g, e, rd, idx, val, q, scale, seed, it, flags, workspace, stream=None):
    _check(lib().gc_ef_topk_compress_lazy(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(rd), _ptr(idx),
                                          _ptr(val), _ptr(q), _ptr(scale), int(seed), int(it), int(flags),
                                          _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_ef_topk_compress_lazy")


def ef_residual_materialize(layout, e, rd, stream=None):
    _check(lib().gc_ef_residual_materialize(layout.dev(), layout.host(), _ptr(e), _ptr(rd), _stream(stream)),
           "gc_ef_residual_materialize")


def ef_topk_compress_clipped(layout, g, e, max_norm, norm, idx, val, q, scale, seed, it, flags, workspace,
                             stream=None):
    _check(lib().gc_ef_topk_compress_clipped(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(max_norm),
                                             _ptr(norm), _ptr(idx), _ptr(val), _ptr(q), _ptr(scale), int(seed),
                                             int(it), int(flags), _ptr(workspace), workspace.numel(),
                                             _stream(stream)), "gc_ef_topk_compress_clipped")


def ef_threshold_compress(layout, g, e, tau, count, idx, val, q, scale, seed, it, flags, workspace, stream=None):
    _check(lib().gc_ef_threshold_compress(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(tau), _ptr(count),
                                          _ptr(idx), _ptr(val), _ptr(q), _ptr(scale), int(seed), int(it),
                                          int(flags), _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_ef_threshold_compress")


WARMUP_KINDS = {"linear": 0, "exponential": 1, "step": 2}


def warmup_density(step, warmup_steps, rho_start, rho_final, kind="exponential", stages=4):
    return float(lib().gc_warmup_density(int(step), int(warmup_steps), float(rho_start), float(rho_final),
                                         WARMUP_KINDS[kind], int(stages)))


def ef_topk_compress_noalloc(layout, g, e, idx, val, q, scale, seed, it, flags, stream=None):
    """gc_ef_topk_compress with the library's built-in scratch instead of a workspace.

    For callers that cannot allocate device memory where they compress; the
    layout's workspace must fit in GC_NOALLOC_MAX_WORKSPACE_BYTES, and calls
    must not overlap on the GPU (they share that scratch).
    """
    _check(lib().gc_ef_topk_compress_noalloc(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(idx),
                                             _ptr(val), _ptr(q), _ptr(scale), int(seed), int(it), int(flags),
                                             _stream(stream)), "gc_ef_topk_compress_noalloc")


def noalloc_device_status(stream=None, raise_on_error=True) -> gc_diag:
    """Diagnostics of the last ef_topk_compress_noalloc call on the current device."""
    d = gc_diag()
    st = lib().gc_ef_topk_compress_noalloc_status(_stream(stream), C.byref(d))
    if st != GC_OK and (raise_on_error or st != GC_ERR_DEVICE):
        raise GCError(st, f"gc_ef_topk_compress_noalloc_status (error bits 0x{d.error_bits:x})")
    return d


def ef_topk_compress_profiled(layout, g, e, idx, val, q, scale, seed, it, flags, workspace, events,
                              stream=None):
    """gc_ef_topk_compress recording `events` (torch.cuda.Event, up to 5) at its phase boundaries."""
    for ev in events:
        if ev is not None and not ev.cuda_event:
            ev.record()          # torch creates its CUDA event lazily, on the first record
    arr = (C.c_void_p * len(events))(*[None if ev is None else ev.cuda_event for ev in events])
    _check(lib().gc_ef_topk_compress_profiled(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(idx),
                                              _ptr(val), _ptr(q), _ptr(scale), int(seed), int(it), int(flags),
                                              _ptr(workspace), workspace.numel(), _stream(stream), arr,
                                              len(events)), "gc_ef_topk_compress_profiled")


def ef_topk_compress_dev_iter(layout, g, e, idx, val, q, scale, seed, iter_dev, flags, workspace, stream=None):
    """ef_topk_compress with the iteration counter in a device int64 tensor
    (`iter_dev`, one element), read by the kernels and advanced by one at
    the end of the call: capturable in a CUDA graph that replays as
    successive steps."""
    _check(lib().gc_ef_topk_compress_dev_iter(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(idx),
                                              _ptr(val), _ptr(q), _ptr(scale), int(seed), _ptr(iter_dev),
                                              int(flags), _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_ef_topk_compress_dev_iter")


def quantize_stochastic_dev_iter(layout, g, e, codes, scale, mode, s_levels, seed, iter_dev, workspace,
                                 stream=None):
    """quantize_stochastic with the iteration counter in a device int64 tensor
    (see ef_topk_compress_dev_iter)."""
    _check(lib().gc_quantize_stochastic_dev_iter(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(codes),
                                                 _ptr(scale), int(mode), int(s_levels), int(seed),
                                                 _ptr(iter_dev), _ptr(workspace), workspace.numel(),
                                                 _stream(stream)),
           "gc_quantize_stochastic_dev_iter")


def ef_topk_compress_momentum(layout, g, u, v, beta, idx, val, q, scale, seed, it, flags, workspace,
                              stream=None):
    _check(lib().gc_ef_topk_compress_momentum(layout.dev(), layout.host(), _ptr(g), _ptr(u), _ptr(v),
                                              float(beta), _ptr(idx), _ptr(val), _ptr(q), _ptr(scale),
                                              int(seed), int(it), int(flags), _ptr(workspace),
                                              workspace.numel(), _stream(stream)),
           "gc_ef_topk_compress_momentum")


def ef_topk_compress_quantized(layout, g, e, idx, val, q, bits, scale, kind, s_levels, seed, it, flags, workspace,
                               stream=None):
    """EF Top-k, then GC_KEPT_INT8 / GC_KEPT_QSGD / GC_KEPT_SIGN of the kept values."""
    _check(lib().gc_ef_topk_compress_quantized(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(idx), _ptr(val),
                                               _ptr(q), _ptr(bits), _ptr(scale), int(kind), int(s_levels), int(seed),
                                               int(it), int(flags), _ptr(workspace), workspace.numel(),
                                               _stream(stream)), "gc_ef_topk_compress_quantized")


def ef_topk_compress_momentum_quantized(layout, g, u, v, beta, idx, val, q, bits, scale, kind, s_levels, seed, it,
                                        flags, workspace, stream=None):
    """Momentum correction + Top-k, then a quantizer of the kept velocity."""
    _check(lib().gc_ef_topk_compress_momentum_quantized(layout.dev(), layout.host(), _ptr(g), _ptr(u), _ptr(v),
                                                        float(beta), _ptr(idx), _ptr(val), _ptr(q), _ptr(bits),
                                                        _ptr(scale), int(kind), int(s_levels), int(seed), int(it),
                                                        int(flags), _ptr(workspace), workspace.numel(),
                                                        _stream(stream)),
           "gc_ef_topk_compress_momentum_quantized")


def sign_compress(layout, g, e, bits, mean_abs, workspace, stream=None):
    _check(lib().gc_sign_compress(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(bits), _ptr(mean_abs),
                                  _ptr(workspace), workspace.numel(), _stream(stream)), "gc_sign_compress")


def sign_compress_lazy(layout, g, e, prev_mean_abs, bits, mean_abs, workspace, stream=None):
    _check(lib().gc_sign_compress_lazy(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(prev_mean_abs),
                                       _ptr(bits), _ptr(mean_abs), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "gc_sign_compress_lazy")


def sign_residual_materialize(layout, e, mean_abs, stream=None):
    _check(lib().gc_sign_residual_materialize(layout.dev(), layout.host(), _ptr(e), _ptr(mean_abs),
                                              _stream(stream)), "gc_sign_residual_materialize")


def quantize_stochastic(layout, g, e, codes, scale, mode, s_levels, seed, it, workspace, stream=None):
    _check(lib().gc_quantize_stochastic(layout.dev(), layout.host(), _ptr(g), _ptr(e), _ptr(codes),
                                        _ptr(scale), int(mode), int(s_levels), int(seed), int(it),
                                        _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_quantize_stochastic")


def _ptr_array(ts):
    if ts is None:
        return None
    arr = (C.c_void_p * len(ts))(*[_ptr(t) for t in ts])
    return arr


def sparse_decompress_accumulate(layout, idx_list, val_list, q_list, scale_list, out, workspace,
                                 stream=None):
    W = len(idx_list)
    ip, vp, qp, sp = _ptr_array(idx_list), _ptr_array(val_list), _ptr_array(q_list), _ptr_array(scale_list)
    _check(lib().gc_sparse_decompress_accumulate(layout.dev(), layout.host(), W, ip, vp, qp, sp, _ptr(out),
                                                 _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_sparse_decompress_accumulate")


def sparse_decompress_accumulate_quantized(layout, kind, s_levels, idx_list, q_list, bits_list, scale_list, out,
                                           workspace, stream=None):
    """Receiver of the GC_KEPT_* payloads of W workers (lists of device tensors)."""
    W = len(idx_list)
    _check(lib().gc_sparse_decompress_accumulate_quantized(layout.dev(), layout.host(), W, int(kind), int(s_levels),
                                                           _ptr_array(idx_list), _ptr_array(q_list),
                                                           _ptr_array(bits_list), _ptr_array(scale_list), _ptr(out),
                                                           _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_sparse_decompress_accumulate_quantized")


def dense_decompress_accumulate(layout, kind, s_levels, data_list, scale_list, out, workspace, stream=None):
    W = len(data_list)
    _check(lib().gc_dense_decompress_accumulate(layout.dev(), layout.host(), W, int(kind), int(s_levels),
                                                _ptr_array(data_list), _ptr_array(scale_list), _ptr(out),
                                                _ptr(workspace), workspace.numel(), _stream(stream)),
           "gc_dense_decompress_accumulate")


def get_device_status(workspace, stream=None, raise_on_error=True) -> gc_diag:
    d = gc_diag()
    st = lib().gc_get_device_status(_ptr(workspace), workspace.numel(), _stream(stream), C.byref(d))
    if st != GC_OK and (raise_on_error or st != GC_ERR_DEVICE):
        raise GCError(st, f"gc_get_device_status (error bits 0x{d.error_bits:x})")
    return d


# ---------------------------------------------------------------------------- convenience

class TopkCompressor:
    """Owns the payload and workspace buffers of gc_ef_topk_compress for one layout."""

    def __init__(self, layout: Layout, flags: int, device="cuda"):
        self.layout, self.flags = layout, flags
        K = layout.total_k
        dev = torch.device(device)
        self.idx = torch.empty(max(K, 1), dtype=torch.int32, device=dev)
        int8 = bool(flags & GC_INT8)
        self.val = None if int8 else torch.empty(max(K, 1), dtype=torch.float32, device=dev)
        self.q = torch.empty(max(K, 1), dtype=torch.int8, device=dev) if int8 else None
        self.scale = torch.empty(layout.T, dtype=torch.float32, device=dev) if int8 else None
        self.workspace = alloc_workspace(layout, GC_OP_TOPK, flags, dev)

    def __call__(self, g, e, seed, it, stream=None):
        ef_topk_compress(self.layout, g, e, self.idx, self.val, self.q, self.scale, seed, it, self.flags,
                         self.workspace, stream)
        return self.idx, self.val, self.q, self.scale
