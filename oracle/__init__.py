"""Oracle for error-feedback gradient compression: TEST INFRASTRUCTURE.

A plain single-threaded C++ implementation (oracle.cpp) wrapped for numpy.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
it; the GPU library never imports, links or calls anything here, and this
package imports nothing from the GPU library.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build_mod

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build_mod.build())
        _declare(_lib)
    return _lib


_P = C.c_void_p
_I64, _I32, _U64, _U32, _F = C.c_int64, C.c_int32, C.c_uint64, C.c_uint32, C.c_float


def _declare(L):
    L.oracle_philox4x32_10.argtypes = [_P, _P, _P]
    L.oracle_draw_u32.argtypes = [_U64, _U64, _U64, _I64, _U32, _P]
    L.oracle_stochastic_round.argtypes = [_F, _U32]
    L.oracle_stochastic_round.restype = C.c_double
    L.oracle_select.argtypes = [_I64, _I64, _P, _I32, _I32, _P]
    L.oracle_ef_topk_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _P, _P, _P, _P, _U64, _U64, _I32, _I32]
    L.oracle_clip_topk_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _F, _P, _P, _P, _P, _P, _P, _U64, _U64, _I32]
    L.oracle_powersgd_tensor.argtypes = [_I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _P, _P]
    L.oracle_powersgd_decode_accumulate.argtypes = [_I64, _I64, _I32, _P, _P, _P]
    L.oracle_threshold_tensor.argtypes = [_I64, _I64, _F, _U64, _P, _P, _P, _P, _P, _P, _P, _U64, _U64, _I32]
    L.oracle_randk_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _P, _P, _U64, _U64, _I32, _I32]
    L.oracle_momentum_topk_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _P, _F, _I32, _P, _P, _P, _P,
                                              _U64, _U64, _I32, _I32]
    L.oracle_sign_tensor.argtypes = [_I64, _P, _P, _P, _P, _P]
    L.oracle_ef_topk_quantized_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32,
                                                  _U64, _U64, _I32]
    L.oracle_momentum_topk_quantized_tensor.argtypes = [_I64, _I64, _U64, _P, _P, _P, _F, _I32, _P, _P, _P, _P,
                                                        _P, _P, _I32, _I32, _U64, _U64, _I32]
    L.oracle_quantize_tensor.argtypes = [_I64, _U64, _P, _P, _P, _P, _I32, _I32, _U64, _U64, _P]
    L.oracle_sparse_accumulate.argtypes = [_I32, _P, _P, _I32, _P, _P, _P, _P, _P]
    L.oracle_sparse_accumulate_quantized.argtypes = [_I32, _P, _P, _I32, _P, _P, _P, _P, _I32, _I32, _P]
    L.oracle_sign_decode_accumulate.argtypes = [_I64, _P, _F, _P]
    L.oracle_warmup_density.argtypes = [_I64, _I64, C.c_double, C.c_double, _I32, _I32]
    L.oracle_warmup_density.restype = C.c_double
    L.oracle_codes_decode_accumulate.argtypes = [_I64, _P, _F, _I32, _I32, _P]
    for name in ("oracle_select", "oracle_ef_topk_tensor", "oracle_randk_tensor", "oracle_threshold_tensor", "oracle_clip_topk_tensor",
                 "oracle_powersgd_tensor", "oracle_powersgd_decode_accumulate",
                 "oracle_momentum_topk_tensor", "oracle_sign_tensor", "oracle_quantize_tensor",
                 "oracle_ef_topk_quantized_tensor", "oracle_momentum_topk_quantized_tensor",
                 "oracle_sparse_accumulate", "oracle_sparse_accumulate_quantized",
                 "oracle_sign_decode_accumulate",
                 "oracle_codes_decode_accumulate"):
        getattr(L, name).restype = C.c_int


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# --------------------------------------------------------------------------- Philox

def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32); k = _c(key, np.uint32); o = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(o))
    return o


def draw_u32(seed: int, it: int, first: int, count: int, purpose: int) -> np.ndarray:
    o = np.zeros(count, np.uint32)
    lib().oracle_draw_u32(seed, it, first, count, purpose, _p(o))
    return o


def stochastic_round(x: float, r: int) -> float:
    return lib().oracle_stochastic_round(float(x), int(r))


# --------------------------------------------------------------------------- selection

def select(key, k: int, largest: bool = True, method: int = 1) -> np.ndarray:
    key = _c(key, np.uint32)
    out = np.zeros(max(k, 0), np.int64)
    _check(lib().oracle_select(key.size, k, _p(key), int(largest), method, _p(out)), "select")
    return out


# --------------------------------------------------------------------------- per tensor

def ef_topk_tensor(g, e, k, base=0, int8=False, seed=0, it=0, method=1):
    """Returns (idx, val, q, scale); e (if given) is updated in place."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    q = np.zeros(k, np.int8) if int8 else None
    sc = np.zeros(1, np.float32) if int8 else None
    _check(lib().oracle_ef_topk_tensor(n, k, base, _p(g), _p(e), _p(idx), _p(val), _p(q), _p(sc),
                                       seed, it, int(int8), method), "ef_topk")
    return idx, val, q, (float(sc[0]) if int8 else None)


def clip_topk_tensor(g, e, k, max_norm, base=0, int8=False, seed=0, it=0, norm_given=None):
    """Returns (idx, val, q, scale, norm computed)."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    q = np.zeros(k, np.int8) if int8 else None
    sc = np.zeros(1, np.float32) if int8 else None
    nout = np.zeros(1, np.float32)
    ng = None if norm_given is None else np.asarray([norm_given], np.float32)
    _check(lib().oracle_clip_topk_tensor(n, k, base, _p(g), _p(e), float(max_norm), _p(ng), _p(nout), _p(idx),
                                         _p(val), _p(q), _p(sc), seed, it, int(int8)), "clip_topk")
    return idx, val, q, (float(sc[0]) if int8 else None), float(nout[0])


def powersgd_tensor(g, e, q, r, p_raw_given=None, p_given=None, q_given=None):
    """One PowerSGD step on an m x n matrix.  g, e: (m, n) fp32 (e updated in
    place); q: (n, r) fp32 warm start, updated in place.  Returns (p, p_raw)."""
    g = _c(g, np.float32)
    m, n = g.shape
    assert e.dtype == np.float32 and e.flags.c_contiguous and e.shape == (m, n)
    assert q.dtype == np.float32 and q.flags.c_contiguous and q.shape == (n, r)
    p = np.zeros((m, r), np.float32); p_raw = np.zeros((m, r), np.float32)
    pr = None if p_raw_given is None else _c(p_raw_given, np.float32)
    pg = None if p_given is None else _c(p_given, np.float32)
    qg = None if q_given is None else _c(q_given, np.float32)
    _check(lib().oracle_powersgd_tensor(m, n, r, _p(g), _p(e), _p(q), _p(p), _p(p_raw), _p(pr), _p(pg), _p(qg)),
           "powersgd")
    return p, p_raw


def powersgd_decode_accumulate(p, q, out):
    m, r = p.shape
    n = q.shape[0]
    _check(lib().oracle_powersgd_decode_accumulate(m, n, r, _p(_c(p, np.float32)), _p(_c(q, np.float32)), _p(out)),
           "powersgd_decode")
    return out


def threshold_tensor(g, e, kmax, tau, base=0, int8=False, seed=0, it=0):
    """Returns (idx, val, q, scale, count); idx/val/q hold `count` entries."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    idx = np.zeros(kmax, np.int32); val = np.zeros(kmax, np.float32)
    q = np.zeros(kmax, np.int8) if int8 else None
    sc = np.zeros(1, np.float32) if int8 else None
    cnt = np.zeros(1, np.int64)
    _check(lib().oracle_threshold_tensor(n, kmax, float(tau), base, _p(g), _p(e), _p(idx), _p(val), _p(q), _p(sc),
                                         _p(cnt), seed, it, int(int8)), "threshold")
    c = int(cnt[0])
    return idx[:c], val[:c], (q[:c] if int8 else None), (float(sc[0]) if int8 else None), c


def warmup_density(step, warmup_steps, rho_start, rho_final, kind):
    """Density of the warm-up schedule (see oracle_warmup_density)."""
    return lib().oracle_warmup_density(int(step), int(warmup_steps), float(rho_start), float(rho_final),
                                       {"linear": 0, "exponential": 1, "step": 2}[kind], 4)


def randk_tensor(g, e, k, base=0, seed=0, it=0, unbiased=False, method=1):
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    _check(lib().oracle_randk_tensor(n, k, base, _p(g), _p(e), _p(idx), _p(val), seed, it,
                                     int(unbiased), method), "randk")
    return idx, val


def momentum_topk_tensor(g, u, v, k, beta, masking=True, base=0, int8=False, seed=0, it=0, method=1):
    g = _c(g, np.float32); n = g.size
    for a in (u, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    q = np.zeros(k, np.int8) if int8 else None
    sc = np.zeros(1, np.float32) if int8 else None
    _check(lib().oracle_momentum_topk_tensor(n, k, base, _p(g), _p(u), _p(v), float(beta), int(masking),
                                             _p(idx), _p(val), _p(q), _p(sc), seed, it, int(int8), method),
           "momentum")
    return idx, val, q, (float(sc[0]) if int8 else None)


KEPT_KINDS = {"qsgd": 2, "sign": 3}


def _kept_buffers(k, kind):
    q = np.zeros(k, np.int8) if kind == "qsgd" else None
    bits = np.zeros((k + 31) // 32, np.uint32) if kind == "sign" else None
    return q, bits


def ef_topk_quantized_tensor(g, e, k, kind, s_levels=16, base=0, seed=0, it=0, scale_given=None, method=1):
    """EF Top-k, then QSGD ('qsgd') or sign ('sign') of the kept values.
    Returns (idx, decoded values, codes or None, bits or None, scale computed);
    e (if given) is updated in place."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    q, bits = _kept_buffers(k, kind)
    sc = np.zeros(1, np.float32)
    sg = None if scale_given is None else np.asarray([scale_given], np.float32)
    _check(lib().oracle_ef_topk_quantized_tensor(n, k, base, _p(g), _p(e), _p(idx), _p(val), _p(q), _p(bits),
                                                 _p(sc), _p(sg), KEPT_KINDS[kind], s_levels, seed, it, method),
           "ef_topk_quantized")
    return idx, val, q, bits, float(sc[0])


def momentum_topk_quantized_tensor(g, u, v, k, beta, kind, s_levels=16, masking=True, base=0, seed=0, it=0,
                                   scale_given=None, method=1):
    """Momentum correction + Top-k, then QSGD or sign of the kept velocity.
    Returns (idx, decoded values, codes or None, bits or None, scale computed)."""
    g = _c(g, np.float32); n = g.size
    for a in (u, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
    idx = np.zeros(k, np.int32); val = np.zeros(k, np.float32)
    q, bits = _kept_buffers(k, kind)
    sc = np.zeros(1, np.float32)
    sg = None if scale_given is None else np.asarray([scale_given], np.float32)
    _check(lib().oracle_momentum_topk_quantized_tensor(n, k, base, _p(g), _p(u), _p(v), float(beta), int(masking),
                                                       _p(idx), _p(val), _p(q), _p(bits), _p(sc), _p(sg),
                                                       KEPT_KINDS[kind], s_levels, seed, it, method),
           "momentum_topk_quantized")
    return idx, val, q, bits, float(sc[0])


def sign_tensor(g, e, mu_given=None):
    """Returns (bits uint32[ceil(n/32)], mu computed); e updated in place."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    bits = np.zeros((n + 31) // 32, np.uint32); mu = np.zeros(1, np.float32)
    mg = None if mu_given is None else np.asarray([mu_given], np.float32)
    _check(lib().oracle_sign_tensor(n, _p(g), _p(e), _p(bits), _p(mu), _p(mg)), "sign")
    return bits, float(mu[0])


def quantize_tensor(g, e, mode, s_levels=16, base=0, seed=0, it=0, scale_given=None):
    """mode 'int8' or 'qsgd'.  Returns (codes int8[n], scale computed)."""
    g = _c(g, np.float32); n = g.size
    if e is not None:
        assert e.dtype == np.float32 and e.flags.c_contiguous and e.size == n
    codes = np.zeros(n, np.int8); sc = np.zeros(1, np.float32)
    sg = None if scale_given is None else np.asarray([scale_given], np.float32)
    m = {"int8": 0, "qsgd": 1}[mode]
    _check(lib().oracle_quantize_tensor(n, base, _p(g), _p(e), _p(codes), _p(sc), m, s_levels,
                                        seed, it, _p(sg)), "quantize")
    return codes, float(sc[0])


# --------------------------------------------------------------------------- receivers

def sparse_accumulate(off, koff, idx_list, val_list, q_list, scale_list, out):
    off = _c(off, np.int64); koff = _c(koff, np.int64)
    T = off.size - 1; W = len(idx_list)
    idxs = [_c(a, np.int32) for a in idx_list]
    ip = (C.c_void_p * W)(*[a.ctypes.data for a in idxs])
    vp = qp = sp = None
    keep = []
    if val_list is not None:
        vals = [_c(a, np.float32) for a in val_list]; keep += vals
        vp = (C.c_void_p * W)(*[a.ctypes.data for a in vals])
    else:
        qs = [_c(a, np.int8) for a in q_list]; ss = [_c(a, np.float32) for a in scale_list]
        keep += qs + ss
        qp = (C.c_void_p * W)(*[a.ctypes.data for a in qs])
        sp = (C.c_void_p * W)(*[a.ctypes.data for a in ss])
    assert out.dtype == np.float32 and out.flags.c_contiguous
    _check(lib().oracle_sparse_accumulate(T, _p(off), _p(koff), W, ip, vp, qp, sp, _p(out)), "sparse_accumulate")
    return out


def sparse_accumulate_quantized(off, koff, kind, idx_list, q_list, bits_list, scale_list, out, s_levels=16):
    """kind 'int8', 'qsgd' or 'sign': the receiver of the quantized kept-value payloads."""
    off = _c(off, np.int64); koff = _c(koff, np.int64)
    T = off.size - 1; W = len(idx_list)
    keep = [_c(a, np.int32) for a in idx_list]
    ip = (C.c_void_p * W)(*[a.ctypes.data for a in keep])
    qp = bp = None
    if q_list is not None:
        qs = [_c(a, np.int8) for a in q_list]; keep += qs
        qp = (C.c_void_p * W)(*[a.ctypes.data for a in qs])
    if bits_list is not None:
        bs = [_c(a, np.uint32) for a in bits_list]; keep += bs
        bp = (C.c_void_p * W)(*[a.ctypes.data for a in bs])
    ss = [_c(a, np.float32) for a in scale_list]; keep += ss
    sp = (C.c_void_p * W)(*[a.ctypes.data for a in ss])
    assert out.dtype == np.float32 and out.flags.c_contiguous
    k = {"int8": 1, "qsgd": 2, "sign": 3}[kind]
    _check(lib().oracle_sparse_accumulate_quantized(T, _p(off), _p(koff), W, ip, qp, bp, sp, k, s_levels, _p(out)),
           "sparse_accumulate_quantized")
    return out


def sign_decode_accumulate(bits, mu, out):
    bits = _c(bits, np.uint32)
    _check(lib().oracle_sign_decode_accumulate(out.size, _p(bits), float(mu), _p(out)), "sign_decode")
    return out


def codes_decode_accumulate(codes, scale, mode, out, s_levels=16):
    codes = _c(codes, np.int8)
    m = {"int8": 0, "qsgd": 1}[mode]
    _check(lib().oracle_codes_decode_accumulate(out.size, _p(codes), float(scale), m, s_levels, _p(out)),
           "codes_decode")
    return out


# --------------------------------------------------------------------------- layouts

def ef_topk_layout(off, k, g, e, int8=False, seed=0, it=0, method=1):
    """Whole arena, tensor by tensor.  Returns (idx, val, q, scale[T])."""
    off = np.asarray(off, np.int64); k = np.asarray(k, np.int64)
    T = off.size - 1
    koff = np.zeros(T + 1, np.int64); koff[1:] = np.cumsum(k)
    idx = np.zeros(int(koff[-1]), np.int32); val = np.zeros(int(koff[-1]), np.float32)
    q = np.zeros(int(koff[-1]), np.int8) if int8 else None
    sc = np.zeros(T, np.float32) if int8 else None
    for t in range(T):
        a, b = int(off[t]), int(off[t + 1])
        et = e[a:b] if e is not None else None
        i, v, qq, s = ef_topk_tensor(g[a:b], et, int(k[t]), base=a, int8=int8, seed=seed, it=it, method=method)
        idx[koff[t]:koff[t + 1]] = i; val[koff[t]:koff[t + 1]] = v
        if int8:
            q[koff[t]:koff[t + 1]] = qq; sc[t] = s
    return idx, val, q, sc
