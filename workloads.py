"""Seeded synthetic inputs for the gradient-compression hot path.

This module is shared by the tests, the oracle checks and the benchmark.  It
holds parameter-list layouts and random-number recipes only: none of the
compression arithmetic lives here.

Layouts are flat fp32 "arenas": tensor t occupies elements [off[t], off[t+1]).
The parameter lists follow the published architectures of ResNet-50,
BERT-large, GPT-2-medium and Llama-3-8B (shapes only; no weights are used).
Gradient distributions stand in for real back-propagated gradients with the
heavy-tailed shape described on the mbrenndoerfer.com "Gradient Compression"
page (section on why gradients are compressible).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


# ----------------------------------------------------------------------------
# layouts
# ----------------------------------------------------------------------------

@dataclass
class Layout:
    name: str
    sizes: list[int]
    kinds: list[str] = field(default_factory=list)   # "w" (weight-like), "bn", "b"
    shapes: list = field(default_factory=list)       # (rows, cols) of each tensor; (n,) for vectors

    @property
    def num_tensors(self) -> int:
        return len(self.sizes)

    @property
    def off(self) -> np.ndarray:
        o = np.zeros(len(self.sizes) + 1, dtype=np.int64)
        o[1:] = np.cumsum(np.asarray(self.sizes, dtype=np.int64))
        return o

    @property
    def numel(self) -> int:
        return int(sum(self.sizes))


def k_per_tensor(sizes, rho: float) -> np.ndarray:
    """k_t = min(n_t, ceil(rho * n_t)), evaluated once on the host in double."""
    return np.asarray([min(int(n), int(math.ceil(rho * float(n)))) for n in sizes], dtype=np.int64)


def prefix(a) -> np.ndarray:
    o = np.zeros(len(a) + 1, dtype=np.int64)
    o[1:] = np.cumsum(np.asarray(a, dtype=np.int64))
    return o


def flat_layout(n: int) -> Layout:
    return Layout("flat", [int(n)], ["w"])


def resnet50_layout() -> Layout:
    sizes, kinds = [], []

    def conv(cin, cout, kh, kw):
        sizes.append(cout * cin * kh * kw); kinds.append("w")

    def bn(c):
        sizes.extend([c, c]); kinds.extend(["bn", "bn"])

    conv(3, 64, 7, 7); bn(64)
    cin = 64
    for planes, blocks in ((64, 3), (128, 4), (256, 6), (512, 3)):
        for b in range(blocks):
            conv(cin, planes, 1, 1); bn(planes)
            conv(planes, planes, 3, 3); bn(planes)
            conv(planes, planes * 4, 1, 1); bn(planes * 4)
            if b == 0:
                conv(cin, planes * 4, 1, 1); bn(planes * 4)
            cin = planes * 4
    sizes.append(1000 * 2048); kinds.append("w")   # fc weight
    sizes.append(1000); kinds.append("w")          # fc bias, scaled like the fc weight
    return Layout("resnet50", sizes, kinds)


def bert_large_layout() -> Layout:
    h, ffn, vocab, layers = 1024, 4096, 30522, 24
    shapes = [(vocab, h), (512, h), (2, h), (h,), (h,)]
    for _ in range(layers):
        for _ in range(4):                     # query, key, value, attention output
            shapes += [(h, h), (h,)]
        shapes += [(h,), (h,)]                 # attention LayerNorm
        shapes += [(ffn, h), (ffn,), (h, ffn), (h,)]   # FFN in / out
        shapes += [(h,), (h,)]                 # output LayerNorm
    shapes += [(h, h), (h,)]                   # pooler
    sizes = [int(np.prod(s)) for s in shapes]
    return Layout("bert_large", sizes, ["w"] * len(sizes), shapes)


def gpt2_medium_layout() -> Layout:
    d, layers, vocab, ctx = 1024, 24, 50257, 1024
    sizes = [vocab * d, ctx * d]
    for _ in range(layers):
        sizes += [d, d]                        # ln_1
        sizes += [d * 3 * d, 3 * d]            # c_attn
        sizes += [d * d, d]                    # attn c_proj
        sizes += [d, d]                        # ln_2
        sizes += [d * 4 * d, 4 * d]            # c_fc
        sizes += [4 * d * d, d]                # mlp c_proj
    sizes += [d, d]                            # ln_f
    return Layout("gpt2_medium", sizes, ["w"] * len(sizes))


def llama3_8b_layout() -> Layout:
    d, ffn, layers, vocab, kv = 4096, 14336, 32, 128256, 1024
    shapes = [(vocab, d)]
    for _ in range(layers):
        shapes += [(d, d), (kv, d), (kv, d), (d, d)]      # q, k, v, o
        shapes += [(ffn, d), (ffn, d), (d, ffn)]          # gate, up, down
        shapes += [(d,), (d,)]                            # two RMSNorm weights
    shapes += [(d,), (vocab, d)]                          # final norm, untied lm_head
    sizes = [int(np.prod(s)) for s in shapes]
    return Layout("llama3_8b", sizes, ["w"] * len(sizes), shapes)


def matrices_of(layout: Layout):
    """(tensor index, rows, cols) of the 2-D tensors of a layout with shapes."""
    return [(t, s[0], s[1]) for t, s in enumerate(layout.shapes) if len(s) == 2]


# ----------------------------------------------------------------------------
# seeded generators (torch; the same recipe on CPU or CUDA)
# ----------------------------------------------------------------------------

def derive_seed(*parts: int) -> int:
    """A 63-bit seed from integer parts (config, iteration, tensor, worker...)."""
    ss = np.random.SeedSequence([int(p) & 0xFFFFFFFF for p in parts])
    return int(ss.generate_state(2, dtype=np.uint64)[0] & np.uint64(0x7FFFFFFFFFFFFFFF))


def _gen(device, *parts) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(derive_seed(*parts))
    return gen


_CHUNK = 1 << 25


def fill_student_t(out: torch.Tensor, nu: float, scale: float, gen: torch.Generator) -> None:
    """out <- scale * Z / sqrt(V / nu), Z ~ N(0,1), V ~ chi^2_nu = 2 Gamma(nu/2)."""
    n = out.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        z = torch.randn(m, generator=gen, device=out.device, dtype=torch.float32)
        a = torch.full((m,), nu / 2.0, device=out.device, dtype=torch.float32)
        v = torch._standard_gamma(a, generator=gen).mul_(2.0 / nu)
        out[s:s + m] = z.div_(v.sqrt_()).mul_(scale)


def fill_laplace(out: torch.Tensor, b: float, gen: torch.Generator) -> None:
    """Laplace(0, b) by inverting its CDF on uniforms in (-1/2, 1/2)."""
    n = out.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        u = torch.rand(m, generator=gen, device=out.device, dtype=torch.float64) - 0.5
        x = -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())
        out[s:s + m] = x.to(torch.float32)


def fill_mixture(out: torch.Tensor, gen: torch.Generator, p_big=1e-3, std_small=1e-4, std_big=1e-2) -> None:
    """Two-component Gaussian mixture; the second BASELINE parameter read as a std."""
    n = out.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        z = torch.randn(m, generator=gen, device=out.device, dtype=torch.float32)
        big = torch.rand(m, generator=gen, device=out.device, dtype=torch.float32) < p_big
        out[s:s + m] = z * torch.where(big, torch.tensor(std_big, device=out.device),
                                       torch.tensor(std_small, device=out.device))


# Per-configuration recipes.  cfg ids: 1 flat 2^20, 2 ResNet-50, 3 BERT-large,
# 4 GPT-2-medium, 5 Llama-3-8B.

LAYOUTS = {1: lambda: flat_layout(1 << 20), 2: resnet50_layout, 3: bert_large_layout,
           4: gpt2_medium_layout, 5: llama3_8b_layout}


def resnet_scales(layout: Layout, cfg_seed: int = 2) -> np.ndarray:
    """Per-tensor Laplace scale b_t: log-uniform in [1e-5, 1e-2], BN tensors 100x."""
    rng = np.random.Generator(np.random.PCG64(derive_seed(cfg_seed, 0xB5)))
    u = rng.uniform(math.log(1e-5), math.log(1e-2), size=layout.num_tensors)
    b = np.exp(u)
    for t, kind in enumerate(layout.kinds):
        if kind == "bn":
            b[t] *= 100.0
    return b


def make_grad(cfg: int, layout: Layout, it: int, device="cpu", worker: int = 0,
              tensors=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Fresh seeded gradient arena for iteration `it` (fp32, flat).

    If `tensors` is given only those tensors are filled (the rest stay zero /
    untouched), which lets a host check regenerate one tensor cheaply.
    """
    off = layout.off
    if out is None:
        out = torch.zeros(layout.numel, dtype=torch.float32, device=device)
    ts = range(layout.num_tensors) if tensors is None else tensors
    scales = resnet_scales(layout) if cfg == 2 else None
    for t in ts:
        view = out[int(off[t]):int(off[t + 1])]
        gen = _gen(out.device, cfg, it, t, worker)
        if cfg in (1, 5):
            fill_student_t(view, 3.0, 1e-3, gen)
        elif cfg == 2:
            fill_laplace(view, float(scales[t]), gen)
        elif cfg == 3:
            fill_student_t(view, 2.5, 1e-3, gen)
        elif cfg == 4:
            fill_mixture(view, gen)
        else:
            raise ValueError(cfg)
    return out


def tensor_grad(cfg: int, layout: Layout, it: int, t: int, device="cpu", worker: int = 0) -> torch.Tensor:
    """Tensor t of the seeded gradient of iteration `it`, alone (same recipe as make_grad)."""
    n = layout.sizes[t]
    out = torch.empty(n, dtype=torch.float32, device=device)
    gen = _gen(out.device, cfg, it, t, worker)
    if cfg in (1, 5):
        fill_student_t(out, 3.0, 1e-3, gen)
    elif cfg == 2:
        fill_laplace(out, float(resnet_scales(layout)[t]), gen)
    elif cfg == 3:
        fill_student_t(out, 2.5, 1e-3, gen)
    elif cfg == 4:
        fill_mixture(out, gen)
    else:
        raise ValueError(cfg)
    return out


def make_sparse_payload(layout: Layout, k: np.ndarray, worker: int, device="cpu", cfg: int = 5,
                        int8: bool = False):
    """A seeded sparse payload for one simulated worker.

    Per tensor: a uniform k_t-subset of local indices in ascending order, with
    Student-t (nu=3, x1e-3) fp32 values, or int8 codes in [-127, 127] plus a
    positive fp32 scale per tensor.  Returns (idx int32, val fp32 | None,
    q int8 | None, scale fp32 | None) as flat tensors over koff.
    """
    koff = prefix(k)
    tot = int(koff[-1])
    idx = torch.empty(tot, dtype=torch.int32, device=device)
    val = None if int8 else torch.empty(tot, dtype=torch.float32, device=device)
    q = torch.empty(tot, dtype=torch.int8, device=device) if int8 else None
    scale = torch.empty(layout.num_tensors, dtype=torch.float32, device=device) if int8 else None
    sizes = layout.sizes
    for t, n in enumerate(sizes):
        kt = int(k[t])
        gen = _gen(device, 0x5A, cfg, worker, t)
        if kt == 0:
            continue
        if kt * 8 >= n:
            sel = torch.randperm(n, generator=gen, device=device)[:kt]
        else:
            # oversample, de-duplicate, then draw exactly k_t of the distinct ones
            sel = torch.empty(0, dtype=torch.int64, device=device)
            while sel.numel() < kt:
                cand = torch.randint(0, n, (int(kt * 1.25) + 64,), generator=gen, device=device)
                sel = torch.unique(torch.cat([sel, cand]))
            pick = torch.randperm(sel.numel(), generator=gen, device=device)[:kt]
            sel = sel[pick]
        sel, _ = torch.sort(sel)
        a, b = int(koff[t]), int(koff[t + 1])
        idx[a:b] = sel.to(torch.int32)
        if int8:
            q[a:b] = torch.randint(-127, 128, (kt,), generator=gen, device=device, dtype=torch.int8)
            u = torch.rand(1, generator=gen, device=device, dtype=torch.float64)
            scale[t] = float(math.exp(math.log(1e-6) + float(u.item()) * math.log(1e3)))
        else:
            fill_student_t(val[a:b], 3.0, 1e-3, gen)
    return idx, val, q, scale
