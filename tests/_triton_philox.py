"""Runs Triton's Philox4x32 rounds in Triton's CPU interpreter (library pin).

Reads whitespace-separated hex words from stdin, six per line
(c0 c1 c2 c3 k0 k1), prints four hex words per line.  Must be started with
TRITON_INTERPRET=1 in the environment.
"""
import sys

import torch
import triton
import triton.language as tl
from triton.language.random import philox_impl


@triton.jit
def _kernel(cp, kp, op, N: tl.constexpr):
    offs = tl.arange(0, N)
    c0 = tl.load(cp + 4 * offs + 0).to(tl.uint32)
    c1 = tl.load(cp + 4 * offs + 1).to(tl.uint32)
    c2 = tl.load(cp + 4 * offs + 2).to(tl.uint32)
    c3 = tl.load(cp + 4 * offs + 3).to(tl.uint32)
    k0 = tl.load(kp + 2 * offs + 0).to(tl.uint32)
    k1 = tl.load(kp + 2 * offs + 1).to(tl.uint32)
    r0, r1, r2, r3 = philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(op + 4 * offs + 0, r0.to(tl.int64))
    tl.store(op + 4 * offs + 1, r1.to(tl.int64))
    tl.store(op + 4 * offs + 2, r2.to(tl.int64))
    tl.store(op + 4 * offs + 3, r3.to(tl.int64))


def main():
    rows = [[int(w, 16) for w in line.split()] for line in sys.stdin if line.strip()]
    n = 1
    while n < len(rows):
        n *= 2
    rows += [[0] * 6] * (n - len(rows))
    c = torch.tensor([r[:4] for r in rows], dtype=torch.int64)
    k = torch.tensor([r[4:] for r in rows], dtype=torch.int64)
    o = torch.zeros(n, 4, dtype=torch.int64)
    _kernel[(1,)](c, k, o, N=n)
    for r in o.tolist():
        print(" ".join("%08x" % (v & 0xFFFFFFFF) for v in r))


if __name__ == "__main__":
    main()
