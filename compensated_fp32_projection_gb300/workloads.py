"""Seeded synthetic inputs for the compensated-FP32 projection.

This module only draws random numbers: it holds none of the method's
arithmetic.  The tests, the benchmark and the oracle checks all take their
inputs from here.

Five projection shapes (x FP32 [M, K], W FP16 [N, K], y FP32 [M, N]):

* ``tiny``        8 x 384 x 256, x ~ N(0, 1) with 16 hand-set values in x[0, 0:16]
                  (exact FP16 values, ties, subnormals, values near +-65504 and
                  +-60000, and ties above 32,000 — the kinds of value the laya.cpp
                  page's operator tests name);
* ``encoder``     512 x 1024 x 1024, x ~ N(0, 1) with exactly round(0.01*M*K)
                  entries (seeded permutation) multiplied by 100;
* ``square``      4096 x 4096 x 4096, x ~ N(0, 1);
* ``skinny``      16 x 14336 x 4096, x ~ N(0, 1) (decode-shaped);
* ``nonaligned``  1000 x 771 x 1027, each x entry independently with
                  probability 0.25 from N(0, 1e-6), else uniform in [-6e4, 6e4].

W is drawn in FP32 from N(0, 0.02) (0.02 is the standard deviation) and
rounded to FP16 with round-to-nearest-even (``Tensor.half()`` on the CPU).
Config i is seeded with 20261202 + i on a CPU ``torch.Generator``.
"""
from __future__ import annotations

import hashlib
import struct
from dataclasses import dataclass

import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Shape:
    name: str
    index: int
    M: int
    N: int
    K: int

    @property
    def flops(self) -> int:
        """Effective FP32 GEMM work, 2*M*N*K."""
        return 2 * self.M * self.N * self.K

    @property
    def fused_bytes(self) -> int:
        """Algorithmic HBM bytes of the fused product: x read, W read, y written once."""
        return 4 * self.M * self.K + 2 * self.N * self.K + 4 * self.M * self.N


SHAPES = {
    s.name: s
    for s in (
        Shape("tiny", 0, 8, 384, 256),
        Shape("encoder", 1, 512, 1024, 1024),
        Shape("square", 2, 4096, 4096, 4096),
        Shape("skinny", 3, 16, 14336, 4096),
        Shape("nonaligned", 4, 1000, 771, 1027),
    )
}


def _f32(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


# The 16 hand-set activations placed in x[0, 0:16] of the tiny shape, as FP32
# bit patterns.  What each one exercises is listed beside it.
HAND_SET_BITS = (
    0x3F800000,  # 1.0: exact in FP16, residual zero
    0xC0200000,  # -2.5: exact negative
    0x476A6000,  # 60000.0: large activation, exact in FP16
    0xC76A6000,  # -60000.0
    0x477FE000,  # 65504.0: largest finite FP16
    0xC77FEFFF,  # -65519.996: just below the overflow tie, largest residual
    0x80000000,  # -0.0: signed zero
    0x3F801000,  # 1 + 2^-11: tie, rounds down to even
    0x3F803000,  # 1 + 3*2^-11: tie, rounds up to even
    0x47001000,  # 32784: tie above 32,000, down
    0x47003000,  # 32816: tie above 32,000, up
    0x33800000,  # 2^-24: smallest FP16 subnormal
    0x33000000,  # 2^-25: subnormal tie to zero
    0x33400000,  # 3*2^-26: subnormal rounding up
    0x358637BD,  # 1e-6: FP16-subnormal hi and lo
    0x800116C2,  # -1e-40: FP32 subnormal, sign kept, no flush to zero
)
HAND_SET = tuple(_f32(b) for b in HAND_SET_BITS)


def _gen(shape: Shape) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + shape.index)
    return g


def make_x(shape: Shape | str, g: torch.Generator | None = None) -> torch.Tensor:
    """The activation matrix x, FP32 [M, K], on the CPU."""
    s = SHAPES[shape] if isinstance(shape, str) else shape
    g = g or _gen(s)
    M, K = s.M, s.K
    if s.name == "nonaligned":
        big = torch.rand((M, K), generator=g, dtype=torch.float32) * 1.2e5 - 6e4
        small = torch.randn((M, K), generator=g, dtype=torch.float32) * 1e-6
        pick = torch.rand((M, K), generator=g, dtype=torch.float32) < 0.25
        return torch.where(pick, small, big).contiguous()
    x = torch.randn((M, K), generator=g, dtype=torch.float32)
    if s.name == "encoder":
        count = round(0.01 * M * K)
        idx = torch.randperm(M * K, generator=g)[:count]
        flat = x.view(-1)
        flat[idx] = flat[idx] * 100.0
    if s.name == "tiny":
        x[0, : len(HAND_SET)] = torch.tensor(HAND_SET, dtype=torch.float32)
    return x.contiguous()


def make_w(shape: Shape | str, g: torch.Generator | None = None) -> torch.Tensor:
    """The weight matrix W, FP16 [N, K], on the CPU (drawn FP32, rounded RNE)."""
    s = SHAPES[shape] if isinstance(shape, str) else shape
    g = g or _gen(s)
    return (torch.randn((s.N, s.K), generator=g, dtype=torch.float32) * 0.02).half().contiguous()


def make_inputs(shape: Shape | str) -> tuple[torch.Tensor, torch.Tensor]:
    """(x, W) for a shape, drawn from one generator in a fixed order."""
    s = SHAPES[shape] if isinstance(shape, str) else shape
    g = _gen(s)
    x = make_x(s, g)
    W = make_w(s, g)
    return x, W


def random_case(M: int, N: int, K: int, seed: int, scale: float = 1.0) -> tuple[torch.Tensor, torch.Tensor]:
    """A generic (x, W) pair for odd sizes: x ~ N(0, scale), W ~ N(0, 0.02) as FP16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, dtype=torch.float32) * scale
    W = (torch.randn((N, K), generator=g, dtype=torch.float32) * 0.02).half()
    return x.contiguous(), W.contiguous()


def random_bits_f32(n: int, seed: int) -> torch.Tensor:
    """n uniformly random FP32 bit patterns (every class: zeros, subnormals, inf, NaN)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b = torch.randint(-(2**31), 2**31, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    return b.view(torch.float32)


def special_values_f32(n: int, seed: int) -> torch.Tensor:
    """n finite FP32 values below 65504 in magnitude that stress an FP16 split:
    a quarter are the midpoints between neighbouring FP16 values (ties) or the
    FP32 values just beside them; 1000 lie in [65000, 65504]; 1000 are drawn
    from N(0, 1e-6) (FP16-subnormal hi and lo); the rest are random bit
    patterns with binary exponents -30 .. 14 (2^-30 <= |x| < 32768, so FP16
    subnormals as well as normals).  Signs random."""
    g = torch.Generator().manual_seed(seed)
    ri = lambda hi, size: torch.randint(0, hi, size, generator=g, dtype=torch.int64)  # noqa: E731
    bits = (ri(2, (n,)) << 31) | ((97 + ri(45, (n,))) << 23) | ri(1 << 23, (n,))
    x = bits.to(torch.int64).to(torch.int32).view(torch.float32).clone()
    k = n // 4
    h = ri(0x7bff, (k,)).to(torch.int16).view(torch.float16)  # finite, positive, below 65504
    up = (h.view(torch.int16) + 1).view(torch.float16)        # the next FP16 value up
    mid = ((h.double() + up.double()) / 2).float()            # an exact tie in FP32
    side = ri(3, (k,))
    mid = torch.where(side == 1, torch.nextafter(mid, torch.full_like(mid, float("inf"))), mid)
    mid = torch.where(side == 2, torch.nextafter(mid, torch.zeros_like(mid)), mid)
    x[:k] = mid * torch.where(ri(2, (k,)) == 0, 1.0, -1.0)
    x[k:k + 1000] = torch.linspace(65000.0, 65504.0, 1000)
    x[k + 1000:k + 2000] = torch.randn(1000, generator=g) * 1e-6
    return x


def sha256(t: torch.Tensor) -> str:
    return hashlib.sha256(t.contiguous().view(torch.uint8).numpy().tobytes()).hexdigest()
