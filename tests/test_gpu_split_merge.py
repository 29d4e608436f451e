"""GPU parity of the standalone split and merge kernels: bit-exact against the
CPU oracle (laya.cpp docs/vulkan.md, split/merge paragraph: the page's operator
tests compare the two components and the merged FP32 values bit for bit).
NaN outputs are compared by class (both NaN), not by payload."""
import os

import numpy as np
import pytest

from conftest import read_golden

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u32(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


def f16_nan(bits):
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x3FF) != 0)


def assert_split_equal(x_np, hi, lo, orc):
    ohi, olo = orc.split(x_np)
    ghi, glo = u16(hi).reshape(-1), u16(lo).reshape(-1)
    ohi, olo = ohi.reshape(-1), olo.reshape(-1)
    nan_h, nan_l = f16_nan(ohi), f16_nan(olo)
    assert np.array_equal(f16_nan(ghi), nan_h) and np.array_equal(f16_nan(glo), nan_l)
    bad = np.nonzero((ghi != ohi) & ~nan_h)[0]
    assert bad.size == 0, f"hi differs at {bad[:5]}: x={x_np.reshape(-1)[bad[:5]]} gpu={ghi[bad[:5]]} or={ohi[bad[:5]]}"
    bad = np.nonzero((glo != olo) & ~nan_l)[0]
    assert bad.size == 0, f"lo differs at {bad[:5]}: x={x_np.reshape(-1)[bad[:5]]} gpu={glo[bad[:5]]} or={olo[bad[:5]]}"


def test_split_handset_golden(pkg):
    rows = read_golden("split_handset.txt")
    x = torch.from_numpy(np.array([r[0] for r in rows], np.uint32).view(np.int32)).view(torch.float32).cuda()
    hi, lo = pkg.comp_split_f32(x)
    assert [int(v) for v in u16(hi)] == [r[1] for r in rows]
    assert [int(v) for v in u16(lo)] == [r[2] for r in rows]


def test_split_random_bit_patterns(pkg, orc):
    rng = np.random.default_rng(21)
    xb = rng.integers(0, 2**32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    x_np = xb.view(np.float32)
    hi, lo = pkg.comp_split_f32(torch.from_numpy(x_np.copy()).cuda())
    assert_split_equal(x_np, hi, lo, orc)


@pytest.mark.parametrize("name", ["tiny", "encoder", "square", "skinny", "nonaligned"])
def test_split_projection_inputs(pkg, orc, name):
    from compensated_fp32_projection_gb300 import workloads

    x = workloads.make_x(name)
    hi, lo = pkg.comp_split_f32(x.cuda())
    assert tuple(hi.shape) == tuple(x.shape)
    assert_split_equal(x.numpy(), hi, lo, orc)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 31, 1023, 1027, 4099, 65537])
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_split_sizes_and_alignments(pkg, orc, n, offset):
    rng = np.random.default_rng(n * 7 + offset)
    base = torch.from_numpy(rng.normal(0, 100, n + 8).astype(np.float32)).cuda()
    x = base[offset:offset + n]
    hbuf = torch.full((n + 8,), float("nan"), dtype=torch.float16, device="cuda")
    lbuf = torch.full((n + 8,), float("nan"), dtype=torch.float16, device="cuda")
    o2 = (offset * 3) % 4
    hi, lo = pkg.comp_split_f32(x, hbuf[o2:o2 + n], lbuf[offset:offset + n])
    assert_split_equal(x.cpu().numpy(), hi, lo, orc)
    # guard bands untouched
    hb, lb = u16(hbuf), u16(lbuf)
    assert np.all(hb[:o2] == 0x7E00) and np.all(hb[o2 + n:] == 0x7E00)
    assert np.all(lb[:offset] == 0x7E00) and np.all(lb[offset + n:] == 0x7E00)


def _exhaustive_chunks():
    step = int(os.environ.get("COMP_SPLIT_SWEEP_STRIDE", "61"))
    return step


def test_split_sweep_all_fp32_bit_patterns(pkg, orc):
    """Every FP32 bit pattern with stride COMP_SPLIT_SWEEP_STRIDE (default 61,
    coprime with every power of two, so all low-bit residues appear); set it
    to 1 for the exhaustive 2^32 sweep."""
    step = _exhaustive_chunks()
    chunk = 1 << 26
    total = 1 << 32
    start = 0
    while start < total:
        idx = np.arange(start, min(total, start + chunk * step), step, dtype=np.uint64)
        x_np = idx.astype(np.uint32).view(np.float32)
        hi, lo = pkg.comp_split_f32(torch.from_numpy(x_np.copy()).cuda())
        assert_split_equal(x_np, hi, lo, orc)
        start += chunk * step


def test_merge_golden(pkg):
    rows = read_golden("merge_special.txt")
    a = torch.from_numpy(np.array([r[0] for r in rows], np.uint32).view(np.int32)).view(torch.float32).cuda()
    b = torch.from_numpy(np.array([r[1] for r in rows], np.uint32).view(np.int32)).view(torch.float32).cuda()
    y = pkg.comp_merge_f32(a, b)
    assert [int(v) for v in u32(y)] == [r[2] for r in rows]


def _merge_inputs(n, seed):
    rng = np.random.default_rng(seed)
    scale = 2.0 ** rng.integers(-140, 120, n)
    a = (rng.normal(0, 1, n) * scale).astype(np.float32)
    with np.errstate(over="ignore"):
        b = (rng.normal(0, 1, n) * scale * 2.0 ** rng.integers(-20, 20, n)).astype(np.float32)
    bits = rng.integers(0, 2**32, n // 4, dtype=np.uint64).astype(np.uint32).view(np.float32)
    a[: n // 4] = bits
    b[n // 4: n // 4 + bits.size] = bits
    return a, b


def assert_merge_equal(a, b, y, orc):
    ref = orc.merge(a, b)
    g = y.detach().cpu().numpy().reshape(-1)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(g), nan)
    bad = np.nonzero((g.view(np.uint32) != ref.view(np.uint32)) & ~nan)[0]
    assert bad.size == 0, f"merge differs at {bad[:5]}"


def test_merge_random(pkg, orc):
    a, b = _merge_inputs(1 << 22, 31)
    y = pkg.comp_merge_f32(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    assert_merge_equal(a, b, y, orc)


@pytest.mark.parametrize("n", [1, 3, 4, 5, 1027, 65539])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_merge_sizes_and_alignments(pkg, orc, n, offset):
    a, b = _merge_inputs(n + 8, n + offset)
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ybuf = torch.full((n + 8,), float("nan"), dtype=torch.float32, device="cuda")
    y = pkg.comp_merge_f32(ta[offset:offset + n], tb[:n], ybuf[(offset + 1) % 4:(offset + 1) % 4 + n])
    assert_merge_equal(a[offset:offset + n], b[:n], y, orc)
    yb = u32(ybuf)
    o = (offset + 1) % 4
    assert np.all(yb[:o] == 0x7FC00000) and np.all(yb[o + n:] == 0x7FC00000)


def test_merge_in_place(pkg, orc):
    a, b = _merge_inputs(1 << 16, 41)
    ta, tb = torch.from_numpy(a.copy()).cuda(), torch.from_numpy(b.copy()).cuda()
    pkg.comp_merge_f32(ta, tb, ta)  # y is acc_hi
    assert_merge_equal(a, b, ta, orc)
    ta, tb = torch.from_numpy(a.copy()).cuda(), torch.from_numpy(b.copy()).cuda()
    pkg.comp_merge_f32(ta, tb, tb)  # y is acc_lo
    assert_merge_equal(a, b, tb, orc)


def test_merge_rejects_partial_overlap(pkg):
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(pkg.CompError):
        pkg.comp_merge_f32(buf[:32], buf[32:], buf[1:33])


def test_split_then_merge_reconstructs(pkg):
    x = torch.randn(1 << 20, device="cuda") * 1000
    hi, lo = pkg.comp_split_f32(x)
    y = pkg.comp_merge_f32(hi.float(), lo.float())
    xd = x.double()
    assert torch.all((y.double() - xd).abs() <= 2.0**-22 * xd.abs() + 2.0**-35)


# Beyond 2^31 elements (64-bit indexing in the grid-stride loops), odd so that
# the scalar tail runs too; inputs drawn on the device, ~1 M sampled indices
# (the first, the last and random ones) checked against the oracle.
N_BIG = (1 << 31) + 8191


def _big_sample(n):
    rng = np.random.default_rng(31)
    idx = np.concatenate([np.arange(4096), np.arange(n - 16384, n), rng.integers(0, n, 1 << 20)])
    return torch.from_numpy(np.unique(idx).astype(np.int64))


def test_split_beyond_2_31_elements(pkg, orc):
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn(N_BIG, device="cuda", generator=g) * 100
    hi, lo = pkg.comp_split_f32(x)
    idx = _big_sample(N_BIG).cuda()
    x_np = x[idx].cpu().numpy()
    assert_split_equal(x_np, hi[idx].cpu(), lo[idx].cpu(), orc)
    del x, hi, lo
    torch.cuda.empty_cache()


def test_merge_beyond_2_31_elements(pkg, orc):
    g = torch.Generator(device="cuda").manual_seed(6)
    a = torch.randn(N_BIG, device="cuda", generator=g)
    b = torch.randn(N_BIG, device="cuda", generator=g) * 1e3
    y = pkg.comp_merge_f32(a, b)
    idx = _big_sample(N_BIG).cuda()
    ref = orc.merge(a[idx].cpu().numpy(), b[idx].cpu().numpy())
    assert np.array_equal(y[idx].cpu().numpy().view(np.uint32), ref.view(np.uint32))
    del a, b, y
    torch.cuda.empty_cache()


def test_device_status_clean(pkg):
    st, where = pkg.device_status()
    assert st == 0 and where == 0
