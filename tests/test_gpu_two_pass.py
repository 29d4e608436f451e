"""GPU parity of the two-pass compensated projection: the split as its own
dispatch (laya.cpp docs/vulkan.md, split/merge paragraph) followed by the two
FP16 products and the merge (compensated-FP32 paragraph), through
comp_gemm_f32x16_ws and comp_gemm_f16x2.  Same gate as the fused kernel:
elementwise within 4e-6 * sum|x||w| of the oracle and 100x more accurate than
a single FP16 cast of x.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gemm_check import check_comp, sample_outputs  # noqa: E402


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def bits(t):
    return t.contiguous().view(torch.int32)


@pytest.mark.parametrize("name", ["tiny", "encoder"])
def test_shapes_full(pkg, orc, name):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs(name)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.parametrize("name", ["square", "skinny"])
def test_shapes_sampled(pkg, orc, name):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs(name)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    r, c = sample_outputs(x.shape[0], W.shape[0])
    e_gpu, e_cast = check_comp(y, x, W, orc, r, c)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
    assert torch.isfinite(y).all()


def test_nonaligned_k_takes_the_padded_two_pass_form(pkg, orc):
    # K = 1027 is not a multiple of 8: with the workspace of
    # comp_gemm_workspace_bytes_mnk the planes and a copy of W are padded to
    # K = 1032 with zeros; with a workspace of only 4*M*K the call is exactly
    # the fused kernel
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("nonaligned")
    M, K = x.shape
    N = W.shape[0]
    xd, Wd = x.cuda(), W.cuda()
    y_pad = pkg.comp_gemm_f32x16_ws(xd, Wd)
    e_gpu, e_cast = check_comp(y_pad, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
    small = torch.empty(pkg.comp_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y_small = pkg.comp_gemm_f32x16_ws(xd, Wd, workspace=small)
    y_fused = pkg.comp_gemm_f32x16(xd, Wd)
    assert torch.equal(bits(y_small), bits(y_fused))


@pytest.mark.parametrize("shape", [(129, 257, 1027), (3, 5, 7), (300, 520, 1001), (2048, 2048, 333)],
                         ids=lambda s: "x".join(map(str, s)))
def test_padded_two_pass_shapes(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + N + K, scale=2.0)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    check_comp(y, x, W, orc)


def test_misaligned_w_takes_the_padded_form(pkg, orc):
    # K a multiple of 8 but W 2 bytes off a 16-byte boundary: W cannot be read
    # with the tensor memory accelerator, so it is copied (padded form)
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 130, 300, 72
    x, W = workloads.random_case(M, N, K, seed=5)
    big = torch.empty(N * K + 8, dtype=torch.float16, device="cuda")
    Wd = big[1:1 + N * K].view(N, K)
    Wd.copy_(W.cuda())
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), Wd)
    check_comp(y, x, W, orc)


# K multiples of 8 only (the planes are read with the tensor memory accelerator);
# ragged M, N and K tails, one and several 128-row / 128..192-column tiles, an
# odd count of 64-wide K blocks, and K below one block
SHAPES = [
    (1, 1, 8),
    (3, 5, 16),
    (8, 384, 256),
    (128, 256, 64),
    (130, 300, 72),
    (257, 513, 200),
    (129, 257, 1032),
    (200, 1000, 520),
    (17, 260, 4096),
    (384, 768, 24),
    (1000, 771, 1024),
    (640, 1152, 192),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tiles_and_ragged_tails(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M * 1_000_003 + N * 101 + K + 7, scale=3.0)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    check_comp(y, x, W, orc)


def test_f16x2_from_split_planes_equals_ws(pkg, orc):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(300, 520, 264, seed=19)
    x, W = x.cuda(), W.cuda()
    hi, lo = pkg.comp_split_f32(x)
    y1 = pkg.comp_gemm_f16x2(hi, lo, W)
    y2 = pkg.comp_gemm_f32x16_ws(x, W)
    assert torch.equal(bits(y1), bits(y2))
    check_comp(y1, x.cpu(), W.cpu(), orc)


def test_hi_only_is_a_plain_fp16_product(pkg, orc):
    # x exact in FP16: lo = 0 and y is the FP16 product with FP32 accumulation
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(256, 512, 512, seed=3)
    x = x.half().float()
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda())
    check_comp(y, x, W, orc)
    hi, lo = pkg.comp_split_f32(x.cuda())
    assert not lo.view(torch.int16).any()


def test_lo_plane_carries_the_residual(pkg, orc):
    # hi = 0, lo = arbitrary FP16: y = 2^-10 * (lo W^T), accumulated in FP32
    g = torch.Generator().manual_seed(23)
    M, N, K = 200, 320, 384
    lo = (torch.randn((M, K), generator=g)).half()
    W = (torch.randn((N, K), generator=g) * 0.05).half()
    hi = torch.zeros_like(lo)
    y = pkg.comp_gemm_f16x2(hi.cuda(), lo.cuda(), W.cuda()).cpu().double()
    exact = (lo.double() @ W.double().t()) * 2.0**-10
    den = (lo.double().abs() @ W.double().abs().t()) * 2.0**-10
    assert torch.all((y - exact).abs() <= 4e-6 * den + 1e-30)


def test_one_hot_and_identity(pkg):
    K, N = 192, 320
    W = (torch.randn(N, K) * 0.02).half()
    x = torch.eye(K, dtype=torch.float32)
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda()).cpu()
    assert torch.equal(y, W.float().t())
    x = torch.randn(200, 256) * 50
    y = pkg.comp_gemm_f32x16_ws(x.cuda(), torch.eye(256, dtype=torch.float16).cuda()).cpu().double()
    assert torch.all((y - x.double()).abs() <= 2.0**-22 * x.double().abs() + 2.0**-35)


def test_small_workspace_falls_back_bitwise(pkg):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 130, 300, 72
    x, W = workloads.random_case(M, N, K, seed=31)
    x, W = x.cuda(), W.cuda()
    need = pkg.comp_gemm_workspace_bytes(M, K)
    assert need == 4 * M * K
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    y_small = pkg.comp_gemm_f32x16_ws(x, W, workspace=ws)
    y_fused = pkg.comp_gemm_f32x16(x, W)
    assert torch.equal(bits(y_small), bits(y_fused))


def test_deterministic_and_workspace_reuse(pkg):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("encoder")
    x, W = x.cuda(), W.cuda()
    ws = torch.full((pkg.comp_gemm_workspace_bytes(*x.shape),), 0xFF, dtype=torch.uint8, device="cuda")
    y1 = pkg.comp_gemm_f32x16_ws(x, W, workspace=ws)
    y2 = pkg.comp_gemm_f32x16_ws(x, W, workspace=ws)
    assert torch.equal(bits(y1), bits(y2))


def test_output_guard_bands(pkg, orc):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 130, 300, 72
    x, W = workloads.random_case(M, N, K, seed=77)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    wsbuf = torch.full((4 * M * K + 2 * pad,), 0xAB, dtype=torch.uint8, device="cuda")
    ws = wsbuf[pad:pad + 4 * M * K]
    pkg.comp_gemm_f32x16_ws(x.cuda(), W.cuda(), y, workspace=ws)
    check_comp(y, x, W, orc)
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()
    assert (wsbuf[:pad] == 0xAB).all() and (wsbuf[pad + 4 * M * K:] == 0xAB).all()


def test_invalid_arguments(pkg):
    from compensated_fp32_projection_gb300 import CompError

    M, N, K = 64, 64, 64
    x = torch.randn(M, K, device="cuda")
    W = torch.randn(N, K, device="cuda").half()
    # workspace overlapping x
    with pytest.raises(CompError):
        pkg.comp_gemm_f32x16_ws(x, W, workspace=x.view(torch.uint8))
    # misaligned planes for the direct call
    planes = torch.zeros(2 * M * K + 8, dtype=torch.float16, device="cuda")
    hi = planes[1:1 + M * K].view(M, K)
    lo = planes[1 + M * K:1 + 2 * M * K].view(M, K)
    with pytest.raises(CompError):
        pkg.comp_gemm_f16x2(hi, lo, W)
    # K not a multiple of 8 for the direct call
    h7 = torch.zeros(M, 7, dtype=torch.float16, device="cuda")
    with pytest.raises(CompError):
        pkg.comp_gemm_f16x2(h7, h7.clone(), torch.zeros(N, 7, dtype=torch.float16, device="cuda"))


def test_k_zero_and_empty(pkg):
    x = torch.empty(4, 0, device="cuda")
    W = torch.empty(6, 0, dtype=torch.float16, device="cuda")
    y = torch.full((4, 6), 7.0, device="cuda")
    pkg.comp_gemm_f32x16_ws(x, W, y)
    assert torch.equal(y.cpu(), torch.zeros(4, 6))
    h = torch.empty(4, 0, dtype=torch.float16, device="cuda")
    y.fill_(7.0)
    pkg.comp_gemm_f16x2(h, h, W, y)
    assert torch.equal(y.cpu(), torch.zeros(4, 6))


def test_device_status_clean(pkg):
    st, where = pkg.device_status()
    assert st == 0 and where == 0


# both product kernels on every tile shape: one CTA per 128-row tile (1) and
# CTA pairs per 256-row tile (2)
# (16, 8000, 1024), (32, 1000, 520): at most 32 rows, K split over clusters of
# 2 CTAs (the second with 9 K blocks, split 4 + 5); (32, 2048, 2048) and
# (17, 260, 4096): clusters of 4.  128-row tiles with K split over a cluster
# and the tile reduced across it (reduce-scatter): (512, 1024, 1024) and
# (129, 257, 4096), ragged, clusters of 4; (300, 500, 520) and
# (1000, 776, 1032), clusters of 2 (9 and 17 K blocks: uneven ranges).
# (256, 2304, 2112) and (256, 2432, 2112): 36 and 38 tiles of 128 x 128, on
# either side of the clusters of 4 that a 152-SM GB300 holds at once (36):
# clusters of 4 for the first, of 2 for the second.
SPLIT_K = [(16, 8000, 1024), (32, 1000, 520), (32, 2048, 2048), (512, 1024, 1024), (129, 257, 4096),
           (300, 500, 520), (1000, 776, 1032), (256, 2304, 2112), (256, 2432, 2112)]


@pytest.mark.parametrize("shape", SHAPES + SPLIT_K + [(2048, 2048, 256), (2000, 2001, 136), (300, 4096, 64)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", [1, 2, 3])
def test_product_kernels(pkg, orc, shape, variant):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    if variant == 3 and M > 32:
        pytest.skip("operands are swapped only for at most 32 rows")
    x, W = workloads.random_case(M, N, K, seed=M * 7 + N * 3 + K, scale=2.0)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), variant)
    check_comp(y, x, W, orc)


def test_product_kernels_agree(pkg, orc):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(1024, 1536, 512, seed=5)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y1 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 1)
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 2)
    e1, _ = check_comp(y1, x, W, orc)
    e2, _ = check_comp(y2, x, W, orc)
    den = (x.double().abs() @ W.double().abs().t()).cuda()
    assert torch.all((y1.double() - y2.double()).abs() <= 2 * 4e-6 * den + 1e-30)


def test_product_variant_out_of_range(pkg):
    from compensated_fp32_projection_gb300 import CompError

    h = torch.zeros(8, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(CompError):
        pkg.comp_gemm_f16x2_variant(h, h.clone(), torch.zeros(16, 64, dtype=torch.float16, device="cuda"), 5)
    h40 = torch.zeros(40, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(CompError):  # swapped operands need M <= 32
        pkg.comp_gemm_f16x2_variant(h40, h40.clone(), torch.zeros(16, 64, dtype=torch.float16, device="cuda"), 3)


@pytest.mark.parametrize("shape", [(16, 14336, 4096), (32, 4100, 1032), (1, 4096, 64), (17, 5000, 520)],
                         ids=lambda s: "x".join(map(str, s)))
def test_swapped_operands_full(pkg, orc, shape):
    # at most 32 rows, many column tiles: the automatic choice is the swapped-operand kernel
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M * 5 + K, scale=2.0)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y = pkg.comp_gemm_f16x2(hi, lo, W.cuda())
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.parametrize("shape", SPLIT_K, ids=lambda s: "x".join(map(str, s)))
def test_split_k_deterministic(pkg, shape):
    # the partial sums of the K ranges are added in a fixed order: bit-identical
    # reruns (a reduction in arrival order would differ between runs)
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=11)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y1 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 1)
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 1)
    assert torch.equal(bits(y1), bits(y2))


@pytest.mark.parametrize("variant,M", [(1, 512), (2, 512), (3, 32)], ids=["one-cta", "pairs", "swapped"])
def test_product_bit_exact_through_identity(pkg, orc, variant, M):
    # W = I: each output is hi + 2^-10 lo of one x value, exact in FP32, so
    # split + product must give the oracle's bits on values that stress the
    # split (FP16 ties, FP16-subnormal hi and lo, magnitudes up to 65504)
    from compensated_fp32_projection_gb300 import workloads

    K = 2048
    x = workloads.special_values_f32(M * K, seed=10 + variant).reshape(M, K)
    W = torch.eye(K, dtype=torch.float16)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), variant).cpu().numpy()
    y_or = orc.gemm_comp(x.numpy(), W.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(y.view(np.uint32), y_or.view(np.uint32)), int(np.sum(y.view(np.uint32) != y_or.view(np.uint32)))


# At most 32 rows: comp_gemm_f32x16_ws runs the swapped kernel with the split
# fused, with K split over a cluster of 2 or 4 CTAs when W has few tiles
# (8 x 4096 x 4096: 4; 16 x 8192 x 4096: 2; 5 x 1000 x 2056, ragged N: 4;
# 32 x 4096 x 4096, 32-row operands: 4), or, with 17 to 32 rows and no split,
# the split and the swapped product (24 x 14336 x 1032).  Both forms give the
# bits of the explicit split + product (identical stages and chunks), and the
# oracle's results within the gate.
FEW_ROWS = [(8, 4096, 4096), (16, 8192, 4096), (5, 1000, 2056), (32, 4096, 4096), (24, 14336, 1032),
            (16, 4096, 14336)]


@pytest.mark.parametrize("shape", FEW_ROWS, ids=lambda s: "x".join(map(str, s)))
def test_ws_few_rows_equals_split_and_product(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + N + K, scale=2.0)
    xd, Wd = x.cuda(), W.cuda()
    y = pkg.comp_gemm_f32x16_ws(xd, Wd)
    hi, lo = pkg.comp_split_f32(xd)
    y2 = pkg.comp_gemm_f16x2(hi, lo, Wd)
    assert torch.equal(bits(y), bits(y2))
    r, c = sample_outputs(M, N)
    e_gpu, e_cast = check_comp(y, x, W, orc, r, c)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.parametrize("shape", [(8, 4096, 4096), (16, 8192, 4096), (5, 1000, 2056), (16, 4608, 1024),
                                   (8, 4864, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_swapped_split_k_deterministic(pkg, shape):
    # the swapped kernel with K split over a cluster adds the ranks' partial
    # sums in rank order: bit-identical reruns
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=5)
    hi, lo = pkg.comp_split_f32(x.cuda())
    y1 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 3)
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, W.cuda(), 3)
    assert torch.equal(bits(y1), bits(y2))
