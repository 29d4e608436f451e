"""GPU parity of the fused compensated projection and the true-FP32 SIMT GEMM.

Gate (the method's acceptance for the projection, laya.cpp docs/vulkan.md,
compensated-FP32 paragraph, with the stated tolerance): every element of the
fused kernel's y satisfies |y - y_oracle| <= 4e-6 * sum_k |x_k||w_k| + 1e-30,
where y_oracle is the oracle's FP64 evaluation of the same formula, and the
max-normalised error against the true product is at least 100x smaller than
that of a single FP16 cast of x.

The SIMT GEMM is the true-FP32 reference (paragraph on the true FP32 matrix
kernels): within the recursive-summation bound gamma_K * sum|x||w|,
gamma_K = K u / (1 - K u), u = 2^-24, of the exact product.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gemm_check import check_comp, sample_outputs, w_bits  # noqa: E402


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def gemm(pkg, x, W, variant):
    if variant is None:
        return pkg.comp_gemm_f32x16(x, W)
    return pkg.comp_gemm_f32x16_variant(x, W, variant)


@pytest.mark.parametrize("name", ["tiny", "encoder", "nonaligned"])
def test_projection_shapes_full(pkg, orc, name):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs(name)
    y = pkg.comp_gemm_f32x16(x.cuda(), W.cuda())
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.parametrize("name", ["square", "skinny"])
def test_projection_shapes_sampled(pkg, orc, name):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs(name)
    y = pkg.comp_gemm_f32x16(x.cuda(), W.cuda())
    r, c = sample_outputs(x.shape[0], W.shape[0])
    e_gpu, e_cast = check_comp(y, x, W, orc, r, c)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
    assert torch.isfinite(y).all()


SHAPES = [
    (1, 1, 1),
    (1, 1, 8),
    (3, 5, 7),
    (8, 384, 256),
    (128, 256, 64),
    (130, 300, 72),
    (257, 513, 200),
    (129, 257, 1027),
    (200, 1000, 520),
    (17, 260, 4096),
    (384, 768, 24),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", [None, 1, 2])
def test_tiles_and_ragged_tails(pkg, orc, shape, variant):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    if variant == 1 and K % 8 != 0:
        pytest.skip("TMA path needs K % 8 == 0")
    x, W = workloads.random_case(M, N, K, seed=M * 1_000_003 + N * 101 + K, scale=3.0)
    y = gemm(pkg, x.cuda(), W.cuda(), variant)
    check_comp(y, x, W, orc)


def test_tma_and_plain_paths_agree_bitwise(pkg):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(300, 520, 264, seed=9)
    x, W = x.cuda(), W.cuda()
    y1 = pkg.comp_gemm_f32x16_variant(x, W, 1)
    y2 = pkg.comp_gemm_f32x16_variant(x, W, 2)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_deterministic(pkg):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("encoder")
    x, W = x.cuda(), W.cuda()
    y1 = pkg.comp_gemm_f32x16(x, W)
    y2 = pkg.comp_gemm_f32x16(x, W)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_exact_fp16_inputs_match_fp16_product(pkg, orc):
    # x exact in FP16: lo = 0, so y is a plain FP16 product with FP32 accumulation
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(256, 512, 512, seed=3)
    x = x.half().float()
    y = pkg.comp_gemm_f32x16(x.cuda(), W.cuda())
    check_comp(y, x, W, orc)


def test_one_hot_rows_select_weights(pkg):
    # x = I (K x K): y[i, j] = W[j, i] exactly
    K, N = 192, 320
    W = (torch.randn(N, K) * 0.02).half()
    x = torch.eye(K, dtype=torch.float32)
    y = pkg.comp_gemm_f32x16(x.cuda(), W.cuda()).cpu()
    assert torch.equal(y, W.float().t())


def test_identity_weights_reconstruct_x(pkg):
    K = 256
    x = torch.randn(200, K) * 50
    W = torch.eye(K, dtype=torch.float16)
    y = pkg.comp_gemm_f32x16(x.cuda(), W.cuda()).cpu().double()
    xd = x.double()
    assert torch.all((y - xd).abs() <= 2.0**-22 * xd.abs() + 2.0**-35)


def test_k_zero_writes_zeros_and_empty_is_noop(pkg):
    x = torch.empty(4, 0, device="cuda")
    W = torch.empty(6, 0, dtype=torch.float16, device="cuda")
    y = torch.full((4, 6), 7.0, device="cuda")
    pkg.comp_gemm_f32x16(x, W, y)
    assert torch.equal(y.cpu(), torch.zeros(4, 6))
    x0 = torch.empty(0, 16, device="cuda")
    y0 = pkg.comp_gemm_f32x16(x0, torch.ones(5, 16, dtype=torch.float16, device="cuda"))
    assert y0.shape == (0, 5)


def test_output_guard_bands(pkg, orc):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 130, 300, 72
    x, W = workloads.random_case(M, N, K, seed=77)
    pad = 4096
    buf = torch.full((M * N + 2 * pad,), float("nan"), device="cuda")
    y = buf[pad:pad + M * N].view(M, N)
    pkg.comp_gemm_f32x16(x.cuda(), W.cuda(), y)
    check_comp(y, x, W, orc)
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + M * N:]).all()


def test_large_and_tiny_magnitudes(pkg, orc):
    # the non-aligned shape's mix, at a multi-tile size: |x| up to 6e4 next to 1e-6
    g = torch.Generator().manual_seed(11)
    M, N, K = 300, 520, 1000
    big = torch.rand((M, K), generator=g) * 1.2e5 - 6e4
    small = torch.randn((M, K), generator=g) * 1e-6
    x = torch.where(torch.rand((M, K), generator=g) < 0.5, small, big)
    W = (torch.randn((N, K), generator=g) * 0.02).half()
    for variant in (1, 2):
        y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), variant)
        e_gpu, e_cast = check_comp(y, x, W, orc)
        assert e_cast >= 100 * e_gpu


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (130, 300, 72), (129, 257, 1027), (512, 1024, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_simt_true_fp32(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=K + 5, scale=2.0)
    y = pkg.comp_gemm_f32_simt(x.cuda(), W.cuda()).cpu().numpy().astype(np.float64)
    xn, wn = x.numpy(), w_bits(W)
    # the oracle's exact product, rounded once to binary32 (within 2^-24 |y| of the FP64 sum)
    y_true = orc.gemm_true(xn, wn).astype(np.float64)
    den = orc.gemm_den(xn, wn)
    u = 2.0**-24
    gamma = K * u / (1 - K * u)
    assert np.all(np.abs(y - y_true) <= gamma * den + u * np.abs(y_true) + 2.0**-149)


def test_simt_vector_and_scalar_loads_agree_bitwise(pkg):
    # 16-byte loads (x and W aligned, K % 8 == 0) and bounds-checked scalar
    # loads (x moved off 16-byte alignment) stage the same values, and the
    # multiply-adds run in the same order: identical bits
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(300, 520, 264, seed=19, scale=2.0)
    xa, Wd = x.cuda(), W.cuda()
    buf = torch.empty(x.numel() + 1, device="cuda")
    xm = buf[1:].view(x.shape)
    xm.copy_(xa)
    y1 = pkg.comp_gemm_f32_simt(xa, Wd)
    y2 = pkg.comp_gemm_f32_simt(xm, Wd)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_device_status_clean_after_gemms(pkg):
    st, where = pkg.device_status()
    assert st == 0 and where == 0


# At most 32 rows: the split fused into the swapped-operand kernel (the
# automatic choice for at most 32 rows; variant 3 forces it), with K split over
# a cluster when W has few tiles.  Ragged N tails, K below one 64-wide block,
# K not a multiple of 64, one and 32 rows.  36 and 38 tiles of W sit on either
# side of the clusters of 4 that a 152-SM GB300 holds at once (36): clusters of
# 4 for the first, pairs for the second.
SWAPPED = [(16, 14336, 4096), (1, 4096, 64), (17, 5000, 520), (32, 4100, 1032), (5, 4096, 8), (32, 8192, 200),
           (8, 384, 256), (3, 130, 72), (16, 4608, 1024), (8, 4864, 1024)]


@pytest.mark.parametrize("shape", SWAPPED, ids=lambda s: "x".join(map(str, s)))
def test_fused_swapped(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M * 13 + N + K, scale=2.0)
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), 3)
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
    y0 = pkg.comp_gemm_f32x16(x.cuda(), W.cuda())  # the automatic choice is the same kernel
    assert torch.equal(y0.view(torch.int32), y.view(torch.int32))


@pytest.mark.parametrize("shape", [(16, 14336, 4096), (32, 4100, 1032), (7, 2048, 136)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_split_equals_standalone_split(pkg, shape):
    # the in-kernel split is the arithmetic of comp_split_f32 and the stages
    # and chunks are those of the two-pass swapped kernel: bit-identical y
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=N + K, scale=3.0)
    x, W = x.cuda(), W.cuda()
    hi, lo = pkg.comp_split_f32(x)
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, W, 3)
    y1 = pkg.comp_gemm_f32x16_variant(x, W, 3)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_fused_swapped_special_values(pkg, orc):
    # the tiny workload's hand-set x values (exact FP16 values, halfway ties,
    # subnormals, +-60000) through the in-kernel split
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("tiny")
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), 3)
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


def test_fused_swapped_rejects(pkg):
    from compensated_fp32_projection_gb300 import CompError

    W = torch.zeros(4096, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(CompError):
        pkg.comp_gemm_f32x16_variant(torch.zeros(33, 64, device="cuda"), W, 3)
    with pytest.raises(CompError):  # K % 8 != 0
        pkg.comp_gemm_f32x16_variant(torch.zeros(4, 60, device="cuda"), torch.zeros(4096, 60, dtype=torch.float16,
                                                                                   device="cuda"), 3)



# More than 128 rows: the split fused into the CTA-pair kernel (variant 4;
# automatic once the output fills about a wave of 128 x 192 tiles).  One pair
# tile, ragged M, N and K tails, K below one 64-wide block, one row, rows
# that fill only the leader CTA of a pair, and a long K (128 chunks of
# promotion) that still has to beat the FP16 cast by 100x.
PAIRED = [(256, 448, 64), (300, 500, 200), (1, 256, 8), (130, 224, 72), (513, 1000, 1032), (1024, 2048, 520),
          (8, 384, 256), (777, 4100, 136), (256, 448, 16384)]


@pytest.mark.parametrize("shape", PAIRED, ids=lambda s: "x".join(map(str, s)))
def test_fused_pair(pkg, orc, shape):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M * 7 + N * 3 + K, scale=2.0)
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), 4)
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


@pytest.mark.parametrize("shape", [(512, 1024, 1024), (300, 500, 200), (1024, 2048, 520), (2048, 4096, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_pair_equals_split_then_pair_product(pkg, shape):
    # the in-place split is the arithmetic of comp_split_f32, and the tiles,
    # stages, chunks and promotion are those of the two-pass pair product:
    # bit-identical y
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + N + K, scale=3.0)
    x, W = x.cuda(), W.cuda()
    hi, lo = pkg.comp_split_f32(x)
    y2 = pkg.comp_gemm_f16x2_variant(hi, lo, W, 2)
    y1 = pkg.comp_gemm_f32x16_variant(x, W, 4)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_fused_pair_encoder_outliers(pkg, orc):
    # the encoder workload (1 % of x scaled by 100) through the in-place split
    # on CTA pairs, every output against the oracle
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("encoder")
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), 4)
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


def test_fused_pair_repeatable(pkg):
    # several calls, each reusing every stage many times: identical bits
    # (a stage read before its split finished would show up as a difference)
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.random_case(2048, 2048, 2048, seed=21, scale=3.0)
    x, W = x.cuda(), W.cuda()
    y0 = pkg.comp_gemm_f32x16_variant(x, W, 4)
    for _ in range(4):
        y = pkg.comp_gemm_f32x16_variant(x, W, 4)
        assert torch.equal(y.view(torch.int32), y0.view(torch.int32))


def test_fused_pair_special_values(pkg, orc):
    # the tiny workload's hand-set x values through the in-place split
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("tiny")
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), 4)
    e_gpu, e_cast = check_comp(y, x, W, orc)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)


def test_fused_pair_is_the_automatic_choice_for_the_square_shape(pkg):
    from compensated_fp32_projection_gb300 import workloads

    x, W = workloads.make_inputs("square")
    x, W = x.cuda(), W.cuda()
    y0 = pkg.comp_gemm_f32x16(x, W)
    y4 = pkg.comp_gemm_f32x16_variant(x, W, 4)
    assert torch.equal(y0.view(torch.int32), y4.view(torch.int32))


def test_fused_pair_rejects(pkg):
    from compensated_fp32_projection_gb300 import CompError

    with pytest.raises(CompError):  # K % 8 != 0
        pkg.comp_gemm_f32x16_variant(torch.zeros(256, 60, device="cuda"),
                                     torch.zeros(256, 60, dtype=torch.float16, device="cuda"), 4)
    with pytest.raises(CompError):  # x not 16-byte aligned
        xb = torch.zeros(256 * 64 + 1, device="cuda")
        pkg.comp_gemm_f32x16_variant(xb[1:].view(256, 64), torch.zeros(256, 64, dtype=torch.float16, device="cuda"), 4)
    with pytest.raises(CompError):
        pkg.comp_gemm_f32x16_variant(torch.zeros(256, 64, device="cuda"),
                                     torch.zeros(256, 64, dtype=torch.float16, device="cuda"), 5)


@pytest.mark.parametrize("variant,M", [(1, 512), (2, 512), (3, 32), (4, 512)], ids=["tma", "plain", "swapped", "pairs"])
def test_fused_split_bit_exact_through_identity(pkg, orc, variant, M):
    # With W = I each output is hi + 2^-10 lo of one x value, a sum that is
    # exact in FP32 (about 22 significant bits), so every fused kernel's
    # in-kernel split must give the oracle's bits for each of M*K values that
    # stress it: FP16 ties and their neighbours, FP16-subnormal hi and lo,
    # magnitudes up to 65504
    from compensated_fp32_projection_gb300 import workloads

    K = 2048
    x = workloads.special_values_f32(M * K, seed=variant).reshape(M, K)
    W = torch.eye(K, dtype=torch.float16)
    y = pkg.comp_gemm_f32x16_variant(x.cuda(), W.cuda(), variant).cpu().numpy()
    y_or = orc.gemm_comp(x.numpy(), W.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(y.view(np.uint32), y_or.view(np.uint32)), int(np.sum(y.view(np.uint32) != y_or.view(np.uint32)))


def test_projection_beyond_2_31_activation_elements(pkg, orc):
    # M*K > 2^31 (64-bit offsets in every path): the fused CTA-pair kernel (the
    # automatic choice) and the two-pass form with a workspace, ~3,000 sampled
    # outputs (first and last rows included) against the oracle
    M, N, K = 524289, 264, 4096
    g = torch.Generator(device="cuda").manual_seed(9)
    x = torch.randn(M, K, device="cuda", generator=g)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.02).half()
    r, c = sample_outputs(M, N)
    rows = np.unique(r)
    x_rows = x[torch.from_numpy(rows).cuda()].cpu()  # only the sampled rows go to the oracle
    r_local = np.searchsorted(rows, r)
    for y in (pkg.comp_gemm_f32x16(x, W), pkg.comp_gemm_f32x16_ws(x, W)):
        ys = y[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu()
        yfull = torch.zeros(rows.size, N)
        yfull[torch.from_numpy(r_local), torch.from_numpy(c)] = ys
        e_gpu, e_cast = check_comp(yfull, x_rows, W.cpu(), orc, r_local, c)
        assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
        del y
    del x
    torch.cuda.empty_cache()


def test_projection_beyond_2_31_weight_elements(pkg, orc):
    # N*K > 2^31 with 16 rows: the swapped-operand kernel with the split fused
    # (the automatic choice), ~3,000 sampled outputs (last columns included)
    # against the oracle
    M, N, K = 16, 524289, 4096
    g = torch.Generator(device="cuda").manual_seed(10)
    x = torch.randn(M, K, device="cuda", generator=g)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.02).half()
    y = pkg.comp_gemm_f32x16(x, W)
    r, c = sample_outputs(M, N)
    cols = np.unique(c)
    W_cols = W[torch.from_numpy(cols).cuda()].cpu()  # only the sampled rows of W go to the oracle
    c_local = np.searchsorted(cols, c)
    ys = y[torch.from_numpy(r).cuda(), torch.from_numpy(c).cuda()].cpu()
    ysub = torch.zeros(M, cols.size)
    ysub[torch.from_numpy(r), torch.from_numpy(c_local)] = ys
    e_gpu, e_cast = check_comp(ysub, x.cpu(), W_cols, orc, r, c_local)
    assert e_cast >= 100 * e_gpu, (e_cast, e_gpu)
    del W, y
    torch.cuda.empty_cache()
