"""GPU parity of the GEGLU step (laya.cpp docs/vulkan.md, feed-forward
paragraph: gate activation and multiplication fused into one dispatch):
out = gelu(gate) * (y + bias) applied by every product kernel to the merged
projection, and by the streaming comp_geglu_f32 dispatch, against the
oracle's epilogue of the oracle's projection.

Tolerance per element: the projection's gate, 4e-6 * sum|x||w|, scaled by
|gelu(g)|, plus the FP32 epilogue's own rounding, 2^-20 * (16 + g^2) relative
to |gelu(g)| * (|y| + |b|): a few binary32 operations and CUDA's erfcf (4 ulp),
and the argument sensitivity of erfc in the negative tail (its relative
condition number grows like g^2).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from gemm_check import w_bits  # noqa: E402


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as p

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return p


def operands(M, N, with_bias, with_gate, seed):
    g = torch.Generator().manual_seed(seed)
    b = (torch.randn(N, generator=g) * 0.5) if with_bias else None
    gate = (torch.randn(M, N, generator=g) * 2.0) if with_gate else None
    return b, gate


def check_epilogue(out, x, W, b, gate, orc):
    xn, wn = x.numpy(), w_bits(W)
    y_or = orc.gemm_comp(xn, wn)
    den = orc.gemm_den(xn, wn)
    bn = None if b is None else b.numpy()
    gn = None if gate is None else gate.numpy()
    out_or = orc.epilogue(y_or, bn, gn).astype(np.float64)
    if gn is None:
        gel = np.ones_like(y_or, dtype=np.float64)
        g2 = np.zeros_like(gel)
    else:
        gel = np.abs(orc.epilogue(np.ones_like(y_or), None, gn).astype(np.float64))  # |gelu(g)|
        g2 = gn.astype(np.float64) ** 2
    babs = 0.0 if bn is None else np.abs(bn.astype(np.float64))[None, :]
    tol = gel * (4e-6 * den + 1e-30) + 2.0**-20 * (16.0 + g2) * gel * (np.abs(y_or.astype(np.float64)) + babs) + 1e-30
    err = np.abs(out.cpu().numpy().astype(np.float64) - out_or)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, f"{bad.shape[0]} elements over tolerance, first {bad[:3].tolist()}"


MODES = [(True, False), (False, True), (True, True)]
MODE_IDS = ["bias", "gate", "bias+gate"]


@pytest.mark.parametrize("mode", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("shape,variant", [((130, 300, 72), 1), ((257, 513, 200), 1), ((17, 260, 4096), 1),
                                           ((512, 1024, 256), 2), ((300, 520, 264), 2), ((16, 4096, 256), 3),
                                           ((5, 700, 136), 3)],
                         ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else f"variant{v}")
def test_product_kernels_apply_the_epilogue(pkg, orc, shape, variant, mode):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=M + N + K + variant, scale=2.0)
    b, gate = operands(M, N, *mode, seed=M * N)
    hi, lo = pkg.comp_split_f32(x.cuda())
    out = pkg.comp_gemm_f16x2_epilogue(hi, lo, W.cuda(), None if b is None else b.cuda(),
                                       None if gate is None else gate.cuda(), variant)
    check_epilogue(out, x, W, b, gate, orc)


@pytest.mark.parametrize("shape,ws", [((16, 4096, 512), "auto"), ((512, 8192, 256), "auto"), ((129, 257, 1027), "auto"),
                                      ((300, 520, 264), "none")],
                         ids=["swapped-fused", "pairs-two-pass", "padded-two-pass", "fused-kernel"])
def test_projection_paths_apply_the_epilogue(pkg, orc, shape, ws):
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=K, scale=2.0)
    b, gate = operands(M, N, True, True, seed=N)
    workspace = torch.empty(16, dtype=torch.uint8, device="cuda") if ws == "none" else None
    out = pkg.comp_gemm_f32x16_epilogue(x.cuda(), W.cuda(), b.cuda(), gate.cuda(), workspace=workspace)
    check_epilogue(out, x, W, b, gate, orc)


def test_fused_pair_epilogue_equals_two_pass(pkg, orc):
    # without a workspace a large projection runs the fused CTA-pair kernel
    # (bias in its epilogue, then the GEGLU dispatch); with one, the two-pass
    # form on CTA pairs: same tiles, chunks and epilogue, so identical bits
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 300, 12800, 136
    x, W = workloads.random_case(M, N, K, seed=31, scale=2.0)
    b, gate = operands(M, N, True, True, seed=7)
    x, W, b, gate = x.cuda(), W.cuda(), b.cuda(), gate.cuda()
    none = torch.empty(16, dtype=torch.uint8, device="cuda")
    y_fused = pkg.comp_gemm_f32x16_epilogue(x, W, b, gate, workspace=none)
    y_two = pkg.comp_gemm_f32x16_epilogue(x, W, b, gate)
    assert torch.equal(y_fused.view(torch.int32), y_two.view(torch.int32))
    check_epilogue(y_fused, x.cpu(), W.cpu(), b.cpu(), gate.cpu(), orc)


def test_no_operands_is_the_plain_projection(pkg):
    from compensated_fp32_projection_gb300 import workloads

    for M, N, K in ((300, 520, 264), (16, 4096, 512), (512, 8192, 256)):
        x, W = workloads.random_case(M, N, K, seed=1)
        x, W = x.cuda(), W.cuda()
        y0 = pkg.comp_gemm_f32x16_ws(x, W)
        y1 = pkg.comp_gemm_f32x16_epilogue(x, W)
        assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))


def test_gate_special_values(pkg):
    # gelu(0) = 0, gelu(g) = g for large g (Phi = 1 in binary32), gelu(-large) = -0
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = 256, 512, 128
    x, W = workloads.random_case(M, N, K, seed=2)
    x, W = x.cuda(), W.cuda()
    y = pkg.comp_gemm_f32x16_ws(x, W)
    for value, expect in ((0.0, lambda y: torch.zeros_like(y)), (30.0, lambda y: y * 30.0)):
        gate = torch.full((M, N), value, device="cuda")
        out = pkg.comp_gemm_f32x16_epilogue(x, W, None, gate)
        assert torch.equal(out, expect(y))
    out = pkg.comp_gemm_f32x16_epilogue(x, W, None, torch.full((M, N), -60.0, device="cuda"))
    assert torch.all(out == 0.0)


def test_epilogue_rejects_overlap_and_bad_shapes(pkg):
    from compensated_fp32_projection_gb300 import CompError

    x = torch.zeros(8, 64, device="cuda")
    W = torch.zeros(16, 64, dtype=torch.float16, device="cuda")
    y = torch.empty(8, 16, device="cuda")
    with pytest.raises(CompError):  # gate is y itself
        pkg.comp_gemm_f32x16_epilogue(x, W, None, y, y=y)
    with pytest.raises(ValueError):
        pkg.comp_gemm_f32x16_epilogue(x, W, torch.zeros(15, device="cuda"))


def _geglu_check(out, gate, up, orc):
    g, u = gate.cpu().numpy(), up.cpu().numpy()
    ref = orc.epilogue(u.reshape(1, -1), None, g.reshape(1, -1)).reshape(-1).astype(np.float64)
    gel = np.abs(orc.epilogue(np.ones((1, g.size), np.float32), None, g.reshape(1, -1)).reshape(-1).astype(np.float64))
    tol = 2.0**-20 * (16.0 + g.astype(np.float64) ** 2) * gel * np.abs(u.astype(np.float64)) + 1e-37
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= tol), f"max err/tol {float(np.max(err / tol))}"


@pytest.mark.parametrize("n", [1, 7, 4096, 1_000_003])
def test_geglu_dispatch(pkg, orc, n):
    # the feed-forward paragraph's single GEGLU dispatch: out = gelu(gate) * up
    g = torch.Generator().manual_seed(n)
    gate = torch.randn(n, generator=g) * 2.5
    up = torch.randn(n, generator=g) * 3.0
    out = pkg.comp_geglu_f32(gate.cuda(), up.cuda())
    _geglu_check(out, gate, up, orc)


def test_geglu_in_place_and_misaligned(pkg, orc):
    g = torch.Generator().manual_seed(4)
    gate = torch.randn(10_001, generator=g) * 2.0
    up = torch.randn(10_001, generator=g)
    ref = pkg.comp_geglu_f32(gate.cuda(), up.cuda())
    u2 = up.cuda()
    pkg.comp_geglu_f32(gate.cuda(), u2, out=u2)  # out is up
    g2 = gate.cuda()
    pkg.comp_geglu_f32(g2, up.cuda(), out=g2)  # out is gate
    assert torch.equal(u2.view(torch.int32), ref.view(torch.int32))
    assert torch.equal(g2.view(torch.int32), ref.view(torch.int32))
    # views starting one element in: 4-byte aligned only, the scalar kernel
    gb, ub = gate.cuda(), up.cuda()
    out = pkg.comp_geglu_f32(gb[1:], ub[1:])
    assert torch.equal(out.view(torch.int32), ref[1:].view(torch.int32))
    _geglu_check(ref, gate, up, orc)


@pytest.mark.parametrize("shape", [(512, 8192, 256), (16, 4096, 512), (300, 520, 264)],
                         ids=lambda s: "x".join(map(str, s)))
def test_streaming_gate_equals_gate_in_the_product(pkg, shape):
    # comp_gemm_f32x16_epilogue applies the gate with the GEGLU dispatch after
    # the product; comp_gemm_f16x2_epilogue inside it: the same operations in
    # the same order, so the same bits
    from compensated_fp32_projection_gb300 import workloads

    M, N, K = shape
    x, W = workloads.random_case(M, N, K, seed=3)
    b, gate = operands(M, N, True, True, seed=9)
    x, W, b, gate = x.cuda(), W.cuda(), b.cuda(), gate.cuda()
    y1 = pkg.comp_gemm_f32x16_epilogue(x, W, b, gate)
    hi, lo = pkg.comp_split_f32(x)
    y2 = pkg.comp_gemm_f16x2_epilogue(hi, lo, W, b, gate)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
