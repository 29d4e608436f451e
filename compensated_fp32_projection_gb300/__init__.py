"""Compensated-FP32 projection for GB300 (sm_103a).

The method (laya.cpp, docs/vulkan.md, compensated-FP32 paragraph): each FP32
input x is split into hi = fp16_rne(x) and lo = fp16_rne((x - hi) * 1024), both
are multiplied by the exact FP16 weights with FP32 accumulators, and the results
are merged in FP32 as y = acc_hi + acc_lo * 2^-10.

The torch-facing calls below carry the C ABI's names and only marshal
arguments (device pointers, sizes, the current CUDA stream) into
``libcompfp32.so``; every step runs in its CUDA kernels.  Outputs that are not
given are allocated with ``torch.empty`` on the input's device.
"""
from __future__ import annotations

from . import _native
from ._native import CompError, device_status, status_string

__all__ = [
    "CompError",
    "comp_split_f32",
    "comp_merge_f32",
    "comp_gemm_f32x16",
    "comp_gemm_f32x16_variant",
    "comp_gemm_f32_simt",
    "comp_gemm_f16x2",
    "comp_gemm_f16x2_variant",
    "comp_gemm_f32x16_ws",
    "comp_geglu_f32",
    "comp_gemm_f32x16_epilogue",
    "comp_gemm_f16x2_epilogue",
    "comp_gemm_workspace_bytes",
    "comp_gemm_workspace_bytes_mnk",
    "comp_gemm_f32x16_noalloc",
    "device_status",
    "status_string",
]


def _torch():
    import torch

    return torch


def _stream(t, stream):
    if stream is not None:
        return int(stream) if isinstance(stream, int) else stream.cuda_stream
    return _torch().cuda.current_stream(t.device).cuda_stream


def _check(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def comp_split_f32(x, hi=None, lo=None, stream=None):
    """(hi, lo) float16 tensors shaped like x: hi = fp16_rne(x), lo = fp16_rne((x-hi)*1024)."""
    torch = _torch()
    _check(x, torch.float32, "x")
    hi = torch.empty(x.shape, dtype=torch.float16, device=x.device) if hi is None else hi
    lo = torch.empty(x.shape, dtype=torch.float16, device=x.device) if lo is None else lo
    _check(hi, torch.float16, "hi")
    _check(lo, torch.float16, "lo")
    if hi.numel() != x.numel() or lo.numel() != x.numel():
        raise ValueError("hi and lo must have as many elements as x")
    _native.call("comp_split_f32", x.data_ptr(), hi.data_ptr(), lo.data_ptr(), x.numel(), _stream(x, stream))
    return hi, lo


def comp_merge_f32(acc_hi, acc_lo, y=None, stream=None):
    """y = acc_hi + acc_lo * 2^-10 (float32, two rounded operations)."""
    torch = _torch()
    _check(acc_hi, torch.float32, "acc_hi")
    _check(acc_lo, torch.float32, "acc_lo")
    if acc_hi.numel() != acc_lo.numel():
        raise ValueError("acc_hi and acc_lo differ in size")
    y = torch.empty(acc_hi.shape, dtype=torch.float32, device=acc_hi.device) if y is None else y
    _check(y, torch.float32, "y")
    if y.numel() != acc_hi.numel():
        raise ValueError("y must have as many elements as acc_hi")
    _native.call("comp_merge_f32", acc_hi.data_ptr(), acc_lo.data_ptr(), y.data_ptr(), acc_hi.numel(),
                 _stream(acc_hi, stream))
    return y


def _gemm_args(x, W, y):
    torch = _torch()
    _check(x, torch.float32, "x")
    _check(W, torch.float16, "W")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError("x must be [M, K] and W [N, K]")
    M, K = x.shape
    N = W.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    _check(y, torch.float32, "y")
    if tuple(y.shape) != (M, N):
        raise ValueError("y must be [M, N]")
    return M, N, K, y


def comp_gemm_f32x16(x, W, y=None, stream=None):
    """The fused compensated projection y = x W^T (FP32 in, FP16 weights, FP32 out)."""
    M, N, K, y = _gemm_args(x, W, y)
    _native.call("comp_gemm_f32x16", x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K, _stream(x, stream))
    return y


def comp_gemm_f32x16_variant(x, W, variant, y=None, stream=None):
    """comp_gemm_f32x16 with a chosen kernel path (0 auto, 1 TMA loads, 2 plain loads,
    3 operands swapped with the split fused, M <= 32, 4 CTA pairs with the split fused)."""
    M, N, K, y = _gemm_args(x, W, y)
    _native.call("comp_gemm_f32x16_variant", x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K, int(variant),
                 _stream(x, stream))
    return y


def comp_gemm_f32_simt(x, W, y=None, stream=None):
    """The true-FP32 reference product on the CUDA cores: y = x float(W)^T."""
    M, N, K, y = _gemm_args(x, W, y)
    _native.call("comp_gemm_f32_simt", x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K, _stream(x, stream))
    return y


def comp_gemm_f16x2(hi, lo, W, y=None, stream=None):
    """y = hi W^T + 2^-10 lo W^T from the split planes of comp_split_f32 (FP32 out)."""
    return comp_gemm_f16x2_variant(hi, lo, W, 0, y, stream)


def comp_gemm_f16x2_variant(hi, lo, W, variant, y=None, stream=None):
    """comp_gemm_f16x2 with a chosen kernel (0 auto, 1 one CTA per 128-row tile, 2 CTA pairs,
    3 operands swapped for M <= 32)."""
    torch = _torch()
    _check(hi, torch.float16, "hi")
    _check(lo, torch.float16, "lo")
    _check(W, torch.float16, "W")
    if hi.shape != lo.shape:
        raise ValueError("hi and lo differ in shape")
    if hi.dim() != 2 or W.dim() != 2 or hi.shape[1] != W.shape[1]:
        raise ValueError("hi and lo must be [M, K] and W [N, K]")
    M, K = hi.shape
    N = W.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=hi.device) if y is None else y
    _check(y, torch.float32, "y")
    if tuple(y.shape) != (M, N):
        raise ValueError("y must be [M, N]")
    _native.call("comp_gemm_f16x2_variant", hi.data_ptr(), lo.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K,
                 int(variant), _stream(hi, stream))
    return y


def comp_gemm_workspace_bytes(M, K):
    """Workspace bytes the two-pass form of comp_gemm_f32x16_ws needs (4*M*K)."""
    return int(_native.load().comp_gemm_workspace_bytes(int(M), int(K)))


def comp_gemm_workspace_bytes_mnk(M, N, K):
    """Workspace bytes of the two-pass form for any K and W alignment (4*M*Kp + 2*N*Kp, Kp = K rounded up to 8)."""
    return int(_native.load().comp_gemm_workspace_bytes_mnk(int(M), int(N), int(K)))


def comp_gemm_f32x16_ws(x, W, y=None, workspace=None, stream=None):
    """comp_gemm_f32x16 with a device workspace (uint8 tensor); with enough room
    it runs the two-pass form: split once, then the two products and the merge.
    Allocated here when not given: comp_gemm_workspace_bytes(M, K) when K is a
    multiple of 8 and W is 16-byte aligned, else comp_gemm_workspace_bytes_mnk."""
    torch = _torch()
    M, N, K, y = _gemm_args(x, W, y)
    if workspace is None:
        aligned = K % 8 == 0 and W.data_ptr() % 16 == 0
        nbytes = comp_gemm_workspace_bytes(M, K) if aligned else comp_gemm_workspace_bytes_mnk(M, N, K)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    _native.call("comp_gemm_f32x16_ws", x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K, workspace.data_ptr(),
                 nbytes, _stream(x, stream))
    return y


def comp_geglu_f32(gate, up, out=None, stream=None):
    """out = gelu(gate) * up elementwise (exact GELU), one dispatch; out may be gate or up."""
    torch = _torch()
    _check(gate, torch.float32, "gate")
    _check(up, torch.float32, "up")
    if gate.shape != up.shape or gate.device != up.device:
        raise ValueError("gate and up must have the same shape and device")
    if out is None:
        out = torch.empty_like(up)
    _check(out, torch.float32, "out")
    if out.shape != up.shape:
        raise ValueError("out must have the shape of up")
    _native.call("comp_geglu_f32", gate.data_ptr(), up.data_ptr(), out.data_ptr(), up.numel(), _stream(up, stream))
    return out


def _epilogue_args(bias, gate, M, N, device):
    torch = _torch()
    if bias is not None:
        _check(bias, torch.float32, "bias")
        if tuple(bias.shape) != (N,) or bias.device != device:
            raise ValueError("bias must be a [N] float32 tensor on the output's device")
    if gate is not None:
        _check(gate, torch.float32, "gate")
        if tuple(gate.shape) != (M, N) or gate.device != device:
            raise ValueError("gate must be a [M, N] float32 tensor on the output's device")
    return (0 if bias is None else bias.data_ptr()), (0 if gate is None else gate.data_ptr())


def comp_gemm_f32x16_epilogue(x, W, bias=None, gate=None, y=None, workspace=None, stream=None):
    """comp_gemm_f32x16_ws followed, in the product kernel's epilogue, by the
    GEGLU step y = gelu(gate) * (y + bias) (bias [N] and gate [M, N] float32,
    each optional; gelu(g) = g * Phi(g))."""
    torch = _torch()
    M, N, K, y = _gemm_args(x, W, y)
    pb, pg = _epilogue_args(bias, gate, M, N, y.device)
    if workspace is None:
        aligned = K % 8 == 0 and W.data_ptr() % 16 == 0
        nbytes = comp_gemm_workspace_bytes(M, K) if aligned else comp_gemm_workspace_bytes_mnk(M, N, K)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=x.device)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    _native.call("comp_gemm_f32x16_epilogue", x.data_ptr(), W.data_ptr(), pb, pg, y.data_ptr(), M, N, K,
                 workspace.data_ptr(), nbytes, _stream(x, stream))
    return y


def comp_gemm_f16x2_epilogue(hi, lo, W, bias=None, gate=None, variant=0, y=None, stream=None):
    """comp_gemm_f16x2_variant with the GEGLU epilogue y = gelu(gate) * (y + bias)."""
    torch = _torch()
    _check(hi, torch.float16, "hi")
    _check(lo, torch.float16, "lo")
    _check(W, torch.float16, "W")
    if hi.shape != lo.shape or hi.dim() != 2 or W.dim() != 2 or hi.shape[1] != W.shape[1]:
        raise ValueError("hi and lo must be [M, K] and W [N, K]")
    M, K = hi.shape
    N = W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=hi.device)
    _check(y, torch.float32, "y")
    pb, pg = _epilogue_args(bias, gate, M, N, y.device)
    _native.call("comp_gemm_f16x2_epilogue", hi.data_ptr(), lo.data_ptr(), W.data_ptr(), pb, pg, y.data_ptr(), M, N,
                 K, int(variant), _stream(hi, stream))
    return y


def comp_gemm_f32x16_noalloc(x, W, y=None, stream=None):
    """comp_gemm_f32x16_ws with the library's static 64 MiB device workspace,
    for callers that cannot allocate device memory per call (4*M*K must fit).
    Calls on unordered streams race on that shared workspace."""
    M, N, K, y = _gemm_args(x, W, y)
    _native.call("comp_gemm_f32x16_noalloc", x.data_ptr(), W.data_ptr(), y.data_ptr(), M, N, K,
                 _stream(x, stream))
    return y
