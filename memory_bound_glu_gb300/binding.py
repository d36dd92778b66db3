"""ctypes binding of libmbglu.so (C ABI in include/mbglu.h).

Argument marshalling only: tensors become device pointers, row strides and
the current CUDA stream; every step of the computation runs in the library's
kernels.  There is no fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmbglu.so")

MODE_FUSED = 0
MODE_HF = 1
_MODES = {"fused": MODE_FUSED, "hf": MODE_HF, MODE_FUSED: MODE_FUSED, MODE_HF: MODE_HF}
MAX_M = 64        # batch rows per call (MBGLU_MAX_M)
BLOCK_M = 16      # batch rows per pass over the weights (MBGLU_BLOCK_M)
WORKSPACE_BYTES = 256

# Every symbol include/mbglu.h declares.
EXPORTS = ("glu_gemv", "add_rmsnorm_glu", "add_rmsnorm_glu_ws", "add_rmsnorm_glu_strided", "add_rmsnorm_glu_noalloc",
           "silu_mul", "gdn_gates", "glu_backward", "glu_backward_workspace_bytes",
           "mbglu_set_launch_policy",
           "mbglu_get_launch_policy",
           "mbglu_status_string", "mbglu_abi_version", "mbglu_last_cuda_error", "mbglu_last_variant",
           "mbglu_last_single_kernel_blocks", "mbglu_noalloc_scratch_read", "mbglu_read_device_error",
           "mbglu_last_backward_path")
POLICY_SERIAL, POLICY_PDL, POLICY_PREFETCH = 0, 1, 2

_lib = None


class MbgluError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().mbglu_status_string(status).decode()
        if status == 7:
            msg += f" (cudaError {lib().mbglu_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


def _bind(l):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    l.glu_gemv.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32, i32, vp]
    l.glu_gemv.restype = i32
    l.add_rmsnorm_glu.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i32, i32, i32, vp]
    l.add_rmsnorm_glu.restype = i32
    l.add_rmsnorm_glu_ws.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i32, i32, i32, vp, ctypes.c_size_t, vp]
    l.add_rmsnorm_glu_ws.restype = i32
    l.add_rmsnorm_glu_noalloc.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i32, i32, i32, vp]
    l.add_rmsnorm_glu_noalloc.restype = i32
    l.add_rmsnorm_glu_strided.argtypes = [vp, vp, vp, ctypes.c_float, vp, i64, vp, i64, vp, i64, i32, i32, i32, i32,
                                          vp, ctypes.c_size_t, vp]
    l.add_rmsnorm_glu_strided.restype = i32
    l.silu_mul.argtypes = [vp, i64, vp, i64, i32, i32, i32, vp]
    l.gdn_gates.argtypes = [vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, i32, i32, vp]
    l.gdn_gates.restype = i32
    l.glu_backward_workspace_bytes.argtypes = [i32, i32, i32]
    l.glu_backward_workspace_bytes.restype = ctypes.c_size_t
    l.glu_backward.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32, i32, i32,
                               vp, ctypes.c_size_t, vp]
    l.glu_backward.restype = i32
    l.silu_mul.restype = i32
    l.mbglu_status_string.argtypes = [i32]
    l.mbglu_status_string.restype = ctypes.c_char_p
    l.mbglu_abi_version.restype = i32
    l.mbglu_last_cuda_error.restype = i32
    l.mbglu_last_variant.restype = i32
    l.mbglu_last_single_kernel_blocks.restype = i32
    l.mbglu_last_backward_path.restype = i32
    l.mbglu_noalloc_scratch_read.argtypes = [ctypes.POINTER(ctypes.c_int), i32]
    l.mbglu_noalloc_scratch_read.restype = i32
    l.mbglu_read_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    l.mbglu_read_device_error.restype = i32
    l.mbglu_set_launch_policy.argtypes = [i32]
    l.mbglu_set_launch_policy.restype = i32
    l.mbglu_get_launch_policy.restype = i32
    return l


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _on(dev):
    """The device context for a call on `dev`: none when it is already the
    current device (the common case; entering torch.cuda.device costs a few
    microseconds per call), else torch.cuda.device(dev)."""
    idx = dev.index
    if idx is None or idx == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


def _stream_handle(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must be {dim}-D, got shape {tuple(t.shape)}")
    if t.numel() and t.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous last dimension")


def glu_gemv(h, gate_w, up_w, out=None, mode="fused", stream=None):
    """out[M,N] = SiLU(h @ gate_w.T) * (h @ up_w.T) in one pass (bf16).

    h is [M,K] (or [K]); gate_w, up_w are [N,K] nn.Linear weights read in
    place; mode "fused" (one rounding) or "hf" (HF bf16 boundaries).  Row
    strides are passed through, so sliced views work without copies.
    """
    squeeze = h.dim() == 1
    h2 = h.unsqueeze(0) if squeeze else h
    _check(h2, "h", 2)
    _check(gate_w, "gate_w", 2)
    _check(up_w, "up_w", 2)
    M, K = h2.shape
    N = gate_w.shape[0]
    if tuple(gate_w.shape) != (N, K) or tuple(up_w.shape) != (N, K):
        raise ValueError(f"weights must be [N,K]=[{N},{K}], got {tuple(gate_w.shape)}, {tuple(up_w.shape)}")
    dev = h2.device
    if gate_w.device != dev or up_w.device != dev:
        raise ValueError("all tensors must be on one device")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    out2 = out.unsqueeze(0) if out.dim() == 1 else out
    _check(out2, "out", 2)
    if tuple(out2.shape) != (M, N) or out2.device != dev:
        raise ValueError(f"out must be [{M},{N}] on {dev}")
    with _on(dev):
        st = lib().glu_gemv(h2.data_ptr(), h2.stride(0), gate_w.data_ptr(), gate_w.stride(0),
                            up_w.data_ptr(), up_w.stride(0), out2.data_ptr(), out2.stride(0),
                            M, N, K, _MODES[mode], _stream_handle(dev, stream))
    if st != 0:
        raise MbgluError(st, "glu_gemv")
    return out2.view(N) if squeeze else out


def column_shard(N: int, world: int, rank: int):
    """Rows [lo, hi) of gate_w and up_w -- and columns of out -- that rank
    `rank` of `world` owns when the GLU GEMV is split column-parallel over N
    (DeepSpeed PR #8602, "Architecture Notes": the gate/up projections are
    column-parallel under AutoTP and the segment needs no communication; the
    all-reduce belongs to the row-parallel down projection after it).  The
    shares are balanced (sizes differ by at most one row), disjoint, in rank
    order, and cover [0, N).  Each rank then calls glu_gemv (or
    add_rmsnorm_glu, whose prologue every rank repeats) on its rows of both
    weights and writes out[:, lo:hi]; no collective is involved."""
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError(f"bad split: N={N}, world={world}, rank={rank}")
    return (N * rank) // world, (N * (rank + 1)) // world


def glu_backward(h, gate_w, up_w, dout, grad_h=None, grad_gate=None, grad_up=None, want_h=True, want_w=True,
                 workspace=None, stream=None):
    """Gradients of glu_gemv's SiLU(h @ gate_w.T) * (h @ up_w.T) for an
    upstream dout [M,N] (bf16): returns (grad_h [M,K], grad_gate [N,K],
    grad_up [N,K]), bf16, each None where not wanted.  Output tensors may be
    passed in (any row stride, contiguous last dimension); the workspace is a
    byte tensor of glu_backward_workspace_bytes(M, N, K), allocated here by
    torch's allocator when not given."""
    _check(h, "h", 2)
    _check(gate_w, "gate_w", 2)
    _check(up_w, "up_w", 2)
    _check(dout, "dout", 2)
    M, K = h.shape
    N = gate_w.shape[0]
    if tuple(gate_w.shape) != (N, K) or tuple(up_w.shape) != (N, K) or tuple(dout.shape) != (M, N):
        raise ValueError(f"expected gate_w, up_w [{N},{K}] and dout [{M},{N}]")
    dev = h.device
    if want_h and grad_h is None:
        grad_h = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    if want_w and grad_gate is None:
        grad_gate = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    if want_w and grad_up is None:
        grad_up = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    if not want_h:
        grad_h = None
    if not want_w:
        grad_gate = grad_up = None
    for t, name, shape in ((grad_h, "grad_h", (M, K)), (grad_gate, "grad_gate", (N, K)), (grad_up, "grad_up", (N, K))):
        if t is not None:
            _check(t, name, 2)
            if tuple(t.shape) != shape or t.device != dev:
                raise ValueError(f"{name} must be {list(shape)} on {dev}")
    need = lib().glu_backward_workspace_bytes(M, N, K)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wsp = workspace.data_ptr() if workspace is not None else None
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0

    def ptr(t):
        return (t.data_ptr(), t.stride(0)) if t is not None else (None, 0)

    with _on(dev):
        st = lib().glu_backward(h.data_ptr(), h.stride(0), gate_w.data_ptr(), gate_w.stride(0), up_w.data_ptr(),
                                up_w.stride(0), dout.data_ptr(), dout.stride(0), *ptr(grad_h), *ptr(grad_gate),
                                *ptr(grad_up), M, N, K, wsp, wsb, _stream_handle(dev, stream))
    if st != 0:
        raise MbgluError(st, "glu_backward")
    return grad_h, grad_gate, grad_up


class DualWeightGlu(torch.autograd.Function):
    """out = SiLU(h @ gate_w.T) * (h @ up_w.T) with the weights read in place
    and gradients for h, gate_w and up_w ([8602/PlanB] "Plan B Design": the
    Function works on the model's own weight tensors, not on a copy, so their
    gradients land on those tensors)."""

    @staticmethod
    def forward(ctx, h, gate_w, up_w, mode="fused"):
        ctx.save_for_backward(h, gate_w, up_w)
        return glu_gemv(h, gate_w, up_w, mode=mode)

    @staticmethod
    def backward(ctx, dout):
        h, gate_w, up_w = ctx.saved_tensors
        squeeze = h.dim() == 1
        h2 = h.unsqueeze(0) if squeeze else h
        d2 = dout.reshape(h2.shape[0], -1).to(torch.bfloat16)
        if d2.stride(-1) != 1:
            d2 = d2.contiguous()
        gh, gg, gu = glu_backward(h2, gate_w, up_w, d2, want_h=ctx.needs_input_grad[0],
                                  want_w=ctx.needs_input_grad[1] or ctx.needs_input_grad[2])
        if gh is not None and squeeze:
            gh = gh.view(-1)
        return gh, gg if ctx.needs_input_grad[1] else None, gu if ctx.needs_input_grad[2] else None, None


def new_workspace(device=None):
    """A zeroed workspace for add_rmsnorm_glu (one per concurrently running stream)."""
    return torch.zeros(WORKSPACE_BYTES, dtype=torch.uint8, device=device or "cuda")


def add_rmsnorm_glu(x, residual, norm_w, eps, gate_w, up_w, out=None, mode="hf", stream=None, workspace=None):
    """residual <- bf16(x + residual); h = zero-centred RMSNorm(residual);
    out = GLU(h).  Returns out; residual is updated in place.  With a
    workspace (new_workspace()) the whole segment runs as one kernel.  x,
    residual and norm_w are contiguous; the weights and out may be row-strided
    views (contiguous last dimension)."""
    _check(x, "x", 2)
    _check(residual, "residual", 2)
    _check(norm_w, "norm_w", 1)
    _check(gate_w, "gate_w", 2)
    _check(up_w, "up_w", 2)
    M, K = x.shape
    N = gate_w.shape[0]
    for t, name in ((x, "x"), (residual, "residual"), (norm_w, "norm_w")):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if tuple(residual.shape) != (M, K) or tuple(norm_w.shape) != (K,):
        raise ValueError("residual must be [M,K] and norm_w [K]")
    if tuple(gate_w.shape) != (N, K) or tuple(up_w.shape) != (N, K):
        raise ValueError("weights must be [N,K]")
    dev = x.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    _check(out, "out", 2)
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out must be a [{M},{N}] tensor")
    if workspace is not None and not (workspace.is_cuda and workspace.device == dev and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on the operands' device")
    with _on(dev):
        if not (gate_w.is_contiguous() and up_w.is_contiguous() and out.is_contiguous()):
            wsp = workspace.data_ptr() if workspace is not None else None
            wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
            st = lib().add_rmsnorm_glu_strided(x.data_ptr(), residual.data_ptr(), norm_w.data_ptr(), float(eps),
                                               gate_w.data_ptr(), gate_w.stride(0), up_w.data_ptr(), up_w.stride(0),
                                               out.data_ptr(), out.stride(0), M, N, K, _MODES[mode], wsp, wsb,
                                               _stream_handle(dev, stream))
        elif workspace is None:
            st = lib().add_rmsnorm_glu(x.data_ptr(), residual.data_ptr(), norm_w.data_ptr(), float(eps),
                                       gate_w.data_ptr(), up_w.data_ptr(), out.data_ptr(), M, N, K, _MODES[mode],
                                       _stream_handle(dev, stream))
        else:
            st = lib().add_rmsnorm_glu_ws(x.data_ptr(), residual.data_ptr(), norm_w.data_ptr(), float(eps),
                                          gate_w.data_ptr(), up_w.data_ptr(), out.data_ptr(), M, N, K, _MODES[mode],
                                          workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                          _stream_handle(dev, stream))
    if st != 0:
        raise MbgluError(st, "add_rmsnorm_glu")
    return out


def silu_mul(x, out=None, mode="fused", stream=None):
    """out[M,N] = SiLU(x[:, :N]) * x[:, N:2N] on the halves layout (the gate
    projection in the first half of each row, the up projection in the second,
    as a GEMM on the concatenated [gate; up] weight leaves them); mode "fused"
    (one rounding) or "hf" (SiLU rounded to bf16 first).  x is [M, 2N] (or
    [2N]) bf16 with a contiguous last dimension; any row stride."""
    squeeze = x.dim() == 1
    x2 = x.unsqueeze(0) if squeeze else x
    _check(x2, "x", 2)
    M, W = x2.shape
    if W % 2:
        raise ValueError(f"x must have an even number of columns (gate half, up half), got {W}")
    N = W // 2
    dev = x2.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    out2 = out.unsqueeze(0) if out.dim() == 1 else out
    _check(out2, "out", 2)
    if tuple(out2.shape) != (M, N) or out2.device != dev:
        raise ValueError(f"out must be [{M},{N}] on {dev}")
    with _on(dev):
        st = lib().silu_mul(x2.data_ptr(), x2.stride(0), out2.data_ptr(), out2.stride(0), M, N, _MODES[mode],
                            _stream_handle(dev, stream))
    if st != 0:
        raise MbgluError(st, "silu_mul")
    return out2.view(N) if squeeze else out


def gdn_gates(a, b, A_log, dt_bias, g=None, beta=None, stream=None):
    """Gated-delta-net gates: g = -exp(A_log) * softplus(a + dt_bias) (fp32)
    and beta = sigmoid(b) (bf16), per token and head.  a, b are [T, H] bf16
    (row-strided views allowed, contiguous last dimension); A_log, dt_bias are
    contiguous [H] float32.  Returns (g, beta)."""
    _check(a, "a", 2)
    _check(b, "b", 2)
    T, H = a.shape
    if tuple(b.shape) != (T, H):
        raise ValueError(f"b must be [{T},{H}]")
    for t, name in ((A_log, "A_log"), (dt_bias, "dt_bias")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or tuple(t.shape) != (H,) \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape [{H}]")
    dev = a.device
    if g is None:
        g = torch.empty((T, H), dtype=torch.float32, device=dev)
    if beta is None:
        beta = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if g.dtype != torch.float32 or tuple(g.shape) != (T, H) or (g.numel() and g.stride(-1) != 1):
        raise ValueError(f"g must be a float32 [{T},{H}] tensor with a contiguous last dimension")
    _check(beta, "beta", 2)
    if tuple(beta.shape) != (T, H):
        raise ValueError(f"beta must be [{T},{H}]")
    with _on(dev):
        st = lib().gdn_gates(a.data_ptr(), a.stride(0), b.data_ptr(), b.stride(0), A_log.data_ptr(),
                             dt_bias.data_ptr(), g.data_ptr(), g.stride(0), beta.data_ptr(), beta.stride(0), T, H,
                             _stream_handle(dev, stream))
    if st != 0:
        raise MbgluError(st, "gdn_gates")
    return g, beta


def last_variant() -> int:
    """Kernel the calling thread's last call launched: 0 none, 1 streaming
    (CUDA-core), 2 generic, 3 zero fill, 4 tensor cores with h in shared
    memory (batch >= 3), 5 silu_mul, 6 gdn_gates, 7 row blocks, 8
    glu_backward, 9 tcgen05, 10 the K-slice tensor-core kernel (batch 1..16)."""
    return lib().mbglu_last_variant()


def last_backward_path() -> int:
    """The second step of the calling thread's last glu_backward: 0 none, 1
    separate kernels, 2 one pass on the CUDA cores, 3 one pass on the tensor
    cores."""
    return lib().mbglu_last_backward_path()


def read_device_error() -> int:
    """Synchronises the current device, returns and clears its error word."""
    w = ctypes.c_int(0)
    st = lib().mbglu_read_device_error(ctypes.byref(w))
    if st != 0:
        raise MbgluError(st, "mbglu_read_device_error")
    return w.value


def set_launch_policy(policy: int) -> None:
    """0 serial, 1 programmatic dependent launch, 2 PDL + weight prefetch
    before the dependency wait (default; see include/mbglu.h for the contract)."""
    st = lib().mbglu_set_launch_policy(int(policy))
    if st != 0:
        raise MbgluError(st, "mbglu_set_launch_policy")


def get_launch_policy() -> int:
    return lib().mbglu_get_launch_policy()
