"""ctypes loader for the fp64 CPU oracle (``mbglu_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the
product path (``memory_bound_glu_gb300``) never does, and this package never
imports the product path.

bf16 values are exchanged as raw bit patterns in ``numpy.uint16`` arrays.
Sources cited in ``mbglu_oracle.c``: DeepSpeed PR #8602 ("Plan B: Dual-Weight
GEMV" comment; "fused_glu" and "old-ki" commits) and PR #9057 ("Changes").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mbglu_oracle.c")
LIB = os.path.join(HERE, "libmbglu_oracle.so")

MODE_FUSED = 0
MODE_HF = 1
MODES = {"fused": MODE_FUSED, "hf": MODE_HF, MODE_FUSED: MODE_FUSED, MODE_HF: MODE_HF}

_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts
# evaluate every binary64 expression identically.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(src: str = SRC, out: str = LIB, extra_cflags=()) -> str:
    """Compile the oracle with gcc (plain C11, libm, pthreads)."""
    cmd = ["gcc", *CFLAGS, *extra_cflags, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64, i32 = ctypes.c_int64, ctypes.c_int
    lib.oracle_abi_version.restype = i32
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_round_array.argtypes = [f64p, u16p, i64]
    lib.oracle_bf16_round_array.restype = None
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_glu_gemv.argtypes = [u16p, i64, u16p, i64, u16p, i64, u16p, i64,
                                    i32, i32, i32, i32, f64p, f64p, f64p, f64p, i32]
    lib.oracle_glu_gemv.restype = i32
    lib.oracle_add_rmsnorm.argtypes = [u16p, u16p, u16p, ctypes.c_float, i32, i32, u16p, u16p]
    lib.oracle_add_rmsnorm.restype = i32
    lib.oracle_add_rmsnorm_glu.argtypes = [u16p, u16p, u16p, ctypes.c_float, u16p, u16p,
                                           u16p, i32, i32, i32, i32, u16p, i32]
    lib.oracle_add_rmsnorm_glu.restype = i32
    lib.oracle_silu_mul.argtypes = [u16p, i64, u16p, i64, i32, i32, i32]
    lib.oracle_silu_mul.restype = i32
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_gdn_gates.argtypes = [u16p, i64, u16p, i64, f32p, f32p, f64p, u16p, i32, i32]
    lib.oracle_gdn_gates.restype = i32
    lib.oracle_glu_backward.argtypes = [u16p, i64, u16p, i64, u16p, i64, u16p, i64, i32, i32, i32,
                                        f64p, f64p, f64p, f64p, f64p, i32]
    lib.oracle_glu_backward.restype = i32
    return lib


def load(path: str = LIB, rebuild_if_missing: bool = True):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path == LIB and _lib is not None:
        return _lib
    stale = path == LIB and os.path.exists(path) and os.path.getmtime(path) < os.path.getmtime(SRC)
    if not os.path.exists(path) or stale:
        if not rebuild_if_missing:
            raise FileNotFoundError(path)
        build(out=path)
    lib = _bind(ctypes.CDLL(path))
    if path == LIB:
        _lib = lib
    return lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _ptr(a, ctype=ctypes.c_uint16):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def bf16_round(x: float, lib=None) -> int:
    return int((lib or load()).oracle_bf16_round(float(x)))


def bf16_round_array(x, lib=None) -> np.ndarray:
    """bf16 bits of every binary64 value in x (bf16_round, elementwise)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    (lib or load()).oracle_bf16_round_array(_ptr(x, ctypes.c_double), _ptr(out), x.size)
    return out


def bf16_to_float(bits: int, lib=None) -> float:
    return float((lib or load()).oracle_bf16_to_double(int(bits)))


def silu(x: float, lib=None) -> float:
    return float((lib or load()).oracle_silu(float(x)))


def glu_gemv(h, gate_w, up_w, mode="fused", diagnostics=False, nthreads=None, lib=None):
    """out[M,N] = GLU(h[M,K], gate_w[N,K], up_w[N,K]) as bf16 bits.

    With ``diagnostics`` also returns a dict of binary64 arrays G, U (the dot
    products) and Ag, Au (the sums of |h*w|, used by the tests' conditioning
    floor).
    """
    lib = lib or load()
    h, gate_w, up_w = (np.ascontiguousarray(_u16(a)) for a in (h, gate_w, up_w))
    M, K = h.shape
    N, K2 = gate_w.shape
    if K2 != K or up_w.shape != (N, K):
        raise ValueError("shape mismatch")
    out = np.zeros((M, N), dtype=np.uint16)
    diag = {k: np.zeros((M, N), dtype=np.float64) for k in ("G", "U", "Ag", "Au")} if diagnostics else {}
    rc = lib.oracle_glu_gemv(_ptr(h), K, _ptr(gate_w), K, _ptr(up_w), K, _ptr(out), N,
                             M, N, K, MODES[mode],
                             *(_ptr(diag.get(k), ctypes.c_double) for k in ("G", "U", "Ag", "Au")),
                             int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_glu_gemv failed: {rc}")
    return (out, diag) if diagnostics else out


def add_rmsnorm(x, residual, norm_w, eps, lib=None):
    """Returns (s, h): the bf16 residual sum and the normed bf16 rows."""
    lib = lib or load()
    x, residual = (np.ascontiguousarray(_u16(a)) for a in (x, residual))
    norm_w = np.ascontiguousarray(_u16(norm_w))
    M, K = x.shape
    s = np.zeros((M, K), dtype=np.uint16)
    h = np.zeros((M, K), dtype=np.uint16)
    rc = lib.oracle_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(norm_w), float(eps), M, K, _ptr(s), _ptr(h))
    if rc != 0:
        raise RuntimeError(f"oracle_add_rmsnorm failed: {rc}")
    return s, h


def add_rmsnorm_glu(x, residual, norm_w, eps, gate_w, up_w, mode="hf", nthreads=None, lib=None):
    """Returns (out, residual_out, h): the fused segment's outputs."""
    lib = lib or load()
    x = np.ascontiguousarray(_u16(x))
    res = np.array(_u16(residual), dtype=np.uint16, copy=True, order="C")
    norm_w, gate_w, up_w = (np.ascontiguousarray(_u16(a)) for a in (norm_w, gate_w, up_w))
    M, K = x.shape
    N = gate_w.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    h = np.zeros((M, K), dtype=np.uint16)
    rc = lib.oracle_add_rmsnorm_glu(_ptr(x), _ptr(res), _ptr(norm_w), float(eps), _ptr(gate_w), _ptr(up_w),
                                    _ptr(out), M, N, K, MODES[mode], _ptr(h),
                                    int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_add_rmsnorm_glu failed: {rc}")
    return out, res, h


def silu_mul(x, mode="fused", lib=None):
    """out[M,N] = epilogue(x[:, :N], x[:, N:2N]) on the halves layout (x is
    [M, 2N] bf16 bits, rows may be wider); see oracle_silu_mul."""
    x = _u16(x)
    if x.ndim != 2 or (x.size and x.strides[1] != 2):
        x = np.ascontiguousarray(x).reshape(x.shape[0], -1)
    M, W = x.shape
    N = W // 2
    out = np.zeros((M, N), dtype=np.uint16)
    ldx = x.strides[0] // 2 if M > 1 else W   # a lone row's stride is arbitrary (numpy gives 0 to a new axis)
    st = (lib or load()).oracle_silu_mul(_ptr(x), ldx, _ptr(out), N, M, N, MODES[mode])
    if st != 0:
        raise ValueError("oracle_silu_mul: bad arguments")
    return out


def gdn_gates(a, b, A_log, dt_bias, lib=None):
    """(g [T,H] float64, beta [T,H] bf16 bits) from a, b [T,H] bf16 bits and
    A_log, dt_bias [H] float32; see oracle_gdn_gates."""
    a, b = np.ascontiguousarray(_u16(a)), np.ascontiguousarray(_u16(b))
    T, H = a.shape
    A_log = np.ascontiguousarray(A_log, dtype=np.float32)
    dt_bias = np.ascontiguousarray(dt_bias, dtype=np.float32)
    g = np.zeros((T, H), dtype=np.float64)
    beta = np.zeros((T, H), dtype=np.uint16)
    st = (lib or load()).oracle_gdn_gates(_ptr(a), H, _ptr(b), H, _ptr(A_log, ctypes.c_float),
                                          _ptr(dt_bias, ctypes.c_float), _ptr(g, ctypes.c_double), _ptr(beta), T, H)
    if st != 0:
        raise ValueError("oracle_gdn_gates: bad arguments")
    return g, beta


def glu_backward(h, gate_w, up_w, dout, nthreads=None, lib=None):
    """Gradients of out = SiLU(h Wg^T) * (h Wu^T) for an upstream dout, in
    binary64: (grad_h [M,K], grad_gate [N,K], grad_up [N,K]); inputs are bf16
    bits (see oracle_glu_backward)."""
    h, gw, uw, d = (np.ascontiguousarray(_u16(a)) for a in (h, gate_w, up_w, dout))
    M, K = h.shape
    N = gw.shape[0]
    dG = np.zeros((M, N)); dU = np.zeros((M, N))
    gh = np.zeros((M, K)); gg = np.zeros((N, K)); gu = np.zeros((N, K))
    f = lambda a: _ptr(a, ctypes.c_double)  # noqa: E731
    st = (lib or load()).oracle_glu_backward(_ptr(h), K, _ptr(gw), K, _ptr(uw), K, _ptr(d), N, M, N, K,
                                             f(dG), f(dU), f(gh), f(gg), f(gu),
                                             nthreads or default_threads())
    if st != 0:
        raise ValueError("oracle_glu_backward: bad arguments")
    return gh, gg, gu
