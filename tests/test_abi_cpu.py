"""The C-ABI library on a host without a GPU: it loads, exports every symbol
include/mbglu.h declares, and its host-side validation rejects bad arguments
before any CUDA call (pointers here are never dereferenced)."""
import ctypes
import os
import re

import pytest

import memory_bound_glu_gb300 as mb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mbglu.h")

OK, NULL, SHAPE, STRIDE, ALIGN, MODE, ALIAS, CUDA, TIMEOUT = range(9)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_api():
    assert declared_functions() == sorted(mb.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = mb.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {mb.LIB_PATH}").read()
    exported = set(re.findall(r" T (\w+)", out))
    assert set(declared_functions()) <= exported


def test_abi_version_matches_header():
    m = re.search(r"#define MBGLU_ABI_VERSION (\d+)", open(HEADER).read())
    assert mb.lib().mbglu_abi_version() == int(m.group(1))


def test_status_strings():
    lib = mb.lib()
    for code, tag in [(OK, b"MBGLU_OK"), (NULL, b"NULL"), (SHAPE, b"SHAPE"), (STRIDE, b"STRIDE"),
                      (ALIGN, b"ALIGN"), (MODE, b"MODE"), (ALIAS, b"ALIAS"), (CUDA, b"CUDA"),
                      (TIMEOUT, b"TIMEOUT")]:
        assert tag in lib.mbglu_status_string(code)
    assert b"unknown" in lib.mbglu_status_string(99)


# fake, never-dereferenced device addresses: 256-byte aligned and far apart
H, G, U, O, X, R, W = (0x7F0000000000 + i * (1 << 32) for i in range(7))


def gemv(h=H, ldh=64, g=G, ldg=64, u=U, ldu=64, o=O, ldo=32, M=2, N=32, K=64, mode=0):
    return mb.lib().glu_gemv(h, ldh, g, ldg, u, ldu, o, ldo, M, N, K, mode, None)


def norm(x=X, r=R, w=W, g=G, u=U, o=O, M=2, N=32, K=64, mode=1):
    return mb.lib().add_rmsnorm_glu(x, r, w, 1e-6, g, u, o, M, N, K, mode, None)


@pytest.mark.parametrize("kw,code", [
    (dict(mode=2), MODE), (dict(mode=-1), MODE),
    (dict(M=-1), SHAPE), (dict(N=-1), SHAPE), (dict(K=-1), SHAPE), (dict(M=65), SHAPE),
    # a batch of row blocks is checked whole before any block launches: out
    # overlaps h only from h's row 30 on, past the first block
    (dict(M=40, o=H + 2 * 64 * 30), ALIAS), (dict(M=40, ldh=64, h=O - 2 * 64 * 39), ALIAS),
    (dict(h=0), NULL), (dict(g=0), NULL), (dict(u=0), NULL), (dict(o=0), NULL),
    (dict(ldh=63), STRIDE), (dict(ldg=10), STRIDE), (dict(ldu=0), STRIDE), (dict(ldo=31), STRIDE),
    (dict(h=H + 1), ALIGN), (dict(g=G + 1), ALIGN), (dict(u=U + 3), ALIGN), (dict(o=O + 1), ALIGN),
    (dict(o=H), ALIAS), (dict(o=G + 128), ALIAS), (dict(o=U + 64 * 31 * 2), ALIAS),
    (dict(M=0), OK), (dict(N=0), OK), (dict(M=0, h=0, g=0, u=0, o=0), OK),
])
def test_glu_gemv_validation(kw, code):
    assert gemv(**kw) == code
    if code != OK:
        assert mb.lib().mbglu_last_variant() == 0


@pytest.mark.parametrize("kw,code", [
    (dict(mode=3), MODE), (dict(K=0), SHAPE), (dict(M=65), SHAPE), (dict(M=16, K=8192), SHAPE),
    (dict(M=40, K=8192), SHAPE),                      # one pass holds 16 rows of s: 16 * K <= 81920
    (dict(M=40, o=R + 2 * 64 * 30), ALIAS),           # out meets residual's row 30, past the first block
    (dict(M=40, r=X + 2 * 64 * 20), ALIAS),           # residual overlaps x partially, from row 20 on
    (dict(x=0), NULL), (dict(r=0), NULL), (dict(w=0), NULL), (dict(g=0), NULL), (dict(o=0), NULL),
    (dict(x=X + 1), ALIGN), (dict(r=R + 1), ALIGN), (dict(o=O + 1), ALIGN),
    (dict(o=X), ALIAS), (dict(o=R + 2), ALIAS), (dict(o=W), ALIAS), (dict(o=G), ALIAS),
    (dict(r=X + 2), ALIAS), (dict(r=G + 256), ALIAS), (dict(r=W), ALIAS),
    (dict(M=0), OK),
])
def test_add_rmsnorm_glu_validation(kw, code):
    assert norm(**kw) == code


def norm_strided(x=X, r=R, w=W, g=G, ldg=96, u=U, ldu=72, o=O, ldo=40, M=2, N=32, K=64, mode=1, ws=None,
                 wsb=256):
    return mb.lib().add_rmsnorm_glu_strided(x, r, w, 1e-6, g, ldg, u, ldu, o, ldo, M, N, K, mode, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ldg=63), STRIDE), (dict(ldu=10), STRIDE), (dict(ldo=31), STRIDE),
    (dict(mode=3), MODE), (dict(K=0), SHAPE), (dict(M=65), SHAPE),
    (dict(M=33, o=G - 2 * 40 * 32), ALIAS),   # only out's row 32 (the third block) meets gate_w
    (dict(g=G + 1), ALIGN), (dict(ws=X + 0x1000000 + 8), ALIGN), (dict(ws=X + 0x1000000, wsb=255), SHAPE),
    (dict(o=G + 2 * 96 * 31), ALIAS), (dict(r=U + 2 * 72 * 5), ALIAS), (dict(ws=O + 2 * 40), ALIAS),
    (dict(M=0), OK),
])
def test_add_rmsnorm_glu_strided_validation(kw, code):
    """Strides are checked against K and N, and the alias checks cover each
    strided operand's true extent (rows times its stride)."""
    assert norm_strided(**kw) == code
    assert mb.lib().mbglu_last_variant() == 0


def gates(a=X, lda=64, b=R, ldb=64, A=W, dt=W + 4096, g=O, ldg=32, be=H, ldbe=32, T=3, Hh=32):
    return mb.lib().gdn_gates(a, lda, b, ldb, A, dt, g, ldg, be, ldbe, T, Hh, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), SHAPE), (dict(Hh=-1), SHAPE),
    (dict(a=0), NULL), (dict(b=0), NULL), (dict(A=0), NULL), (dict(dt=0), NULL), (dict(g=0), NULL), (dict(be=0), NULL),
    (dict(lda=31), STRIDE), (dict(ldb=0), STRIDE), (dict(ldg=31), STRIDE), (dict(ldbe=8), STRIDE),
    (dict(a=X + 1), ALIGN), (dict(A=W + 2), ALIGN), (dict(g=O + 2), ALIGN), (dict(be=H + 1), ALIGN),
    (dict(g=X + 64), ALIAS), (dict(be=R + 2 * 64 * 2), ALIAS), (dict(g=W), ALIAS), (dict(be=O + 4 * 32 * 2), ALIAS),
    (dict(T=0), OK), (dict(Hh=0), OK),
])
def test_gdn_gates_validation(kw, code):
    """Host-side validation of gdn_gates (no GPU: rejections and no-op sizes)."""
    assert gates(**kw) == code
    assert mb.lib().mbglu_last_variant() == 0


def silu(x=X, ldx=64, o=O, ldo=32, M=2, N=32, mode=0):
    return mb.lib().silu_mul(x, ldx, o, ldo, M, N, mode, None)


@pytest.mark.parametrize("kw,code", [
    (dict(mode=2), MODE), (dict(M=-1), SHAPE), (dict(N=-1), SHAPE), (dict(N=2 ** 30), SHAPE),
    (dict(x=0), NULL), (dict(o=0), NULL),
    (dict(ldx=63), STRIDE), (dict(ldo=31), STRIDE),
    (dict(x=X + 1), ALIGN), (dict(o=O + 3), ALIGN),
    (dict(o=X), ALIAS), (dict(o=X + 64 * 2), ALIAS), (dict(o=X - 2 * 31), ALIAS),
    (dict(M=0), OK), (dict(N=0), OK), (dict(M=0, x=0, o=0), OK),
])
def test_silu_mul_validation(kw, code):
    """Host-side validation of silu_mul (no GPU: only rejections and the
    no-op sizes, which launch nothing)."""
    assert silu(**kw) == code
    assert mb.lib().mbglu_last_variant() == 0


def test_binding_rejects_cpu_tensors():
    import torch
    h = torch.zeros(2, 64, dtype=torch.bfloat16)
    w = torch.zeros(8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mb.glu_gemv(h, w, w)
    with pytest.raises(TypeError):
        mb.glu_gemv(h.float(), w, w)


def test_launch_policy_roundtrip_and_validation():
    lib = mb.lib()
    old = lib.mbglu_get_launch_policy()
    assert old == mb.POLICY_PREFETCH          # the default
    try:
        for p in (mb.POLICY_SERIAL, mb.POLICY_PDL, mb.POLICY_PREFETCH):
            assert lib.mbglu_set_launch_policy(p) == OK
            assert lib.mbglu_get_launch_policy() == p
        assert lib.mbglu_set_launch_policy(3) == MODE
        assert lib.mbglu_set_launch_policy(-1) == MODE
        assert lib.mbglu_get_launch_policy() == mb.POLICY_PREFETCH
    finally:
        lib.mbglu_set_launch_policy(old)


WS = 0x7F0000000000 + 9 * (1 << 32)


def norm_ws(ws=WS, nbytes=256, **kw):
    a = dict(x=X, r=R, w=W, g=G, u=U, o=O, M=2, N=32, K=64, mode=1)
    a.update(kw)
    return mb.lib().add_rmsnorm_glu_ws(a["x"], a["r"], a["w"], 1e-6, a["g"], a["u"], a["o"], a["M"], a["N"], a["K"],
                                       a["mode"], ws, nbytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), NULL), (dict(nbytes=255), SHAPE), (dict(ws=WS + 8), ALIGN),
    (dict(ws=X), ALIAS), (dict(ws=O + 64), ALIAS), (dict(ws=G + 1024), ALIAS),
    (dict(M=65), SHAPE), (dict(mode=2), MODE), (dict(x=0), NULL), (dict(M=0), OK),
    (dict(M=48, ws=X + 2 * 64 * 47), ALIAS),          # the workspace sits in x's last block
])
def test_add_rmsnorm_glu_ws_validation(kw, code):
    assert norm_ws(**kw) == code


D, GH, GG, GU, BW = (0x7F0000000000 + i * (1 << 32) for i in range(10, 15))


def bwd(h=H, ldh=64, g=G, ldg=64, u=U, ldu=64, d=D, ldd=32, gh=GH, ldgh=64, gg=GG, ldgg=64, gu=GU, ldgu=64,
        M=2, N=32, K=64, ws=BW, wsb=1 << 20):
    return mb.lib().glu_backward(h, ldh, g, ldg, u, ldu, d, ldd, gh, ldgh, gg, ldgg, gu, ldgu, M, N, K, ws, wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), SHAPE), (dict(N=-1), SHAPE), (dict(K=-1), SHAPE), (dict(M=65), SHAPE),
    (dict(h=0), NULL), (dict(d=0), NULL), (dict(ws=0), NULL), (dict(gg=0), NULL), (dict(gu=0), NULL),
    (dict(ldh=63), STRIDE), (dict(ldd=31), STRIDE), (dict(ldgh=60), STRIDE), (dict(ldgu=1), STRIDE),
    (dict(h=H + 1), ALIGN), (dict(gh=GH + 1), ALIGN), (dict(ws=BW + 8), ALIGN),
    (dict(wsb=1000), SHAPE),
    (dict(gh=H), ALIAS), (dict(gg=G + 64), ALIAS), (dict(gu=D), ALIAS), (dict(ws=GG), ALIAS),
    (dict(gu=GG + 2 * 64 * 31), ALIAS),
    (dict(K=0), OK), (dict(K=0, h=0, d=0, ws=0), OK), (dict(M=0, N=0), OK),
])
def test_glu_backward_validation(kw, code):
    """Host-side validation of glu_backward (no GPU: rejections and the
    shapes that launch nothing)."""
    assert bwd(**kw) == code
    assert mb.lib().mbglu_last_variant() == 0


def test_glu_backward_workspace_bytes():
    lib = mb.lib()
    # dG and dU in fp32, then one fp32 [M][K] partial per row split (N / 256, 1..48)
    # dG, dU [M][N] fp32, then the grad_h partials of one pass: 256 CTAs x
    # min(M, 8) rows, or 48 splits x min(M, 16) rows, whichever is larger
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert lib.glu_backward_workspace_bytes(4, 1000, 512) == 32000 + 256 * 4 * 512 * 4
    assert lib.glu_backward_workspace_bytes(16, 9728, 2560) == 16 * 9728 * 8 + 256 * 8 * 2560 * 4
    assert lib.glu_backward_workspace_bytes(1, 100000, 64) == 800000 + 256 * 64 * 4
    assert lib.glu_backward_workspace_bytes(64, 10, 10) == r256(64 * 10 * 8) + r256(256 * 8 * 10 * 4)
    assert lib.glu_backward_workspace_bytes(65, 10, 10) == 0 and lib.glu_backward_workspace_bytes(0, 10, 10) == 0


def _c_params():
    """{function: [parameter type category, ...]} from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"#.*", "", text)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.M | re.S):
        name, params = m.group(1), " ".join(m.group(2).split())
        cats = []
        for p in ([] if params in ("", "void") else params.split(",")):
            p = p.strip()
            if "*" in p or p.startswith("cudaStream_t"):
                cats.append("ptr")
            elif p.startswith("int64_t"):
                cats.append("i64")
            elif p.startswith("size_t"):
                cats.append("size")
            elif p.startswith("float"):
                cats.append("f32")
            elif p.split()[0] in ("int", "mbglu_mode", "mbglu_status"):
                cats.append("i32")
            else:
                cats.append("?" + p)
        out[name] = cats
    return out


def _ctypes_category(t):
    if t is ctypes.c_void_p or (isinstance(t, type) and issubclass(t, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int64: "i64", ctypes.c_size_t: "size", ctypes.c_float: "f32", ctypes.c_int: "i32"}[t]


def test_binding_argument_types_match_the_prototypes():
    """Every entry point the binding declares argument types for takes, in
    the header, the same number of arguments of the same kinds (pointer,
    64-bit, size_t, float, 32-bit), so ctypes marshals each call as the
    C ABI expects."""
    protos = _c_params()
    lib = mb.lib()
    checked = 0
    for name in mb.EXPORTS:
        fn = getattr(lib, name)
        if fn.argtypes is None:
            assert protos[name] == [], name
            continue
        assert [_ctypes_category(t) for t in fn.argtypes] == protos[name], name
        checked += 1
    assert checked >= 10
