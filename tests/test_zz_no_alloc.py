"""add_rmsnorm_glu_noalloc: the single-kernel norm + GLU path for callers that
cannot allocate device memory (for instance code that runs under a runtime
owning all device memory, or inside stream capture where cudaMalloc is not
allowed).  Its scratch is a fixed array inside the library, so the caller
passes only the op's own inputs and outputs.

This file is collected last on purpose: a failure here leaves every other
test already run.  It calls the entry point through the C ABI, twice in a
row -- the second call reads the residual the first one wrote, and finds the
library's scratch where the first call left it -- and checks each result
against the existing add_rmsnorm_glu entry point within the parity tolerance.
"""
import ctypes

import numpy as np
import pytest
import torch

import glu_inputs as gi
import tolerance as tol

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")


def _call_noalloc(x, residual, norm_w, eps, gate_w, up_w, out, mode):
    M, K = x.shape
    N = gate_w.shape[0]
    lib = mb.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.add_rmsnorm_glu_noalloc(x.data_ptr(), residual.data_ptr(), norm_w.data_ptr(), float(eps),
                                       gate_w.data_ptr(), up_w.data_ptr(), out.data_ptr(), M, N, K,
                                       mb.MODE_HF if mode == "hf" else mb.MODE_FUSED, stream)


def _scratch_words(count=64):
    """The library's scratch array as it stands (synchronous read)."""
    words = (ctypes.c_int * count)()
    st = mb.lib().mbglu_noalloc_scratch_read(words, count)
    assert st == 0, mb.lib().mbglu_status_string(st)
    return np.array(words[:], dtype=np.int64)


# M = 20 runs as two row blocks (16 + 4), each a single kernel on the same array
@pytest.mark.parametrize("M,mode", [(1, "hf"), (4, "fused"), (8, "hf"), (20, "hf")])
def test_noalloc_matches_the_existing_entry_point_twice_in_a_row(M, mode):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    N, K = 3000, 2560
    blocks = -(-M // mb.BLOCK_M)
    w = gi.normal_bf16((K,), 0.1, M, "na-w").to(dev)
    r0 = gi.normal_bf16((M, K), 1.0, M, "na-r").to(dev)
    r_ref, r_na = r0.clone(), r0.clone()
    for call in range(2):
        x = gi.normal_bf16((M, K), 1.0, M, "na-x", call).to(dev)
        g = gi.normal_bf16((N, K), K ** -0.5, M, "na-g", call).to(dev)
        u = gi.normal_bf16((N, K), K ** -0.5, M, "na-u", call).to(dev)
        ref = mb.add_rmsnorm_glu(x, r_ref, w, 1e-6, g, u, mode=mode)       # existing entry point (two kernels)
        assert mb.lib().mbglu_last_single_kernel_blocks() == 0
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        st = _call_noalloc(x, r_na, w, 1e-6, g, u, out, mode)
        assert st == 0, mb.lib().mbglu_status_string(st)
        # every row block ran as the single kernel that uses the scratch
        assert mb.lib().mbglu_last_single_kernel_blocks() == blocks
        torch.cuda.synchronize()
        # the residual update is one correctly rounded addition: identical bits
        assert torch.equal(r_na.view(torch.int16), r_ref.view(torch.int16)), f"residual differs on call {call}"
        stats = tol.compare(gi.bits(out.cpu()), gi.bits(ref.cpu()))
        assert tol.passes(stats), (call, stats)
        # the kernel returns its arrival counters to zero
        assert not _scratch_words().any(), f"scratch not left at zero after call {call}"
    assert mb.read_device_error() == 0


def test_noalloc_scratch_is_left_at_zero():
    """Each call clears the counters first and the kernel returns them to
    zero: read back through the diagnostics export after each call."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    M, N, K = 2, 700, 1024
    x = gi.normal_bf16((M, K), 1.0, 1, "nz-x").to(dev)
    r = gi.normal_bf16((M, K), 1.0, 1, "nz-r").to(dev)
    w = gi.normal_bf16((K,), 0.1, 1, "nz-w").to(dev)
    g = gi.normal_bf16((N, K), K ** -0.5, 1, "nz-g").to(dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for _ in range(2):
        assert _call_noalloc(x, r, w, 1e-6, g, g, out, "hf") == 0
        assert mb.lib().mbglu_last_single_kernel_blocks() == 1
        words = _scratch_words()
        assert not words.any(), words[:8]
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert mb.read_device_error() == 0
