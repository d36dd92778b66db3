"""glu_backward at full size: the K = 2560, N = 9728 layer at batch 1, 8 and 16,
against the fp64 oracle (grad_h whole, 512 sampled rows of each weight
gradient).  Collected after every other GPU test file, so that with -x a
failure here leaves them all already run."""
import numpy as np
import pytest
import torch

import glu_inputs as gi
import test_backward_gpu as bw

pytestmark = pytest.mark.gpu

mb = pytest.importorskip("memory_bound_glu_gb300")
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def test_backward_full_size_headline_layer():
    """K = 2560, N = 9728 (the headline layer) at batch 1, 8 and 16: every
    gradient on the GPU; grad_h whole and 512 sampled rows of the weight
    gradients against the oracle."""
    w = gi.WORKLOADS["gemv_k2560_n9728"]
    g, u = gi.layer_weights(w, 0)
    rows = np.sort(np.random.default_rng(2).choice(w.N, 512, replace=False))
    for M in (1, 8, 16):
        h = gi.hidden(w, M)
        d = gi.normal_bf16((M, w.N), 1.0, M, "bwf-d")
        got = mb.glu_backward(h.to(DEV), g.to(DEV), u.to(DEV), d.to(DEV))
        torch.cuda.synchronize()
        bw._check(tuple(t.cpu() for t in got), h, g, u, d, f"full size M={M}", rows=rows)
    assert mb.read_device_error() == 0
