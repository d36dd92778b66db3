"""The seeded input generators (glu_inputs.py) shared by the oracle and the
GPU path: deterministic, distinct per name, and shaped as the workloads state
-- including the outlier reading (whole rows and columns scaled x50 once) and
the bytes each call must move."""
import numpy as np
import torch

import glu_inputs as gi


def test_seeds_are_deterministic_and_distinct():
    a = gi.bits(gi.normal_bf16((64, 32), 1.0, 0, "w", "gate", 3))
    b = gi.bits(gi.normal_bf16((64, 32), 1.0, 0, "w", "gate", 3))
    c = gi.bits(gi.normal_bf16((64, 32), 1.0, 0, "w", "gate", 4))
    d = gi.bits(gi.normal_bf16((64, 32), 1.0, 1, "w", "gate", 3))
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    assert gi.derive_seed(0, "x") == gi.derive_seed(0, "x") != gi.derive_seed(0, "y")


def test_outlier_weights_scale_whole_rows_and_columns_once():
    """round(0.005 N) rows and round(0.005 K) columns scaled by 50 once (the
    crossings too), about 1% of the entries: the reading of "1% of weight
    entries scaled x50 (outlier rows/columns)"."""
    N, K = 1200, 800
    w = gi.outlier_weight_bf16(N, K, 0.02, 0, "out", "gate", 0).float().numpy()
    row_std, col_std = w.std(axis=1), w.std(axis=0)
    hot_rows = np.nonzero(row_std > 10 * np.median(row_std))[0]
    assert hot_rows.size == round(0.005 * N)
    cold = np.setdiff1d(np.arange(N), hot_rows)
    col_std_cold = w[cold].std(axis=0)
    hot_cols = np.nonzero(col_std_cold > 10 * np.median(col_std_cold))[0]
    assert hot_cols.size == round(0.005 * K)
    assert abs(np.median(w[np.ix_(cold, hot_cols)].std(axis=0)) / 0.02 - 50) < 5
    assert abs(w[np.ix_(hot_rows, hot_cols)].std() / 0.02 - 50) < 15     # crossings: x50, not x2500
    frac = (hot_rows.size * K + hot_cols.size * N - hot_rows.size * hot_cols.size) / (N * K)
    assert 0.009 < frac < 0.011


def test_workload_bytes_per_call():
    w = gi.WORKLOADS["gemv_k2560_n9728"]
    assert w.algorithmic_bytes(1) == 2 * 9728 * 2560 * 2 + 2560 * 2 + 9728 * 2 == 99639296
    n = gi.WORKLOADS["norm_gemv_k2560_n9728"]
    assert n.algorithmic_bytes(4) == 2 * 9728 * 2560 * 2 + 4 * 9728 * 2 + 3 * 4 * 2560 * 2 + 2560 * 2
    s = gi.WORKLOADS["silu_mul_m4096_n9728"]
    assert s.algorithmic_bytes(4096) == 4096 * 9728 * 2 * 3 and s.weight_bytes() == 0
    g = gi.WORKLOADS["gdn_gates_t262144_h32"]
    assert g.algorithmic_bytes(262144) == 262144 * 32 * (2 + 2 + 4 + 2) + 2 * 32 * 4


def test_generator_shapes_and_types():
    s = gi.WORKLOADS["silu_mul_m4096_n9728"]
    x = gi.projections(s, 3, 1)
    assert x.shape == (3, 2 * 9728) and x.dtype == torch.bfloat16
    g = gi.WORKLOADS["gdn_gates_t262144_h32"]
    a, b, A_log, dt = gi.gdn_inputs(g, 5, 2)
    assert a.shape == b.shape == (5, 32) and a.dtype == torch.bfloat16
    assert A_log.shape == dt.shape == (32,) and A_log.dtype == torch.float32
    assert not torch.equal(a, b)
