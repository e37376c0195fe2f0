"""The seeded input generator: numpy and torch paths give the same bits."""
import numpy as np
import pytest

import kvq3_inputs as I


def test_torch_generator_matches_numpy_bitwise():
    torch = pytest.importorskip("torch")
    spec = I.DataSpec(128, 8, 1001, 0.03, 20.0)
    for which, b, h, t0, n in ((0, 3, 2, 1000, 3000), (1, 0, 7, 5, 777), (0, 15, 0, 32000, 768)):
        a = I.kv_rows_np(spec, which, b, h, t0, n)
        t = I.kv_rows_torch(spec, which, b, h, t0, n, "cpu").numpy()
        assert np.array_equal(a.view(np.uint16), t.view(np.uint16))


def test_fp16_rounding_helper_single_rounding():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp(rng.uniform(-20, 10, 200000))
    x = x[np.abs(x) < 65504]
    got = I._round_fp16_torch(torch.tensor(x)).numpy()
    assert np.array_equal(got.view(np.uint16), x.astype(np.float16).view(np.uint16))


def test_slices_are_consistent():
    spec = I.DataSpec(64, 2, 5, 0.05, 30.0)
    whole = I.kv_rows_np(spec, 0, 1, 1, 0, 100)
    part = I.kv_rows_np(spec, 0, 1, 1, 37, 20)
    assert np.array_equal(whole[37:57], part)


def test_workload_shapes():
    w = I.workloads()
    assert w["llama8b"].group == 4 and w["long70b"].group == 8 and w["ragged"].group == 4
    lens = I.seq_lens_np(w["ragged"].data.seed, 64, 1024, 65536)
    assert lens.min() >= 1024 and lens.max() <= 65536 and len(set(lens.tolist())) > 50
    table, n = I.page_table_np(1, np.array([20, 0, 33]), 16, 3)
    assert n == 2 + 0 + 3
    assert sorted(table[table >= 0].tolist()) == list(range(5))
