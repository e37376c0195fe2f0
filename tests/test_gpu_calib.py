"""SO(4) calibration on the GPU: the objective kernel (kvq3_calib_sse) against
the oracle's (oracle.calib_sse), and the search (kvq3_calibrate_so4).

"Orthogonally mixed 3-bit KV cache", Implementation notes: the rotations are
calibrated by minimising the reconstruction MSE after quantisation.  The
objective is fp32 on the GPU against fp64 in the oracle: per block within
1e-4 relative.  The search is checked by its properties: unit quaternions,
no block's error above the starting one (the current set is always a
candidate), and a final error that the oracle reproduces."""
import numpy as np
import pytest

import kvq3_inputs as I
from oracle import kvq3_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_kvq3_gb300  # noqa: F401


def _desc(K, d, block, kind, bits):
    return K.CacheDesc(d, 1, block, bits, K.SCALE_TYPES[kind], 1e-6, 16, 1, 1, 0, 1)


def _sample(d, n, seed):
    spec = I.DataSpec(d, 1, seed, 0.03, 20.0)
    return I.kv_rows_np(spec, 0, 0, 0, 0, n)     # fp16 [n][d]


@pytest.mark.parametrize("d,block,kind,bits", [(128, 64, "f16", 3), (128, 64, "e4m3", 3), (128, 32, "f32", 4),
                                               (64, 32, "f16", 2), (256, 64, "e4m3zp", 3), (128, 64, "e4m3zp", 3)])
def test_calib_sse_matches_oracle(d, block, kind, bits):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    rot = K.Rotation(d, 42, 3)
    signs, q0 = O.rotation_params(d, 42)
    rng = np.random.default_rng(d + bits)
    P = 5
    cand = rng.standard_normal((P, d // 4, 4))
    cand[0] = q0
    cand /= np.linalg.norm(cand, axis=2, keepdims=True)
    cand = cand.astype(np.float32)
    x = _sample(d, 300, 9)
    sse = torch.empty((P, d // block), dtype=torch.float64, device="cuda")
    K.kvq3_calib_sse(rot.handle, _desc(K, d, block, kind, bits), torch.as_tensor(cand, device="cuda"),
                     torch.as_tensor(x, device="cuda"), sse)
    got = sse.cpu().numpy()
    for p in range(P):
        ref = O.calib_sse(x.astype(np.float64), signs, cand[p].astype(np.float64), block, kind, bits)
        assert np.all(np.abs(got[p] - ref) <= 1e-4 * ref), (p, got[p], ref)


@pytest.mark.parametrize("kind", ["f16", "e4m3zp"])
def test_calibrate_so4_lowers_the_error(kind):
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    d, block, n = 128, 64, 1024
    rot = K.Rotation(d, 42, 3)
    signs, q0 = O.rotation_params(d, 42)
    desc = _desc(K, d, block, kind, 3)
    x = _sample(d, n, 21)
    xd = torch.as_tensor(x, device="cuda")
    ws = torch.empty(K.kvq3_calibrate_workspace_size(desc, 32), dtype=torch.uint8, device="cuda")
    q, sse = K.kvq3_calibrate_so4(rot.handle, desc, xd, rounds=10, num_candidates=32, step=0.5, seed=7,
                                  workspace=ws)
    assert q.shape == (d // 4, 4) and np.all(np.abs(np.linalg.norm(q, axis=1) - 1.0) < 1e-6)
    before = O.calib_sse(x.astype(np.float64), signs, q0.astype(np.float32).astype(np.float64), block, kind)
    after = O.calib_sse(x.astype(np.float64), signs, q.astype(np.float64), block, kind)
    print(f"{kind}: reconstruction error {before.sum():.4f} -> {after.sum():.4f} "
          f"({100 * (1 - after.sum() / before.sum()):.1f} % lower)")
    assert np.all(after <= before * (1 + 1e-4))
    assert np.all(np.abs(sse - after) <= 1e-4 * after)
    # zero rounds return the starting quaternions (in fp32)
    q0b, _ = K.kvq3_calibrate_so4(rot.handle, desc, xd, rounds=0, num_candidates=2, step=0.5, seed=7,
                                  workspace=ws)
    assert np.array_equal(q0b, q0.astype(np.float32))


def test_calibrate_rejects_bad_arguments():
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    rot = K.Rotation(128, 42, 3)
    desc = _desc(K, 128, 64, "f16", 3)
    x = torch.zeros((16, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(K.Kvq3Error):
        K.kvq3_calibrate_workspace_size(desc, 1)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.Kvq3Error) as e:
        K.kvq3_calibrate_so4(rot.handle, desc, x, 1, 4, 0.5, 1, small)
    assert e.value.status == 4
