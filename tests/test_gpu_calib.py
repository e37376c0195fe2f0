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


def test_calibration_study_held_out():
    """The calibration study (the MVP's block-max and attention-RMSE analogues
    on the seeded llama8b-shaped data, fp16 scales, m = 64, 3-bit codes).
    Calibration sample: K and V of (sequence 0, kv head 0), positions
    0..4095.  Held out: sequences 1..2, kv heads 0..3, positions 0..1023.
    Printed per rotation: the sample's mean squared reconstruction error per
    element; on the held-out vectors the mean block crest factor
    max|y| / rms(y) of the rotated blocks, the relative reconstruction error
    sum (x - x_hat)^2 / sum x^2, and the relative RMS error of decode attention
    over the quantised cache (oracle, fp64) against exact attention over the
    fp16 K/V (4 query heads per kv head, N = 1024).  Asserts that every search
    keeps the sample error at or below its start."""
    import torch
    import hadamard_rotated_bit_kvq3_gb300 as K
    d, blk, n_cal = 128, 64, 4096
    spec = I.DataSpec(d, 8, 1001, 0.03, 20.0)
    x_cal = np.concatenate([I.kv_rows_np(spec, w, 0, 0, 0, n_cal) for w in (0, 1)])
    desc = _desc(K, d, blk, "f16", 3)
    xd = torch.as_tensor(x_cal, device="cuda")
    ws = torch.empty(K.kvq3_calibrate_workspace_size(desc, 64), dtype=torch.uint8, device="cuda")
    held = [(b, h) for b in (1, 2) for h in range(4)]
    N, G = 1024, 4

    def evaluate(U):
        crest, err, tot, att = [], 0.0, 0.0, []
        lay = O.Layout(d, 1, blk, "f16", 16, 1, N // 16, N // 16)
        for b, h in held:
            k = I.kv_rows_np(spec, 0, b, h, 0, N)
            v = I.kv_rows_np(spec, 1, b, h, 0, N)
            for x in (k, v):
                y = x.astype(np.float64) @ U.T
                yb = y.reshape(-1, d // blk, blk)
                crest.append((np.abs(yb).max(-1) / np.sqrt((yb ** 2).mean(-1))).ravel())
                c, sq, _ = O.quantize(y, blk, 1e-6, "f16")
                yh = (c.reshape(-1, d // blk, blk) * sq[..., None]).reshape(-1, d)
                err += float(((y - yh) ** 2).sum())
                tot += float((y ** 2).sum())
            pool = np.zeros(lay.pool_bytes, np.uint8)
            O.write(pool, lay, U, k[:, None], v[:, None], np.zeros(N, np.int32), np.arange(N))
            q = I.q_np(spec, b + 1, 8 * G)[b, h * G:(h + 1) * G][None]
            o_q = O.decode(pool, lay, U, q, np.array([N]))[0]
            o = np.stack([O.attention_plain(q[0, g], k, v, 1.0 / np.sqrt(d)) for g in range(G)])
            att.append(np.sqrt(((o_q - o) ** 2).mean()) / np.sqrt((o ** 2).mean()))
        return float(np.concatenate(crest).mean()), err / tot, float(np.mean(att))

    def train_mse(signs, q, r=None):
        return float(O.calib_sse(x_cal.astype(np.float64), signs, q, blk, "f16", quats_r=r).sum()) / x_cal.size

    rows = []
    s1, q_id = O.rotation_params(d, 42, True, False)
    s3, q3 = O.rotation_params(d, 42)
    _, _, r7 = O.rotation_params_pair(d, 42)
    rows.append(("none", None, np.eye(d)))
    rows.append(("H D", train_mse(s1, q_id), O.rotation_matrix(s1, q_id)))
    rows.append(("H D + random SO(4) (seed 42)", train_mse(s3, q3), O.rotation_matrix(s3, q3)))
    start3 = train_mse(s3, q3)
    # one quaternion per block, from the random set and from the identity
    for name, flags, start, rounds in (("calibrated from the random set", 3, start3, 40),
                                       ("calibrated from the identity", 1, train_mse(s1, q_id), 60)):
        rot = K.Rotation(d, 42, flags)
        q, _ = K.kvq3_calibrate_so4(rot.handle, desc, xd, rounds=rounds, num_candidates=64, step=0.5, seed=7,
                                    workspace=ws)
        qq = q.astype(np.float64)
        tm = train_mse(s3, qq)
        assert tm <= start * (1 + 1e-4)
        rows.append(("H D + SO(4) " + name, tm, O.rotation_matrix(s3, qq)))
    # the general two-quaternion blocks, from the random p with q = 1 and from a random pair
    for name, flags, start in (("pairs calibrated from the random p, q = 1", 3, start3),
                               ("pairs calibrated from a random pair (seed 42)", 7, train_mse(s3, q3, r7))):
        rot = K.Rotation(d, 42, flags)
        q, r, _ = K.kvq3_calibrate_so4_pair(rot.handle, desc, xd, rounds=40, num_candidates=64, step=0.5, seed=7,
                                            workspace=ws)
        qq, rr = q.astype(np.float64), r.astype(np.float64)
        tm = train_mse(s3, qq, rr)
        assert tm <= start * (1 + 1e-4)
        rows.append(("H D + SO(4) " + name, tm, O.rotation_matrix(s3, qq, rr)))
    print("\n| Rotation | Train MSE | Held-out crest | Held-out rel. reconstruction error | Held-out attention rel. RMSE |")
    for name, tm, U in rows:
        crest, rel, att = evaluate(U)
        print(f"| {name} | {'-' if tm is None else f'{tm:.4f}'} | {crest:.3f} | {rel:.4f} | {att:.4f} |")
