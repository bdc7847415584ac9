"""The seeded synthetic inputs follow their stated recipe: shapes, storage
formats, outlier channels, the planted low-rank spectrum (through Weyl's
inequality), independent streams per tensor, and reproducibility."""
import numpy as np

import workloads


def _is_bf16(x):
    return np.array_equal(workloads.to_bf16_values(x), x)


def test_activations_recipe():
    case = workloads.CASES["attn_out"]
    X = workloads.make_activations(case)
    assert X.shape == (4096, 3072) and X.dtype == np.float32 and _is_bf16(X)
    std = X.std(axis=0)
    outliers = np.nonzero(std > 10)[0]
    assert len(outliers) == case.outlier_channels == round(0.01 * 3072)   # 1% of channels
    assert np.allclose(std[outliers], 50.0, rtol=0.05)                    # x50
    assert np.allclose(np.delete(std, outliers), 1.0, atol=0.05)          # N(0, 1)
    assert np.array_equal(X, workloads.make_activations(case))            # reproducible
    tiny = workloads.make_activations(workloads.CASES["tiny"])
    assert tiny.shape == (128, 256) and np.sum(tiny.std(axis=0) > 10) == 4   # 4 channels x40


def test_weights_recipe_planted_spectrum():
    """W = N(0, 0.02^2) noise + a planted part with singular values 3/i: by
    Weyl's inequality each singular value of W lies within the noise's
    spectral norm (about 0.02 (sqrt N + sqrt K)) of the planted one."""
    case = workloads.CASES["tiny"]
    W, b = workloads.make_weights(case)
    assert W.shape == (256, 256) and W.dtype == np.float32
    sv = np.linalg.svd(W.astype(np.float64), compute_uv=False)
    noise_norm = 0.02 * (np.sqrt(256) + np.sqrt(256)) * 1.2
    planted = np.zeros(256)
    planted[:4] = 3.0 / np.arange(1, 5)
    assert np.all(np.abs(sv - planted) <= noise_norm), sv[:6]
    assert b.shape == (256,) and _is_bf16(b)
    assert 0.005 < np.std(workloads.make_weights(workloads.CASES["attn_out"])[1]) < 0.015


def test_streams_are_independent_and_reproducible():
    c1, c2 = workloads.CASES["fc1"], workloads.CASES["fc2"]
    W2, b2 = workloads.make_fc2_weights(c2)
    assert W2.shape == (3072, 12288) and b2.shape == (3072,)
    W2b, _ = workloads.make_fc2_weights(c2)
    assert np.array_equal(W2, W2b)
    # fc2's noise is not fc1's (same seed, later child streams)
    W1, _ = workloads.make_weights(c1)
    assert not np.allclose(W1[:64, :64], W2[:64, :64])
    # AWQ blocks: one X, independent weight sets
    assert (workloads.AWQ_K, workloads.AWQ_N, workloads.AWQ_BLOCKS) == (3072, 18432, 57)
    Wa0, ba0 = workloads.make_awq_weights(0, N=512)
    Wa1, _ = workloads.make_awq_weights(1, N=512)
    assert Wa0.shape == (512, 3072) and not np.allclose(Wa0, Wa1)
    assert abs(Wa0.std() - 0.02) < 0.001 and _is_bf16(ba0)
    Xa = workloads.make_awq_activations(4)
    assert Xa.shape == (4, 3072) and _is_bf16(Xa)
    assert np.array_equal(Xa[:1], workloads.make_awq_activations(1))  # one conditioning stream


def test_qk_norm_weights_recipe():
    wq, wk = workloads.make_qk_norm_weights()
    assert wq.shape == wk.shape == (128,) and _is_bf16(wq) and _is_bf16(wk)
    assert abs(wq.mean() - 1.0) < 0.05 and 0.05 < wq.std() < 0.15
    assert not np.array_equal(wq, wk)
