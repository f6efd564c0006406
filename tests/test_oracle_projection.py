"""Pins of the oracle's per-head projection (query absorption q_nope . w_kc,
output projection o_latent . w_vc), on the CPU: brute-force loops on tiny
inputs, a closed form (identity weights copy the input) and head
independence."""
import numpy as np
import torch

import oracle


def _bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _vals(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_projection_matches_brute_force():
    rng = np.random.default_rng(1)
    M, H, K, N = 3, 2, 5, 4
    xb, wb = _bits(rng.standard_normal((M, H, K))), _bits(rng.standard_normal((H, K, N)))
    x, w = _vals(xb), _vals(wb)
    y = oracle.head_projection(xb, wb)
    for m in range(M):
        for h in range(H):
            for n in range(N):
                s = 0.0
                for k in range(K):
                    s += x[m, h, k] * w[h, k, n]
                assert abs(y[m, h, n] - s) <= 1e-12 * max(1.0, abs(s))


def test_identity_weights_copy_and_heads_are_independent():
    rng = np.random.default_rng(2)
    M, H, K, N = 4, 3, 8, 16
    xb = _bits(rng.standard_normal((M, H, K)))
    w = np.zeros((H, K, N), np.float32)
    for h in range(H):
        w[h, :, :K] = np.eye(K)
    y = oracle.head_projection(xb, _bits(w))
    np.testing.assert_array_equal(y[:, :, :K], _vals(xb))
    assert not y[:, :, K:].any()
    w2 = w.copy()
    w2[1] = rng.standard_normal((K, N))
    y2 = oracle.head_projection(xb, _bits(w2))
    np.testing.assert_array_equal(y2[:, [0, 2]], y[:, [0, 2]])
