"""Pins for oracle.gemm: brute-force loops, exact small-integer products, shape derivation."""
import numpy as np

from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q

rng = np.random.default_rng(7)


def test_gemm_matches_brute_force_loops():
    M, N, K = 5, 7, 9
    a = rng.standard_normal((M, K))
    b = rng.standard_normal((N, K))
    bias = rng.standard_normal(N)
    d = G.gemm(a, b, alpha=0.5, bias=bias)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for k in range(K):
                s += a[m, k] * b[n, k]
            assert abs(d[m, n] - (0.5 * s + bias[n])) < 1e-12


def test_fp8_small_integer_products_exact():
    # small integers are exact in E4M3; power-of-two scales keep the product exact
    M, N, K = 16, 32, 48
    ai = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    bi = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    qa, _, _, sia = Q.fp8_quantize(ai, np.float32(4.0), "e4m3")
    qb, _, _, sib = Q.fp8_quantize(bi, np.float32(0.5), "e4m3")
    d = G.gemm(Q.fp8_dequant(qa, sia, "e4m3"), Q.fp8_dequant(qb, sib, "e4m3"))
    exact = ai.astype(np.int64) @ bi.astype(np.int64).T
    np.testing.assert_array_equal(d, exact.astype(np.float64))


def test_dgrad_wgrad_orientation():
    # Y = X W^T; dX = dY W; dW = dY^T X, each as D = A B^T over K-major operands
    X = rng.standard_normal((8, 16))
    W = rng.standard_normal((24, 16))
    dY = rng.standard_normal((8, 24))
    np.testing.assert_allclose(G.gemm(X, W), X @ W.T)
    np.testing.assert_allclose(G.gemm(dY, W.T), dY @ W)
    np.testing.assert_allclose(G.gemm(dY.T, X.T), dY.T @ X)


def test_twelve_codonfm_shapes():
    shapes = G.linear_shapes(4096, 16384, 31 * 512)
    assert len(shapes) == 12
    M = 15872
    expect = {
        ("qkv", "fprop"): (M, 12288, 4096), ("qkv", "dgrad"): (M, 4096, 12288), ("qkv", "wgrad"): (12288, 4096, M),
        ("attn_out", "fprop"): (M, 4096, 4096), ("attn_out", "wgrad"): (4096, 4096, M),
        ("mlp_up", "fprop"): (M, 16384, 4096), ("mlp_up", "dgrad"): (M, 4096, 16384),
        ("mlp_down", "fprop"): (M, 4096, 16384), ("mlp_down", "wgrad"): (4096, 16384, M),
    }
    got = {(n, p): (m, nn, k) for n, p, m, nn, k in shapes}
    for key, v in expect.items():
        assert got[key] == v
    flops = sum(2 * m * n * k for _, _, m, n, k in shapes)
    assert abs(flops / 1e12 - 19.17) < 0.01      # one layer ~ 19.17 TFLOP


def test_rel_frobenius_and_bf16_rounding():
    ref = rng.standard_normal((64, 64))
    assert G.rel_frobenius(ref, ref) == 0.0
    bf = F.bf16_bits_to_f32(F.f64_to_bf16_bits(ref))
    e = G.rel_frobenius(bf, ref)
    assert 5e-4 < e < 3e-3                        # bf16 output rounding alone is ~1.7e-3


def test_gemm_accumulate_sums_micro_batches():
    # splitting the contraction (the token dimension of Wgrad) into micro-batches and
    # accumulating gives the full product: sum_j A_j^T B_j over token blocks j
    rng = np.random.default_rng(5)
    dy = rng.standard_normal((96, 12))      # tokens x out
    x = rng.standard_normal((96, 20))       # tokens x in
    full = dy.T @ x                          # out x in
    acc = np.zeros((12, 20))
    for j in range(0, 96, 32):
        acc = G.gemm_accumulate(acc, dy[j:j + 32].T, x[j:j + 32].T)
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-12)
    # zero operands leave D unchanged; identity operands add B
    d0 = rng.standard_normal((4, 4))
    assert np.array_equal(G.gemm_accumulate(d0, np.zeros((4, 3)), np.zeros((4, 3))), d0)
    np.testing.assert_array_equal(G.gemm_accumulate(d0, np.eye(4), np.eye(4)), d0 + np.eye(4))
