"""Pins of the oracle's router: top-k of E experts per token (NVIDIA AI releases Nemotron 3
Ultra, architecture paragraph: 512 experts, top-22), softmax over the selected logits."""
import itertools

import numpy as np
import pytest

import oracle


def _brute_topk(logits, k):
    """Max-sum subset; among max-sum subsets the lexicographically smallest sorted tuple."""
    best, best_sum = None, None
    for sub in itertools.combinations(range(len(logits)), k):
        s = sum(float(logits[i]) for i in sub)
        if best is None or s > best_sum or (s == best_sum and sub < best):
            best, best_sum = sub, s
    return list(best)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (8, 3), (10, 4), (7, 7)])
def test_topk_matches_brute_force_with_exact_integer_logits(E, k):
    rng = np.random.default_rng(E * 10 + k)
    T, d = 40, 64
    # integer x and W with small magnitudes: every partial sum is an exact fp32 integer,
    # so the logits are exactly the integer dot products and ties are frequent.
    x = rng.integers(-2, 3, (T, d)).astype(np.float32)
    W = rng.integers(-1, 2, (E, d)).astype(np.float32)
    b = rng.integers(-2, 3, E).astype(np.float32)
    logits, idx, w, counts = oracle.router(x, W, b, k)
    exact = x.astype(np.int64) @ W.astype(np.int64).T + b.astype(np.int64)
    assert np.array_equal(logits, exact.astype(np.float32))
    for t in range(T):
        assert list(idx[t]) == _brute_topk(exact[t], k)
    assert counts.sum() == T * k
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))


def test_weights_are_softmax_over_selected_and_sum_to_one():
    rng = np.random.default_rng(1)
    T, d, E, k = 64, 128, 32, 6
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    W = (rng.normal(0, 1, (E, d)) / np.sqrt(d)).astype(np.float32)
    logits, idx, w, _ = oracle.router(x, W, None, k)
    assert np.allclose(w.sum(1), 1.0, atol=1e-6)
    sel = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), 1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-7)
    assert np.all(np.diff(idx, axis=1) > 0)          # slots in ascending expert id


def test_k1_is_one_hot_and_all_equal_logits_pick_lowest_indices():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, (8, 64)).astype(np.float32)
    W = rng.normal(0, 1, (9, 64)).astype(np.float32)
    _, idx, w, _ = oracle.router(x, W, None, 1)
    assert np.all(w == 1.0)
    _, idx, w, _ = oracle.router(np.zeros((3, 64), np.float32), W, None, 4)
    assert np.array_equal(idx, np.tile(np.arange(4), (3, 1)))
    assert np.allclose(w, 0.25)


def test_canonical_two_level_order_worked_example():
    # d = 2048: two groups of 16 chunks.  Chunk 0 gives p0 = 2^24 (group 0); chunks 16 and 17
    # give 1 and -2^24 (group 1).  Group sums: G0 = 2^24, G1 = (0 + 1) + (-2^24) = 1 - 2^24
    # (exact in fp32); logit = (0 + G0) + G1 = 1.  A flat left-to-right sum of the chunk
    # partials would give ((2^24 + 1) -> 2^24) - 2^24 = 0.  Worked by hand from the order.
    d = 2048
    x = np.zeros((1, d), np.float32)
    W = np.zeros((1, d), np.float32)
    x[0, 0], W[0, 0] = 2.0 ** 12, 2.0 ** 12
    x[0, 16 * 64], W[0, 16 * 64] = 1.0, 1.0
    x[0, 17 * 64], W[0, 17 * 64] = -(2.0 ** 12), 2.0 ** 12
    lg, _, _, _ = oracle.router(x, W, None, 1)
    assert lg[0, 0] == 1.0


def test_group_is_sixteen_chunks_worked_example():
    # d = 1024: one group of 16 chunks.  Chunks 0, 8 and 9 give 2^24, 1 and -2^24.  In the
    # group's left-to-right sum 2^24 + 1 rounds back to 2^24 (a tie, to even), then -2^24:
    # the logit is 0.  Groups of 8 chunks would give G0 = 2^24 and G1 = 1 - 2^24 (exact in
    # fp32), logit 1.  Worked by hand from the order.
    d = 1024
    x = np.zeros((1, d), np.float32)
    W = np.zeros((1, d), np.float32)
    x[0, 0], W[0, 0] = 2.0 ** 12, 2.0 ** 12
    x[0, 8 * 64], W[0, 8 * 64] = 1.0, 1.0
    x[0, 9 * 64], W[0, 9 * 64] = -(2.0 ** 12), 2.0 ** 12
    lg, _, _, _ = oracle.router(x, W, None, 1)
    assert lg[0, 0] == 0.0


def test_chunk_chain_is_fused_multiply_add_worked_example():
    # One chunk: p = fma(1, -1, 0) = -1, then fma(x1, w1, p) with x1 = w1 = 1 + 2^-12.  The exact
    # product is 1 + 2^-11 + 2^-24, and a fused multiply-add adds it to -1 with a single
    # rounding: 2^-11 + 2^-24, exact in fp32.  Rounding the product first (2^-24 is half an ulp
    # of 1, and the tie goes to the even neighbour 1 + 2^-11) and then adding would give 2^-11.
    # Worked by hand from the definition of the chunk's fmaf chain.
    x = np.zeros((1, 64), np.float32)
    W = np.zeros((1, 64), np.float32)
    x[0, 0], W[0, 0] = 1.0, -1.0
    x[0, 1] = W[0, 1] = 1.0 + 2.0 ** -12
    lg, _, _, _ = oracle.router(x, W, None, 1)
    assert lg[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)


def test_canonical_chunked_fp32_order_worked_example():
    # d = 192: three chunks of 64.  Chunk sums p0 = 2^24, p1 = 1, p2 = -2^24 (each exact).
    # Canonical order ((0 + p0) + p1) + p2 = (2^24 + 1 -> 2^24 in fp32) - 2^24 = 0, whereas
    # the exact value is 1.  Worked by hand from the definition of the order.
    d = 192
    x = np.zeros((1, d), np.float32)
    W = np.zeros((2, d), np.float32)
    x[0, 0], W[0, 0] = 2.0 ** 12, 2.0 ** 12
    x[0, 64], W[0, 64] = 1.0, 1.0
    x[0, 128], W[0, 128] = -(2.0 ** 12), 2.0 ** 12
    W[1, 5] = 0.5                                 # expert 1: logit 0 (x[5] = 0)
    x2 = np.vstack([x])
    logits, idx, _, _ = oracle.router(x2, W, np.array([0.0, 0.25], np.float32), 1)
    assert logits[0, 0] == 0.0 and logits[0, 1] == 0.25
    assert idx[0, 0] == 1
    # inside one chunk the fma chain is sequential: 2^24 then +1 then -2^24 -> 0 as well
    x3 = np.zeros((1, 64), np.float32)
    W3 = np.zeros((1, 64), np.float32)
    x3[0, :3] = [2.0 ** 12, 1.0, -(2.0 ** 12)]
    W3[0, :3] = [2.0 ** 12, 1.0, 2.0 ** 12]
    lg, _, _, _ = oracle.router(x3, W3, None, 1)
    assert lg[0, 0] == 0.0
