"""Pins of the oracle's two other weight layouts: the compressed-tensors packing
(every output feature's reduction row contiguous, [C, R/8] words, [C, R/32]
scales) and GPTQ quantised in activation order (a group index per reduction
element). Hand-derived goldens, special cases that reduce to the pinned GPTQ
decoder, element-by-element construction from an arithmetic encoder, and planted
mistakes that the goldens must catch."""
import numpy as np
import pytest

import oracle
from oracle import moe_oracle
from int4_weight_only_moe_gb300 import inputs
from tests.conftest import read_golden
from tests.test_oracle_pins import bf16_bits_of, bf16_value, encode_codes


def encode_codes_ct(values: np.ndarray) -> np.ndarray:
    """Pack symmetric INT4 values ``[R, C]`` into compressed-tensors words ``[C, R/8]``.

    Word ``[c, r]`` = sum_i (value[8r+i, c] + 8) * 16**i, with integer arithmetic.
    """
    R, C = values.shape
    words = np.zeros((C, R // 8), dtype=np.int64)
    for i in range(8):
        words += (values[i::8, :].T.astype(np.int64) + 8) * (16 ** i)
    return words.astype(np.uint32).view(np.int32)


def golden_ct():
    rows = read_golden("ct_layout.txt")
    words = np.array([[int(w, 16) for w in r[2:6]] for r in rows], dtype=np.uint32)
    scales = np.array([[bf16_bits_of(float(r[1]))] for r in rows], dtype=np.uint16)
    want = np.array([[float(v) for v in r[6:]] for r in rows])
    return words.view(np.int32), scales, want


def test_ct_golden():
    q, s, want = golden_ct()
    W = oracle.dequantize_ct(q, s)
    assert W.shape == (2, 32)
    np.testing.assert_array_equal(W, want)


def test_ct_scale_is_per_feature_and_group():
    # two features, two groups each, four different scales: feature c, group j -> scale[c, j]
    vals = np.ones((64, 2), dtype=np.int64)
    sc = [[0.5, 4.0], [2.0, 0.25]]
    sbits = np.array([[bf16_bits_of(v) for v in row] for row in sc], dtype=np.uint16)
    W = oracle.dequantize_ct(encode_codes_ct(vals), sbits)
    for c in range(2):
        assert np.all(W[c, :32] == sc[c][0]) and np.all(W[c, 32:] == sc[c][1])


@pytest.mark.parametrize("seed", [0, 1])
def test_ct_equals_gptq_of_the_same_codes(seed):
    # the same codes and scales in the two layouts dequantise to the same matrix,
    # and both to the element-by-element construction
    rng = np.random.default_rng(seed)
    R, C = 96, 40
    vals = rng.integers(-8, 8, size=(R, C))
    sbits = rng.integers(0x3A00, 0x4100, size=(R // 32, C)).astype(np.uint16)
    W_ct = oracle.dequantize_ct(encode_codes_ct(vals), np.ascontiguousarray(sbits.T))
    W_gptq = oracle.dequantize(encode_codes(vals), sbits)
    np.testing.assert_array_equal(W_ct, W_gptq)
    for c in range(0, C, 7):
        for r in range(0, R, 5):
            assert W_ct[c, r] == float(vals[r, c]) * bf16_value(sbits[r // 32, c])
    np.testing.assert_array_equal(oracle.unpack_codes_ct(encode_codes_ct(vals)), vals + 8)


def golden_act_order():
    out = []
    for row in read_golden("act_order_example.txt"):
        arrow = row.index("->")
        out.append((row[0], np.array([int(v) for v in row[1:arrow]]),
                    np.array([float(v) for v in row[arrow + 1:]])))
    return out


def act_order_case():
    q = encode_codes(np.ones((64, 1), dtype=np.int64))
    s = np.array([[bf16_bits_of(0.5)], [bf16_bits_of(4.0)]], dtype=np.uint16)
    return q, s


def test_act_order_golden():
    q, s = act_order_case()
    for name, g_idx, want in golden_act_order():
        W = oracle.dequantize_g_idx(q, s, g_idx)
        np.testing.assert_array_equal(W[0], want, err_msg=name)


def test_act_order_with_natural_groups_is_plain_gptq():
    rng = np.random.default_rng(5)
    R, C = 128, 24
    vals = rng.integers(-8, 8, size=(R, C))
    sbits = rng.integers(0x3A00, 0x4100, size=(R // 32, C)).astype(np.uint16)
    q = encode_codes(vals)
    np.testing.assert_array_equal(oracle.dequantize_g_idx(q, sbits, np.arange(R) // 32),
                                  oracle.dequantize(q, sbits))


def test_act_order_reordering_leaves_the_product_unchanged():
    # Sorting the reduction elements by group (codes moved with them) turns an
    # act-order matrix into a plain one; the product with x reordered the same way
    # is unchanged. This is the identity the library's repack relies on.
    rng = np.random.default_rng(9)
    R, C = 128, 16
    vals = rng.integers(-8, 8, size=(R, C))
    sbits = rng.integers(0x3A00, 0x4100, size=(R // 32, C)).astype(np.uint16)
    g_idx = inputs.act_order_g_idx(0, R, 0)
    assert np.all(np.bincount(g_idx) == 32)
    perm = np.argsort(g_idx, kind="stable")
    W = oracle.dequantize_g_idx(encode_codes(vals), sbits, g_idx)
    W_sorted = oracle.dequantize(encode_codes(vals[perm]), sbits)
    np.testing.assert_array_equal(W[:, perm], W_sorted)
    x = rng.standard_normal((3, R))
    np.testing.assert_allclose(x @ W.T, x[:, perm] @ W_sorted.T, rtol=1e-12, atol=1e-12)


def test_dense_source_forward_matches_packed_forward():
    rng = np.random.default_rng(2)
    E, K, N, M, k = 3, 64, 32, 5, 2
    ws = [inputs.expert_weights(e, K, N) for e in range(E)]
    q1, s1, q2, s2 = (np.stack([w[i] for w in ws]) for i in range(4))
    x = inputs.hidden_states(M, K)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(M)]).astype(np.int32)
    wts = rng.uniform(0.1, 1.0, size=(M, k))
    want = oracle.moe_forward(x, ids, wts, q1, s1, q2, s2)
    got = oracle.moe_forward(x, ids, wts, None, None, None, None,
                             dense_source=lambda e: oracle.expert_dense(q1, s1, q2, s2, e))
    np.testing.assert_array_equal(got, want)


def test_planted_layout_mistakes_are_caught(monkeypatch):
    q, s, want = golden_ct()
    orig = moe_oracle.unpack_codes_ct
    orig_g = moe_oracle.dequantize_g_idx

    def reversed_nibbles(weight_packed):
        u = orig(weight_packed)
        return u.reshape(-1, 8, u.shape[1])[:, ::-1, :].reshape(u.shape)

    def words_of_one_feature_swapped(weight_packed):
        u = orig(weight_packed)
        return u[:, ::-1]

    for fn in (reversed_nibbles, words_of_one_feature_swapped):
        with monkeypatch.context() as m:
            m.setattr(moe_oracle, "unpack_codes_ct", fn)
            assert not np.array_equal(moe_oracle.dequantize_ct(q, s), want), fn.__name__

    qa, sa = act_order_case()

    def ignore_g_idx(qweight, scales, g_idx):
        return moe_oracle.dequantize(qweight, scales)

    def group_of_first_in_run(qweight, scales, g_idx):
        g = np.asarray(g_idx)[np.arange(len(g_idx)) // 32 * 32]
        return orig_g(qweight, scales, g)

    for fn in (ignore_g_idx, group_of_first_in_run):
        with monkeypatch.context() as m:
            m.setattr(moe_oracle, "dequantize_g_idx", fn)
            bad = [not np.array_equal(moe_oracle.dequantize_g_idx(qa, sa, g)[0], w)
                   for _, g, w in golden_act_order()]
            assert any(bad), fn.__name__
