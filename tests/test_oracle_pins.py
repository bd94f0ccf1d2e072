"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each check is built so that a plausible slip in the oracle (wrong nibble order,
dropped -8 offset, swapped gate/up, transposed w2, wrong group index, wrong
activation, lost routing weight, unstable or unpadded align) fails at least one
of them; ``test_planted_mistakes_are_caught`` plants those slips and checks.
"""
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle
from tests.conftest import read_golden

# ---------------------------------------------------------------------------
# independent helpers (encode direction, written with arithmetic, not bit ops)


def encode_codes(values: np.ndarray) -> np.ndarray:
    """Pack symmetric INT4 values ``[R, C]`` into ``[R/8, C]`` int32 words.

    Word = sum_i (value[8r+i] + 8) * 16**i, built with integer arithmetic.
    """
    R, C = values.shape
    words = np.zeros((R // 8, C), dtype=np.int64)
    for i in range(8):
        words += (values[i::8, :].astype(np.int64) + 8) * (16 ** i)
    return words.astype(np.uint32).view(np.int32)


def bf16_bits_of(v: float) -> int:
    """bf16 pattern of a float that is exactly representable in bf16."""
    (b,) = struct.unpack(">I", struct.pack(">f", v))
    assert b & 0xFFFF == 0, v
    return b >> 16


def bf16_value(bits: int) -> float:
    (v,) = struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))
    return v


def dense_by_loops(values: np.ndarray, scale_bits: np.ndarray, g: int = 32) -> np.ndarray:
    """Output-major dense matrix from integer values and bf16 scale bits, element by element."""
    R, C = values.shape
    out = np.zeros((C, R))
    for r in range(R):
        for c in range(C):
            out[c, r] = float(values[r, c]) * bf16_value(scale_bits[r // g, c])
    return out


def torch_swiglu(x, w1, w2):
    """Dense SwiGLU MLP with torch's own SiLU and matmul (float64)."""
    x, w1, w2 = (torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)) for a in (x, w1, w2))
    n = w1.shape[0] // 2
    h = torch.nn.functional.silu(x @ w1[:n].T) * (x @ w1[n:].T)
    return (h @ w2.T).numpy()


def random_problem(rng, E, K, N, M, k, dup_experts=False):
    v1 = rng.integers(-8, 8, size=(E, K, 2 * N))
    v2 = rng.integers(-8, 8, size=(E, N, K))
    s1 = rng.integers(0x3B00, 0x3D00, size=(E, K // 32, 2 * N)).astype(np.uint16)  # ~[0.002, 0.03]
    s2 = rng.integers(0x3B00, 0x3D00, size=(E, N // 32, K)).astype(np.uint16)
    if dup_experts:
        v1[:] = v1[0]
        v2[:] = v2[0]
        s1[:] = s1[0]
        s2[:] = s2[0]
    w1_q = np.stack([encode_codes(v1[e]) for e in range(E)])
    w2_q = np.stack([encode_codes(v2[e]) for e in range(E)])
    x = rng.standard_normal((M, K)).astype(np.float32)
    x_bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 is a valid input
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(M)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(M, k)).astype(np.float32)
    return dict(v1=v1, v2=v2, s1=s1, s2=s2, w1_q=w1_q, w2_q=w2_q, x_bits=x_bits,
                ids=ids, w=w)


def x_f64(bits):
    return np.array([[bf16_value(b) for b in row] for row in bits])


# ---------------------------------------------------------------------------
# dequantisation


def test_nibble_order_golden():
    rows = read_golden("nibble_order.txt")
    C = len(rows)
    q = np.full((4, C), 0x88888888, dtype=np.uint32)  # 32 reduction elements per column
    for c, row in enumerate(rows):
        q[0, c] = int(row[0], 16)
    ones = np.full((1, C), bf16_bits_of(1.0), dtype=np.uint16)
    W = oracle.dequantize(q.view(np.int32), ones)
    assert W.shape == (C, 32)
    for c, row in enumerate(rows):
        expect = [float(v) for v in row[1:9]]
        assert W[c, :8].tolist() == expect, row[0]
        assert np.all(W[c, 8:] == 0.0)


def test_dequant_matches_elementwise_construction():
    rng = np.random.default_rng(123)
    R, C = 64, 24
    vals = rng.integers(-8, 8, size=(R, C))
    sbits = rng.integers(0x3A00, 0x4100, size=(R // 32, C)).astype(np.uint16)
    W = oracle.dequantize(encode_codes(vals), sbits)
    np.testing.assert_array_equal(W, dense_by_loops(vals, sbits))


def test_scale_group_runs_along_reduction_axis():
    # one column, two groups with different scales: elements 0..31 use scale 0, 32..63 scale 1
    vals = np.ones((64, 1), dtype=np.int64)
    sbits = np.array([[bf16_bits_of(0.5)], [bf16_bits_of(4.0)]], dtype=np.uint16)
    W = oracle.dequantize(encode_codes(vals), sbits)
    assert np.all(W[0, :32] == 0.5) and np.all(W[0, 32:] == 4.0)


# ---------------------------------------------------------------------------
# expert MLP and mixture


def closed_form_problem():
    E, K, N, M, k = 2, 64, 32, 2, 2
    v1 = np.zeros((E, K, 2 * N), dtype=np.int64)
    v2 = np.zeros((E, N, K), dtype=np.int64)
    s1 = np.full((E, K // 32, 2 * N), bf16_bits_of(1.0), dtype=np.uint16)
    s2 = np.full((E, N // 32, K), bf16_bits_of(1.0), dtype=np.uint16)
    v1[1, 37, 5] = 4
    s1[1, 1, 5] = bf16_bits_of(0.5)
    v1[1, 37, N + 5] = -2
    s1[1, 1, N + 5] = bf16_bits_of(0.25)
    v2[1, 5, 10] = 7
    s2[1, 0, 10] = bf16_bits_of(0.125)
    w1_q = np.stack([encode_codes(v1[e]) for e in range(E)])
    w2_q = np.stack([encode_codes(v2[e]) for e in range(E)])
    x = np.zeros((M, K), dtype=np.uint16)
    x[0, 37] = bf16_bits_of(1.5)
    x[0, 3] = bf16_bits_of(2.0)
    x[1, 37] = bf16_bits_of(-1.0)
    ids = np.array([[1, 0], [0, 1]], dtype=np.int32)
    w = np.array([[0.75, 0.25], [0.5, 0.5]], dtype=np.float32)
    return x, ids, w, w1_q, s1, w2_q, s2


def closed_form_mismatch(forward=None):
    """Largest deviation of the oracle from the hand-derived closed form."""
    forward = forward or oracle.moe_forward
    out = forward(*closed_form_problem())
    expect = np.zeros_like(out)
    for t, col, val in read_golden("closed_form_swiglu.txt"):
        expect[int(t), int(col)] = float(val)
    return float(np.max(np.abs(out - expect)))


def test_closed_form_golden():
    assert closed_form_mismatch() < 1e-14


def test_single_expert_k1_is_dense_swiglu():
    rng = np.random.default_rng(7)
    E, K, N, M = 3, 64, 32, 5
    p = random_problem(rng, E, K, N, M, 1)
    p["w"][:] = 1.0
    out = oracle.moe_forward(p["x_bits"], p["ids"], p["w"], p["w1_q"], p["s1"], p["w2_q"], p["s2"])
    x = x_f64(p["x_bits"])
    for t in range(M):
        e = int(p["ids"][t, 0])
        w1 = dense_by_loops(p["v1"][e], p["s1"][e])
        w2 = dense_by_loops(p["v2"][e], p["s2"][e])
        ref = torch_swiglu(x[t:t + 1], w1, w2)[0]
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-12)


def test_identical_experts_reduce_to_one_dense_mlp():
    rng = np.random.default_rng(8)
    E, K, N, M, k = 6, 64, 32, 4, 3
    p = random_problem(rng, E, K, N, M, k, dup_experts=True)
    p["w"] /= p["w"].sum(axis=1, keepdims=True)
    out = oracle.moe_forward(p["x_bits"], p["ids"], p["w"], p["w1_q"], p["s1"], p["w2_q"], p["s2"])
    w1 = dense_by_loops(p["v1"][0], p["s1"][0])
    w2 = dense_by_loops(p["v2"][0], p["s2"][0])
    ref = torch_swiglu(x_f64(p["x_bits"]), w1, w2)
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-9)  # weights were renormalised in fp32


def test_mixture_invariants():
    rng = np.random.default_rng(9)
    E, K, N, M, k = 5, 64, 32, 6, 3
    p = random_problem(rng, E, K, N, M, k)
    args = (p["w1_q"], p["s1"], p["w2_q"], p["s2"])
    base = oracle.moe_forward(p["x_bits"], p["ids"], p["w"], *args)
    # linear in the routing weights
    scaled = oracle.moe_forward(p["x_bits"], p["ids"], p["w"] * 2.0, *args)
    np.testing.assert_allclose(scaled, 2.0 * base, rtol=1e-13, atol=1e-12)
    # the order of a token's k slots does not matter
    perm = rng.permutation(k)
    sl = oracle.moe_forward(p["x_bits"], p["ids"][:, perm], p["w"][:, perm], *args)
    np.testing.assert_allclose(sl, base, rtol=1e-12, atol=1e-12)
    # permuting tokens permutes output rows
    tp = rng.permutation(M)
    tk = oracle.moe_forward(p["x_bits"][tp], p["ids"][tp], p["w"][tp], *args)
    np.testing.assert_allclose(tk, base[tp], rtol=1e-12, atol=1e-12)
    # sampled rows equal the full computation
    sub = oracle.moe_forward(p["x_bits"], p["ids"], p["w"], *args, tokens=[4, 1])
    np.testing.assert_allclose(sub, base[[4, 1]], rtol=1e-12, atol=1e-15)  # BLAS blocking may differ
    # a zero routing weight removes that expert's contribution exactly
    w0 = p["w"].copy()
    w0[:, 1:] = 0.0
    one = oracle.moe_forward(p["x_bits"], p["ids"], w0, *args)
    x = x_f64(p["x_bits"])
    for t in range(M):
        e = int(p["ids"][t, 0])
        ref = w0[t, 0] * torch_swiglu(x[t:t + 1], dense_by_loops(p["v1"][e], p["s1"][e]),
                                      dense_by_loops(p["v2"][e], p["s2"][e]))[0]
        np.testing.assert_allclose(one[t], ref, rtol=1e-12, atol=1e-12)


def test_silu_special_values():
    z = np.array([0.0, 1e-300, 50.0, -50.0, -800.0])
    y = oracle.silu(z)
    assert y[0] == 0.0
    assert abs(y[2] - 50.0) < 1e-15 * 50
    assert abs(y[3]) < 1e-19
    assert y[4] == 0.0 or abs(y[4]) < 1e-300
    torch_ref = torch.nn.functional.silu(torch.tensor([-3.0, -0.5, 0.25, 2.0, 7.5], dtype=torch.float64))
    np.testing.assert_allclose(oracle.silu(np.array([-3.0, -0.5, 0.25, 2.0, 7.5])), torch_ref.numpy(),
                               rtol=1e-15)


# ---------------------------------------------------------------------------
# align


def align_brute_force(ids, E, block):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    sentinel = len(flat)
    out, offsets = [], [0]
    for e in range(E):
        mine = [i for i, v in enumerate(flat) if v == e]
        while len(mine) % block:
            mine.append(sentinel)
        out.extend(mine)
        offsets.append(len(out))
    return out, offsets


@pytest.mark.parametrize("block", [1, 3, 4, 16, 64])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_align_matches_brute_force(block, seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 20))
    M = int(rng.integers(0, 30))
    k = int(rng.integers(1, min(E, 5) + 1))
    ids = rng.integers(0, E, size=(M, k)).astype(np.int32)  # duplicates allowed: still well defined
    sorted_ids, offsets, num_padded = oracle.moe_align(ids, E, block)
    bf_ids, bf_off = align_brute_force(ids, E, block)
    assert sorted_ids.tolist() == bf_ids
    assert offsets.tolist() == bf_off
    assert num_padded == len(bf_ids)


def test_align_invariants_and_skew():
    rng = np.random.default_rng(5)
    E, M, k, block = 12, 200, 4, 16
    p = np.arange(1, E + 1, dtype=float) ** -1.1
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(M)]).astype(np.int32)
    ids[3, 1] = -1   # out-of-range slots are left out
    ids[7, 0] = E
    s, off, n = oracle.moe_align(ids, E, block)
    flat = ids.reshape(-1)
    real = s[s < M * k]
    valid = np.nonzero((flat >= 0) & (flat < E))[0]
    assert sorted(real.tolist()) == valid.tolist()          # every valid slot exactly once
    assert np.all(np.diff(off) % block == 0)
    for e in range(E):
        seg = s[off[e]:off[e + 1]]
        body = seg[seg < M * k]
        assert np.all(flat[body] == e)
        assert np.all(np.diff(body) > 0)                    # ascending inside an expert
        assert len(seg) == -(-np.count_nonzero(flat == e) // block) * block
    assert n == off[-1]


def test_align_empty():
    s, off, n = oracle.moe_align(np.zeros((0, 8), np.int32), 16, 16)
    assert n == 0 and s.size == 0 and off.tolist() == [0] * 17


# ---------------------------------------------------------------------------
# sizes printed on the pages


def test_packed_bytes_match_page_figures():
    kv = {r[0]: float(r[1]) for r in read_golden("page_sizes.txt")}
    E, K, N, nb = int(kv["E"]), int(kv["K"]), int(kv["N"]), int(kv["num_bits"])
    marlin_w1 = (K // 16) * (2 * N * (nb // 2)) * 4
    marlin_w2 = (N // 16) * (K * (nb // 2)) * 4
    scale_bytes = (2 * N * (K // 32) + K * (N // 32)) * 2
    per_expert = oracle.roofline_bytes_per_expert(K, N)
    assert per_expert - scale_bytes == marlin_w1 + marlin_w2 == 22_020_096
    total = E * (marlin_w1 + marlin_w2)
    assert abs(total - kv["approx_total_weight_bytes"]) / kv["approx_total_weight_bytes"] < 0.01


# ---------------------------------------------------------------------------
# planted mistakes (in the oracle, on the CPU) must trip the pins


def _mutants():
    orig_unpack = moe_oracle.unpack_codes
    orig_ffn = moe_oracle.expert_ffn
    orig_deq = moe_oracle.dequantize

    def unpack_reversed(q):
        u = orig_unpack(q)
        r8 = u.shape[0] // 8
        return u.reshape(r8, 8, -1)[:, ::-1, :].reshape(u.shape)

    def deq_no_offset(q, s, g=32):
        return orig_deq(q, s, g) + 8.0 * np.repeat(moe_oracle.bf16_to_f64(s), g, axis=0).T

    def deq_wrong_group(q, s, g=32):
        s2 = s[::-1].copy() if s.shape[0] > 1 else s
        return orig_deq(q, s2, g)

    def ffn_swapped(x, w1, w2):
        n = w1.shape[0] // 2
        return orig_ffn(x, np.concatenate([w1[n:], w1[:n]]), w2)

    def ffn_sigmoid(x, w1, w2):
        n = w1.shape[0] // 2
        g, u = x @ w1[:n].T, x @ w1[n:].T
        return ((1 / (1 + np.exp(-g))) * u) @ w2.T

    def ffn_transposed_down(x, w1, w2):
        n = w1.shape[0] // 2
        h = moe_oracle.silu(x @ w1[:n].T) * (x @ w1[n:].T)
        w2t = np.zeros_like(w2)
        m = min(w2.shape)
        w2t[:m, :m] = w2[:m, :m].T
        return h @ w2t.T

    return {
        "unpack_codes": [unpack_reversed],
        "dequantize": [deq_no_offset, deq_wrong_group],
        "expert_ffn": [ffn_swapped, ffn_sigmoid, ffn_transposed_down],
    }


def test_planted_mistakes_are_caught(monkeypatch):
    for name, variants in _mutants().items():
        for fn in variants:
            with monkeypatch.context() as m:
                m.setattr(moe_oracle, name, fn)
                assert closed_form_mismatch(moe_oracle.moe_forward) > 1e-3, (name, fn.__name__)


def test_planted_align_mistakes_are_caught():
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 6, size=(20, 3)).astype(np.int32)
    good, off, _ = oracle.moe_align(ids, 6, 4)
    bf, bf_off = align_brute_force(ids, 6, 4)
    assert good.tolist() == bf
    # unstable order inside an expert, or missing padding, must differ from brute force
    bad = good.copy()
    seg = bad[off[2]:off[3]]
    real = seg[seg < 60]
    if len(real) > 1:
        seg[:len(real)] = real[::-1]
        assert bad.tolist() != bf
    unpadded = [v for v in good.tolist() if v < 60]
    assert unpadded != bf or all(np.diff(bf_off) % 4 == 0)


# ---------------------------------------------------------------------------
# routing (softmax -> top-k -> renormalise)


def test_route_golden():
    from fractions import Fraction
    for k, logits, want_ids, want_w in read_golden_rows("route_examples.txt"):
        lg = np.array([[float(v) for v in logits.split(",")]], dtype=np.float64)
        ids, w = oracle.route(lg, int(k))
        assert ids[0].tolist() == [int(v) for v in want_ids.split(",")], (logits, ids)
        np.testing.assert_allclose(w[0], [float(Fraction(v)) for v in want_w.split(",")], rtol=1e-12)


def read_golden_rows(name):
    rows = []
    for fields in read_golden(name):
        rows.append([f.strip() for f in " ".join(fields).split("|")])
    return rows


def _beats(l, a, b):
    return l[a] > l[b] or (l[a] == l[b] and a < b)


@pytest.mark.parametrize("seed", range(6))
def test_route_matches_subset_enumeration(seed):
    """Brute force: the top-k set is the one k-subset whose every member beats every
    non-member; the order inside it is by how many members each beats; weights are
    probabilities exp(l)/sum exp(l) (plain math.exp) renormalised over the set."""
    import itertools
    import math
    rng = np.random.default_rng(seed)
    E, k = int(rng.integers(3, 8)), int(rng.integers(1, 4))
    k = min(k, E)
    lg = np.round(rng.standard_normal((5, E)) * 2) / 2  # coarse grid: ties happen
    ids, w = oracle.route(lg, k)
    for t in range(lg.shape[0]):
        l = [float(v) for v in lg[t]]
        winners = [S for S in itertools.combinations(range(E), k)
                   if all(_beats(l, a, b) for a in S for b in range(E) if b not in S)]
        assert len(winners) == 1
        S = winners[0]
        order = sorted(S, key=lambda a: -sum(_beats(l, a, b) for b in S))
        assert ids[t].tolist() == order
        z = sum(math.exp(v) for v in l)
        p = [math.exp(l[a]) / z for a in order]
        np.testing.assert_allclose(w[t], [v / sum(p) for v in p], rtol=1e-12)


def test_route_full_softmax_and_shift_invariance():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((7, 12))
    ids, w = oracle.route(lg, 12)  # k = E: the whole softmax, in descending order
    ref = torch.softmax(torch.from_numpy(lg), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids.astype(np.int64), axis=1), rtol=1e-12)
    ids2, w2 = oracle.route(lg + 17.25, 4)
    ids3, w3 = oracle.route(lg, 4)
    assert (ids2 == ids3).all()
    np.testing.assert_allclose(w2, w3, rtol=1e-12)
    np.testing.assert_allclose(w3.sum(axis=1), 1.0, rtol=1e-12)


def test_planted_route_mistakes_are_caught(monkeypatch):
    """A router that forgets to renormalise, or breaks ties towards the higher id,
    fails the golden rows."""
    real = oracle.route

    def no_renorm(logits, topk):
        lg = np.asarray(logits, dtype=np.float64)
        ids, _ = real(lg, topk)
        p = np.exp(lg - lg.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(p, ids.astype(np.int64), axis=1)

    def high_id_ties(logits, topk):
        lg = np.asarray(logits, dtype=np.float64)
        flipped_ids, w = real(lg[:, ::-1], topk)
        return (lg.shape[1] - 1 - flipped_ids).astype(np.int32), w

    for bad in (no_renorm, high_id_ties):
        monkeypatch.setattr(oracle, "route", bad)
        with pytest.raises(AssertionError):
            test_route_golden()
    monkeypatch.setattr(oracle, "route", real)
