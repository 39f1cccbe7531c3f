"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks an oracle function against something fixed independently of
it: a hand-derived example, a closed form, a library routine that computes the
same mathematical object by another route (numpy's full convolution), brute
force enumeration, or an invariant of the recurrence. Shapes use dk != dv and
several heads so that a transposed state, a wrong head map, a dropped term or
a sign error fails at least one of them.
"""
import itertools

import numpy as np
import pytest

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth


def bits(x):
    """Exact BF16 bit patterns of values that BF16 represents exactly."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in BF16"
    return (u >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# BF16 storage
# ----------------------------------------------------------------------------

def test_bf16_round_trip_all_finite_patterns():
    p = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = O.from_bf16(p)
    fin = np.isfinite(v)
    assert np.array_equal(O.to_bf16(v[fin]), p[fin])


def test_bf16_rounding_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7            # BF16 spacing at 1.0
    assert O.to_bf16([one])[0] == 0x3F80
    assert O.to_bf16([one + ulp / 2])[0] == 0x3F80          # tie -> even (down)
    assert O.to_bf16([one + 3 * ulp / 2])[0] == 0x3F82      # tie -> even (up)
    assert O.to_bf16([one + ulp / 2 + 2.0 ** -20])[0] == 0x3F81
    assert O.to_bf16([-2.0])[0] == 0xC000
    assert np.isnan(O.from_bf16(O.to_bf16([np.nan])))[0]


# ----------------------------------------------------------------------------
# a1: descriptors
# ----------------------------------------------------------------------------

def test_chunks_tiny_by_hand():
    # cu_seqlens [0, 5, 18]: sequence 0 has 5 tokens (one chunk), sequence 1
    # has 13 tokens starting at 5 (chunks of 8 and 5 tokens).
    got = O.build_conv_chunks([0, 5, 18])
    assert got.tolist() == [[0, 0, 5, 0], [1, 5, 8, 0], [1, 13, 5, 8]]


def _chunks_by_token_walk(cu, chunk):
    """Brute force: walk every token; a token whose position in its sequence is
    a multiple of ``chunk`` opens a new record, the others extend it."""
    recs = []
    for s in range(len(cu) - 1):
        for t in range(cu[s], cu[s + 1]):
            pos = t - cu[s]
            if pos % chunk == 0:
                recs.append([s, t, 1, pos])
            else:
                recs[-1][2] += 1
    return recs


@pytest.mark.parametrize("chunk", [1, 3, 8])
def test_chunks_brute_force(chunk):
    for n in range(0, 4):
        for lengths in itertools.product(range(0, 21, 3 if n == 3 else 1), repeat=n):
            cu = np.concatenate([[0], np.cumsum(lengths)]).astype(int).tolist()
            got = O.build_conv_chunks(cu, chunk).tolist()
            assert got == _chunks_by_token_walk(cu, chunk), (cu, chunk)
            assert len(got) == sum(-(-L // chunk) for L in lengths)


def test_chunks_whole_sequence_mode():
    cu = [0, 7, 7, 30, 31]
    got = O.build_conv_chunks(cu, 1 << 20).tolist()
    assert got == [[0, 0, 7, 0], [2, 7, 23, 0], [3, 30, 1, 0]]


# ----------------------------------------------------------------------------
# a2 / a3: conv
# ----------------------------------------------------------------------------

def test_conv_by_hand():
    # One channel, taps w = (1, 1/2, 1/4, 2) on (x[t-3], x[t-2], x[t-1], x[t]),
    # initial state (5, 6, 7), x = (1, 2, 3, 4), no bias, no SiLU:
    #   y0 = 5 + 3 + 1.75 + 2 = 11.75     y1 = 6 + 3.5 + .25 + 4 = 13.75
    #   y2 = 7 + .5 + .5 + 6 = 14         y3 = 1 + 1 + .75 + 8 = 10.75
    # new state = last three of (5, 6, 7, 1, 2, 3, 4) = (2, 3, 4).
    y, st = O.causal_conv1d_fwd(bits([[1], [2], [3], [4]]), bits([[1, .5, .25, 2]]), None,
                                bits([[[5, 6, 7]]]), [1], [0, 4], apply_silu=False)
    assert y[:, 0].tolist() == [11.75, 13.75, 14.0, 10.75]
    assert st[0, 0].tolist() == [2.0, 3.0, 4.0]


def test_silu_closed_forms():
    x = np.linspace(-30, 30, 1001)
    assert O.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.silu(np.array([40.0])), [40.0], rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([1.0])), [1.0 / (1.0 + np.exp(-1.0))], rtol=1e-15)


def _conv_by_np_convolve(x, w, bias, state, has, cu):
    """Full convolution of (state ++ x) per sequence and channel, by numpy."""
    T, C = x.shape
    K = w.shape[1]
    y = np.zeros((T, C))
    new_state = state.copy()
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        if a == e:
            continue
        for c in range(C):
            init = state[s, c] if has[s] else np.zeros(K - 1)
            seq = np.concatenate([init, x[a:e, c]])
            full = np.convolve(seq, w[c, ::-1])      # full[n] = sum_j w[c,j] seq[n-(K-1)+j]
            y[a:e, c] = full[K - 1:K - 1 + (e - a)] + bias[c]
            new_state[s, c] = seq[-(K - 1):]
    return y, new_state


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_conv_vs_numpy_convolution(seed):
    lengths = [1, 2, 0, 3, 11, 17]
    case = synth.conv_case(seed, lengths, 6, bias=True)
    case["has_initial_state"] = np.array([1, 0, 1, 1, 0, 1], np.uint8)
    x, w, b, st = (O.from_bf16(case[k]) for k in ("x", "w", "bias", "conv_state"))
    ref_pre, ref_state = _conv_by_np_convolve(x, w, b, st, case["has_initial_state"], case["cu_seqlens"])
    y, new_state = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], case["conv_state"],
                                       case["has_initial_state"], case["cu_seqlens"], apply_silu=False)
    np.testing.assert_allclose(y, ref_pre, rtol=0, atol=1e-12)
    assert np.array_equal(new_state, ref_state)
    ys, _ = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], case["conv_state"],
                                case["has_initial_state"], case["cu_seqlens"])
    np.testing.assert_allclose(ys, ref_pre / (1 + np.exp(-ref_pre)), rtol=1e-13, atol=1e-13)


def test_conv_last_tap_is_silu_of_x_and_other_taps_shift():
    case = synth.conv_case(5, [2, 9], 4)
    x, st = O.from_bf16(case["x"]), O.from_bf16(case["conv_state"])
    cu = case["cu_seqlens"]
    for j in range(4):
        w = np.zeros((4, 4), np.float32)
        w[:, j] = 1.0
        y, _ = O.causal_conv1d_fwd(case["x"], bits(w), None, case["conv_state"], [1, 1], cu,
                                   apply_silu=False)
        shift = 3 - j          # tap j reads x[t - shift]
        for s in range(2):
            for i in range(cu[s + 1] - cu[s]):
                m = i - shift
                want = x[cu[s] + m] if m >= 0 else st[s, :, 3 + m]
                assert np.array_equal(y[cu[s] + i], want)
        if j == 3:
            ys, _ = O.causal_conv1d_fwd(case["x"], bits(w), None, case["conv_state"], [1, 1], cu)
            np.testing.assert_allclose(ys, x / (1 + np.exp(-x)), rtol=1e-14)


def test_conv_no_initial_state_equals_zero_state():
    case = synth.conv_case(7, [1, 5, 12], 8, bias=True)
    zeros = np.zeros_like(case["conv_state"])
    y0, s0 = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], case["conv_state"],
                                 [0, 0, 0], case["cu_seqlens"])
    y1, s1 = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], zeros,
                                 [1, 1, 1], case["cu_seqlens"])
    assert np.array_equal(y0, y1) and np.array_equal(s0, s1)


def test_conv_empty_sequence_keeps_state():
    case = synth.conv_case(8, [3, 0, 4], 8)
    _, st = O.causal_conv1d_fwd(case["x"], case["w"], None, case["conv_state"], [1, 1, 1],
                                case["cu_seqlens"])
    assert np.array_equal(st[1], O.from_bf16(case["conv_state"][1]))


def test_conv_split_prefill_equals_whole():
    # Prefill 13 tokens at once == prefill 5 then 8 (state handed over),
    # and == prefill 10 then three single-token updates.
    case = synth.conv_case(9, [13], 16, bias=True)
    x, w, b, st = case["x"], case["w"], case["bias"], case["conv_state"]
    y, s = O.causal_conv1d_fwd(x, w, b, st, [1], [0, 13])
    ya, sa = O.causal_conv1d_fwd(x[:5], w, b, st, [1], [0, 5])
    yb, sb = O.causal_conv1d_fwd(x[5:], w, b, O.to_bf16(sa), [1], [0, 8])
    assert np.array_equal(np.concatenate([ya, yb]), y) and np.array_equal(sb, s)
    yp, sp = O.causal_conv1d_fwd(x[:10], w, b, st, [1], [0, 10])
    ys = [yp]
    for t in range(10, 13):
        yu, sp = O.causal_conv1d_update(x[t:t + 1], w, b, O.to_bf16(sp))
        ys.append(yu)
    assert np.array_equal(np.concatenate(ys), y) and np.array_equal(sp, s)


def test_conv_short_sequence_shifts_old_state():
    # A 2-token sequence: new state = (old[2], x0, x1).
    case = synth.conv_case(10, [2], 3)
    _, st = O.causal_conv1d_fwd(case["x"], case["w"], None, case["conv_state"], [1], [0, 2])
    old, x = O.from_bf16(case["conv_state"][0]), O.from_bf16(case["x"])
    assert np.array_equal(st[0], np.stack([old[:, 2], x[0], x[1]], axis=1))


# ----------------------------------------------------------------------------
# a4: L2 norm
# ----------------------------------------------------------------------------

def test_l2norm():
    x = np.array([[3.0, 4.0], [0.0, 0.0], [1e3, 0.0]])
    y = O.l2norm(x)
    np.testing.assert_allclose(y[0], [3 / np.sqrt(25 + 1e-6), 4 / np.sqrt(25 + 1e-6)], rtol=1e-15)
    assert np.array_equal(y[1], [0.0, 0.0])
    np.testing.assert_allclose(np.linalg.norm(y[2]), 1.0, rtol=1e-12)


# ----------------------------------------------------------------------------
# a4: gate activation from raw logits
# ----------------------------------------------------------------------------

def test_gate_activation_by_hand():
    # a = 1 / (1 + e^{z_a}), b = 1 / (1 + e^{-z_b}); z = ln 3 gives a = 1/4, b = 3/4.
    za = np.array([0.0, np.log(3.0), -np.log(3.0)])
    zb = np.array([0.0, np.log(3.0), -np.log(3.0)])
    a, b = O.gate_activation(za, zb)
    np.testing.assert_allclose(a, [0.5, 0.25, 0.75], rtol=1e-15)
    np.testing.assert_allclose(b, [0.5, 0.75, 0.25], rtol=1e-15)


def test_gate_activation_complementary_and_saturating():
    # exp(-softplus(z)) = 1 - sigmoid(z): a(z) + b(z) = 1 for the same z.
    z = np.linspace(-30.0, 30.0, 121)
    a, b = O.gate_activation(z, z)
    np.testing.assert_allclose(a + b, 1.0, rtol=0, atol=1e-15)
    assert np.all(np.diff(a) < 0) and np.all(np.diff(b) > 0)
    # no overflow at large |z|: the limits 0 and 1
    a, b = O.gate_activation([1000.0, -1000.0], [1000.0, -1000.0])
    assert a.tolist() == [0.0, 1.0] and b.tolist() == [1.0, 0.0]


# ----------------------------------------------------------------------------
# The parity metrics
# ----------------------------------------------------------------------------

def test_rel_err_by_hand():
    assert O.rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
    # the denominator is max|ref| (2), not max|x| (4)
    assert O.rel_err([1.0, 4.0], [1.0, 2.0]) == 1.0
    # absolute values in both maxima: a signed max would give 1 / 1 here
    assert O.rel_err([-4.0, 2.0], [-4.0, 1.0]) == 0.25
    # |x - ref|: a signed difference max would give 0 here
    assert O.rel_err([1.0, -1.0], [1.0, 1.0]) == 2.0
    # an all-zero reference: the absolute error
    assert O.rel_err([0.0, 3e-3], [0.0, 0.0]) == 3e-3
    assert O.rel_err([0.0, 0.0], [0.0, 0.0]) == 0.0
    # a zero candidate against a non-zero reference: 1
    assert O.rel_err([0.0, 0.0], [0.5, -2.0]) == 1.0
    assert O.rel_err(np.zeros((0, 3)), np.zeros((0, 3))) == 0.0


def test_rel_err_slices_by_hand():
    ref = np.array([[[100.0, 0.0]], [[1.0, -1.0]]])     # two slices of shape [1, 2]
    x = np.array([[[100.0, 0.5]], [[1.0, -1.5]]])
    # whole tensor: 0.5 / 100; per slice: 0.5 / 100 and 0.5 / 1
    assert O.rel_err(x, ref) == 0.005
    assert O.rel_err_slices(x, ref, 2) == 0.5
    assert O.rel_err_slices(x, ref, 1) == 0.5
    # the floor: slice scale at least floor * max|ref| of the tensor
    assert O.rel_err_slices(x, ref, 2, floor=0.1) == 0.05
    # an all-zero slice without a floor: its absolute error
    ref0 = np.array([[0.0, 0.0], [2.0, 2.0]])
    x0 = np.array([[0.25, 0.0], [2.0, 2.0]])
    assert O.rel_err_slices(x0, ref0, 1) == 0.25
    assert O.rel_err_slices(x0, ref0, 1, floor=0.5) == 0.25
    # one slice equals rel_err
    rng = np.random.default_rng(3)
    r = rng.standard_normal((4, 5))
    c = r + 1e-3 * rng.standard_normal((4, 5))
    assert O.rel_err_slices(c, r, 2) == O.rel_err(c, r)


# ----------------------------------------------------------------------------
# a5 / prefill: the delta rule
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("literal", [True, False])
def test_delta_by_hand(literal):
    # dk = dv = 2, S0 = [[1, 2], [3, 4]].
    # Token 1: k = (1, 0), v = (5, 6), a = b = 1/2, q = (0, 1):
    #   S0 (I - b k k^T) = [[0.5, 2], [1.5, 4]]; times a -> [[.25, 1], [.75, 2]];
    #   + b v k^T = [[2.5, 0], [3, 0]] -> S1 = [[2.75, 1], [3.75, 2]]; o1 = (1, 2).
    # Token 2: k = (1/2, 1/2), v = (1, -1), a = b = 1, q = (1, 0):
    #   I - k k^T = [[.75, -.25], [-.25, .75]];
    #   S1 (I - k k^T) = [[1.8125, .0625], [2.3125, .5625]];
    #   + v k^T = [[.5, .5], [-.5, -.5]] -> S2 = [[2.3125, .5625], [1.8125, .0625]];
    #   o2 = (2.3125, 1.8125).
    q = bits([[[0, 1]], [[1, 0]]])
    k = bits([[[1, 0]], [[.5, .5]]])
    v = bits([[[5, 6]], [[1, -1]]])
    a = np.array([[.5], [1.0]], np.float32)
    b = np.array([[.5], [1.0]], np.float32)
    S0 = np.array([[[[1, 2], [3, 4]]]], np.float32)
    o, S = O.delta_rule_prefill(q, k, v, a, b, [0, 2], S0, [1], literal=literal)
    assert o[:, 0].tolist() == [[1.0, 2.0], [2.3125, 1.8125]]
    assert S[0, 0].tolist() == [[2.3125, 0.5625], [1.8125, 0.0625]]


def test_delta_literal_and_expanded_agree():
    c = synth.delta_case(11, [7, 9], 2, 4, 5, 3, s0_std=0.5, normed_qk=False)
    args = (c["q"], c["k"], c["v"], c["a"], c["b"], c["cu_seqlens"], c["S0"], c["has_initial_state"])
    o1, S1 = O.delta_rule_prefill(*args, literal=True)
    o2, S2 = O.delta_rule_prefill(*args, literal=False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("literal", [True, False])
def test_delta_no_write_is_pure_decay(literal):
    # b = 0: S_t = (prod_{s<=t} a_s) S0 and o_t = S_t q_t.
    c = synth.delta_case(12, [6], 1, 2, 5, 3, s0_std=1.0)
    b = np.zeros_like(c["b"])
    o, S = O.delta_rule_prefill(c["q"], c["k"], c["v"], c["a"], b, c["cu_seqlens"], c["S0"], [1],
                                literal=literal)
    decay = np.cumprod(c["a"].astype(np.float64), axis=0)      # [T, Hv]
    S0 = c["S0"][0].astype(np.float64)
    np.testing.assert_allclose(S[0], decay[-1][:, None, None] * S0, rtol=1e-13)
    q = O.from_bf16(c["q"])[:, 0]
    want_o = decay[:, :, None] * np.einsum("hij,tj->thi", S0, q)
    np.testing.assert_allclose(o, want_o, rtol=1e-12, atol=1e-14)
    o1, S1 = O.delta_rule_prefill(c["q"], c["k"], c["v"], np.ones_like(c["a"]), b,
                                  c["cu_seqlens"], c["S0"], [1], literal=literal)
    assert np.array_equal(S1[0], S0)


@pytest.mark.parametrize("literal", [True, False])
def test_delta_write_invariant(literal):
    # For every token: S_t k_t = a (1 - b |k|^2) S_{t-1} k_t + b |k|^2 v_t;
    # with b = 1 and |k| = 1 the write is exact: S_t k_t = v_t.
    c = synth.delta_case(13, [5], 1, 1, 6, 4, s0_std=1.0, normed_qk=False)
    q, k, v = O.from_bf16(c["q"])[:, 0], O.from_bf16(c["k"])[:, 0], O.from_bf16(c["v"])[:, 0]
    a, b = c["a"][:, 0].astype(np.float64), c["b"][:, 0].astype(np.float64)
    S = c["S0"][0, 0].astype(np.float64)
    for t in range(5):
        _, Snew = O.delta_rule_prefill(c["q"][t:t + 1], c["k"][t:t + 1], c["v"][t:t + 1],
                                       c["a"][t:t + 1], c["b"][t:t + 1], [0, 1],
                                       S[None, None].astype(np.float64), [1], literal=literal)
        Snew = Snew[0, 0]
        kk = k[t] @ k[t]
        want = a[t] * (1 - b[t] * kk) * (S @ k[t]) + b[t] * kk * v[t]
        np.testing.assert_allclose(Snew @ k[t], want, rtol=1e-12, atol=1e-12)
        S = Snew
    # Exact write with b = 1 on unit keys.
    e = np.eye(6)[[0, 2, 5]]
    o, S = O.delta_rule_prefill(bits(e[:, None]), bits(e[:, None]), c["v"][:3],
                                c["a"][:3], np.ones((3, 1), np.float32), [0, 3], c["S0"], [1],
                                literal=literal)
    np.testing.assert_allclose(S[0, 0] @ e[2], v[2], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[2, 0], v[2], rtol=0, atol=1e-12)


def test_delta_associative_memory():
    # a = b = 1, orthonormal keys e_t, S0 = 0: S_T = sum_t v_t e_t^T.
    dk, dv, T = 5, 3, 4
    e = np.eye(dk)[[4, 1, 0, 2]]
    c = synth.delta_case(14, [T], 1, 1, dk, dv)
    ones = np.ones((T, 1), np.float32)
    for literal in (True, False):
        _, S = O.delta_rule_prefill(bits(e[:, None]), bits(e[:, None]), c["v"], ones, ones,
                                    [0, T], np.zeros((1, 1, dv, dk)), [0], literal=literal)
        v = O.from_bf16(c["v"])[:, 0]
        assert np.array_equal(S[0, 0], sum(np.outer(v[t], e[t]) for t in range(T)))


def test_delta_head_map_contiguous_groups():
    # Hk = 2, Hv = 4: v-heads 0,1 read k-head 0 and v-heads 2,3 read k-head 1.
    # Same result as Hk = Hv = 4 with k-heads laid out as (k0, k0, k1, k1).
    c = synth.delta_case(15, [4, 3], 2, 4, 6, 5, s0_std=0.3)
    args = (c["v"], c["a"], c["b"], c["cu_seqlens"], c["S0"], c["has_initial_state"])
    o1, S1 = O.delta_rule_prefill(c["q"], c["k"], *args)
    rep = [0, 0, 1, 1]
    o2, S2 = O.delta_rule_prefill(c["q"][:, rep], c["k"][:, rep], *args)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_delta_decode_is_one_prefill_token():
    c = synth.delta_case(16, [1, 1, 1], 2, 4, 8, 6, s0_std=0.1)
    o1, S1 = O.delta_rule_decode(c["q"], c["k"], c["v"], c["a"], c["b"], c["S0"])
    o2, S2 = O.delta_rule_prefill(c["q"], c["k"], c["v"], c["a"], c["b"], c["cu_seqlens"],
                                  c["S0"], [1, 1, 1])
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_delta_prefill_then_decode_equals_longer_prefill():
    c = synth.delta_case(17, [12], 2, 4, 8, 6, s0_std=0.2)
    f = lambda sl, S0, has: O.delta_rule_prefill(c["q"][sl], c["k"][sl], c["v"][sl], c["a"][sl],
                                                 c["b"][sl], [0, sl.stop - sl.start], S0, has)
    o, S = f(slice(0, 12), c["S0"], [1])
    oa, Sa = f(slice(0, 9), c["S0"], [1])
    parts = [oa]
    for t in range(9, 12):
        od, Sa = O.delta_rule_decode(c["q"][t:t + 1], c["k"][t:t + 1], c["v"][t:t + 1],
                                     c["a"][t:t + 1], c["b"][t:t + 1], Sa)
        parts.append(od)
    assert np.array_equal(np.concatenate(parts), o) and np.array_equal(Sa, S)


@pytest.mark.parametrize("chunk", [1, 3, 4, 8, 64])
def test_chunked_equals_sequential(chunk):
    c = synth.delta_case(18, [13, 0, 5, 21], 2, 4, 8, 6, s0_std=0.3)
    c["has_initial_state"] = np.array([1, 1, 0, 1], np.uint8)
    args = (c["q"], c["k"], c["v"], c["a"], c["b"], c["cu_seqlens"], c["S0"], c["has_initial_state"])
    o_seq, S_seq = O.delta_rule_prefill(*args)
    o_chk, S_chk = O.delta_rule_prefill_chunked(*args, chunk=chunk)
    np.testing.assert_allclose(o_chk, o_seq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_chk, S_seq, rtol=0, atol=1e-12)


def test_qk_l2norm_flag_matches_pre_normalised_values():
    c = synth.delta_case(19, [6], 1, 2, 4, 4, s0_std=0.1, normed_qk=False)
    q, k = O.from_bf16(c["q"]), O.from_bf16(c["k"])
    qn = O.l2norm(q)
    kn = O.l2norm(k)
    o1, S1 = O.delta_rule_prefill(c["q"], c["k"], c["v"], c["a"], c["b"], [0, 6], c["S0"], [1],
                                  qk_l2norm=True)
    # Same recurrence run on the normalised values (float64, not re-rounded).
    v = O.from_bf16(c["v"])
    S = c["S0"][0].astype(np.float64)
    for t in range(6):
        o, S = O.delta_rule_step_literal(S, qn[t, [0, 0]], kn[t, [0, 0]], v[t],
                                         c["a"][t].astype(np.float64), c["b"][t].astype(np.float64))
        np.testing.assert_allclose(o1[t], o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S1[0], S, rtol=1e-12, atol=1e-14)


def test_oracle_matches_committed_tiny_fixture():
    import json
    import os
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    sys.path.insert(0, os.path.join(here, "golden"))
    from make_golden import tiny_expectations
    with open(os.path.join(here, "golden", "tiny_oracle.json")) as f:
        stored = json.load(f)
    now = tiny_expectations()
    for key in ("chunks", "conv_y_bf16", "conv_state_bf16", "delta_o_bf16"):
        assert now[key] == stored[key], key
    assert abs(now["delta_S_sum"] - stored["delta_S_sum"]) <= 1e-12 * max(1.0, stored["delta_S_abs_sum"])
