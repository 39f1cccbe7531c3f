"""Pins of the oracle's synthetic serving stack (CPU only).

The stack wraps the pinned conv and delta-rule oracles in model glue; these
tests pin the glue and the generation loop against what the mathematics fixes:
special cases with closed forms and the prefill-then-decode invariant at the
level of the whole stack.
"""
import numpy as np
import pytest

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth

TINY = dict(layers=2, n_seqs=3, vocab=50, hk=1, hv=2, d=16, len_lo=5, len_hi=40)


def tiny_stack(seed=4):
    return synth.serving_stack(seed, **TINY)


def test_rms_norm_unit_mean_square_and_power_of_two_invariance():
    rng = np.random.default_rng(11)
    h = rng.standard_normal((7, 64)) * rng.uniform(0.1, 10.0, (7, 1))
    x = O.from_bf16(O.rms_norm_bf16(h))
    # mean(x^2) = 1 up to the 1e-6 epsilon and BF16 rounding (|rel| <= 2^-8 each)
    assert np.all(np.abs(np.mean(x * x, axis=1) - 1.0) < 2.0 ** -7)
    # scaling by a power of two scales mean(h^2) exactly; only eps can move it
    big = 64.0
    assert np.array_equal(O.rms_norm_bf16(h * big), O.rms_norm_bf16(h * big * 4.0))


def test_gates_closed_forms():
    """exp(-softplus(z)) = 1 / (1 + e^z) and sigmoid(z) = 1 / (1 + e^-z)."""
    rng = np.random.default_rng(12)
    hk, hv, d = 1, 3, 8
    x = rng.standard_normal((5, 2 * hk * d + hv * d))
    u = rng.standard_normal((hv, d))
    r = rng.standard_normal((hv, d))
    a, b = O._gates(x, u, r, hk, hv, d)
    xv = x[:, 2 * hk * d:].reshape(5, hv, d)
    for t in range(5):
        for h in range(hv):
            za = sum(xv[t, h, j] * u[h, j] for j in range(d)) / np.sqrt(d)
            zb = sum(xv[t, h, j] * r[h, j] for j in range(d)) / np.sqrt(d)
            assert a[t, h] == pytest.approx(1.0 / (1.0 + np.exp(za)), rel=1e-6)
            assert b[t, h] == pytest.approx(1.0 / (1.0 + np.exp(-zb)), rel=1e-6)
    assert a.dtype == np.float32 and b.dtype == np.float32


def test_zero_residual_scale_reduces_to_a_bigram_map():
    """With s = 0 every layer leaves h = embedding, so the next id is a fixed
    function of the current one: argmax over bf16(rms(E[t])) . W."""
    st = tiny_stack()
    st["res_scale"] = [np.zeros_like(s) for s in st["res_scale"]]
    E = O.from_bf16(st["embed"])
    W = O.from_bf16(st["head"])

    def next_id(t):
        e = E[t]
        x = O.from_bf16(O.to_bf16(e / np.sqrt(np.mean(e * e) + 1e-6)))
        return int(np.argmax(x @ W))

    for s in range(3):
        ids, margins, _ = O.serving_stack_sequence(st, s, n_decode=5)
        expect = [next_id(int(st["prompts"][s][-1]))]
        for _ in range(5):
            expect.append(next_id(expect[-1]))
        assert ids == expect
        assert all(m >= 0 for m in margins)


def test_argmax_takes_the_first_of_equal_logits():
    st = tiny_stack()
    st["res_scale"] = [np.zeros_like(s) for s in st["res_scale"]]
    # make columns 3 and 7 of the head identical and dominant: every token ties
    head = O.from_bf16(st["head"])
    col = np.abs(head).max() * 4.0 * np.ones(head.shape[0])
    head[:, 3] = col
    head[:, 7] = col
    st["head"] = O.to_bf16(head)
    # x has entries of both signs, so force a positive logit with x>0 rows:
    E = np.abs(O.from_bf16(st["embed"]))
    st["embed"] = O.to_bf16(E)
    ids, margins, _ = O.serving_stack_sequence(st, 0, n_decode=3)
    assert ids == [3, 3, 3, 3]
    assert margins == [0.0] * 4


@pytest.mark.parametrize("s", [0, 1, 2])
def test_prefill_then_decode_equals_one_longer_prefill(s):
    """Generating n tokens step by step (conv_state and S handed from the
    prompt to the decode forms, layer by layer) gives the logits that one
    prefill of prompt + generated[:-1] gives at the same positions."""
    st = tiny_stack()
    ids, margins, rows = O.serving_stack_sequence(st, s, n_decode=6)
    prompt = list(st["prompts"][s])
    full = O.serving_stack_prefill_logits(st, prompt + ids[:-1])
    L = len(prompt)
    assert np.max(np.abs(full[L - 1:] - rows)) <= 1e-9 * np.max(np.abs(rows))
    assert [int(np.argmax(r)) for r in full[L - 1:]] == ids


def test_stack_depends_on_every_layer():
    """Changing the last layer's conv weights changes the logits (no layer is
    skipped) while zeroing its residual scale removes its effect exactly."""
    st = tiny_stack()
    _, _, rows = O.serving_stack_sequence(st, 1, n_decode=2)
    st2 = tiny_stack()
    st2["conv_w"][-1] = O.to_bf16(-O.from_bf16(st2["conv_w"][-1]))
    _, _, rows2 = O.serving_stack_sequence(st2, 1, n_decode=2)
    assert np.max(np.abs(rows2 - rows)) > 1e-3
    st3 = tiny_stack()
    st3["res_scale"][-1] = np.zeros_like(st3["res_scale"][-1])
    st4 = tiny_stack()
    st4["res_scale"][-1] = np.zeros_like(st4["res_scale"][-1])
    st4["conv_w"][-1] = st2["conv_w"][-1]
    _, _, r3 = O.serving_stack_sequence(st3, 1, n_decode=2)
    _, _, r4 = O.serving_stack_sequence(st4, 1, n_decode=2)
    assert np.array_equal(r3, r4)
