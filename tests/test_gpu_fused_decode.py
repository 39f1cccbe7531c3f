"""The fused decode step (conv update + delta-rule decode in one launch) on the GPU.

Two checks:
  * against the two separate calls on the GPU: o, S and the new conv state
    are bit-identical (the fused kernel rounds the conv output to BF16 exactly
    where the separate conv update stores it);
  * against the oracle: conv update, BF16 rounding, split into q | k | v, then
    the decode, with the tolerances of the separate calls (state bytes exact).
Workload: 32 sequences, 16 q/k heads and 32 v-heads of 128 (8192 conv
channels), S ~ N(0, 0.02^2), in-kernel q/k L2 norm; with and without bias,
with and without SiLU; several steps in a row with alternating state buffers.
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, bf16_host_bits, bf16_values, dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_STATE = 1e-4
HK, HV, D, N = 16, 32, 128, 32
C = 2 * HK * D + HV * D


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


def make_case(seed, bias, steps=1):
    rng = np.random.default_rng(seed)
    return dict(
        x=[synth.normal_bf16(rng, (N, C)) for _ in range(steps)],
        w=synth.normal_bf16(rng, (C, 4), std=0.5),
        bias=synth.normal_bf16(rng, (C,), std=0.5) if bias else None,
        state=synth.normal_bf16(rng, (N, C, 3)),
        gates=[synth.gates(rng, (N, HV)) for _ in range(steps)],
        S0=(0.02 * rng.standard_normal((N, HV, D, D))).astype(np.float32),
    )


def two_calls(G, case, silu, l2):
    """The separate conv update and decode, step after step."""
    w = bf16_dev(case["w"])
    bias = bf16_dev(case["bias"]) if case["bias"] is not None else None
    st = bf16_dev(case["state"])
    S = dev(case["S0"])
    outs = []
    for x_bits, (a, b) in zip(case["x"], case["gates"]):
        x = bf16_dev(x_bits)
        y = torch.empty_like(x)
        G.causal_conv1d_update(x, w, bias, st, y, silu=silu)
        q = y[:, :HK * D].view(N, HK, D)
        k = y[:, HK * D:2 * HK * D].view(N, HK, D)
        v = y[:, 2 * HK * D:].view(N, HV, D)
        o = torch.empty((N, HV, D), dtype=torch.bfloat16, device="cuda")
        G.delta_rule_decode(q, k, v, dev(a), dev(b), S, o, qk_l2norm=l2)
        outs.append(o)
    torch.cuda.synchronize()
    return outs, S, st


def fused(G, case, silu, l2):
    w = bf16_dev(case["w"])
    bias = bf16_dev(case["bias"]) if case["bias"] is not None else None
    st = [bf16_dev(case["state"]), torch.empty((N, C, 3), dtype=torch.bfloat16, device="cuda")]
    S = dev(case["S0"])
    outs = []
    for i, (x_bits, (a, b)) in enumerate(zip(case["x"], case["gates"])):
        o = torch.empty((N, HV, D), dtype=torch.bfloat16, device="cuda")
        G.decode_step_fused(bf16_dev(x_bits), w, bias, st[i % 2], st[(i + 1) % 2], dev(a), dev(b),
                            S, o, Hk=HK, silu=silu, qk_l2norm=l2)
        outs.append(o)
    torch.cuda.synchronize()
    return outs, S, st[len(case["x"]) % 2]


def same_bits(x, y):
    return torch.equal(x.contiguous().view(torch.int32 if x.dtype == torch.float32 else torch.int16),
                       y.contiguous().view(torch.int32 if y.dtype == torch.float32 else torch.int16))


@pytest.mark.parametrize("bias,silu,l2", [(False, True, True), (True, True, True),
                                          (True, False, False)])
def test_fused_equals_two_calls_bitwise(G, bias, silu, l2):
    case = make_case(51 + int(bias) + 2 * int(silu), bias, steps=3)
    o1, S1, st1 = two_calls(G, case, silu, l2)
    o2, S2, st2 = fused(G, case, silu, l2)
    for a_, b_ in zip(o1, o2):
        assert same_bits(a_, b_)
    assert same_bits(S1, S2)
    assert same_bits(st1, st2)


def test_fused_against_oracle(G):
    case = make_case(57, bias=True, steps=1)
    outs, S, st = fused(G, case, silu=True, l2=True)
    y, new_state = O.causal_conv1d_update(case["x"][0], case["w"], case["bias"], case["state"])
    yb = O.to_bf16(y)
    q = yb[:, :HK * D].reshape(N, HK, D)
    k = yb[:, HK * D:2 * HK * D].reshape(N, HK, D)
    v = yb[:, 2 * HK * D:].reshape(N, HV, D)
    a, b = case["gates"][0]
    o_ref, S_ref = O.delta_rule_decode(q, k, v, a, b, case["S0"], qk_l2norm=True)
    assert O.rel_err(bf16_values(outs[0]), o_ref) < TOL_BF16
    assert O.rel_err(S.cpu().numpy(), S_ref) < TOL_STATE
    assert np.array_equal(bf16_host_bits(st), O.to_bf16(new_state))
