"""The allocation-free chunked prefill against the regular one, on the GPU.

gdn_delta_rule_prefill_chunked_noalloc serves callers that may not call
cudaMalloc (host frameworks that own every device allocation, plugins in a
foreign CUDA context, allocation-free call sites): its scratch is a fixed
64 MiB array inside the library instead of a caller workspace. This file runs
last (pytest collects it after the other test files), so a failure here
cannot hide the results of the rest of the suite; it also passes when run on
its own in a fresh process.

Two calls in a row, with different inputs and shapes, must each match the
regular entry point (which gets its own workspace) within the tolerances of
the parity tests: the array keeps the first call's contents, and the second
call must not be affected by them. (The regular entry point is itself checked
against the oracle by the parity tests; this variant only changes where the
scratch lives, so it is compared with the regular call.) The device-side
status words, which live in the library's array, are read back through
gdn_delta_rule_prefill_chunked_noalloc_status: GDN_OK after a good call,
GDN_ERR_INVALID_ARG after one with malformed cu_seqlens (which then leaves
state and outputs untouched).
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_STATE = 1e-4


def rel(x, ref):
    x, ref = x.double(), ref.double()
    return float((x - ref).abs().max() / ref.abs().max().clamp_min(1e-30))


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


def run_both(G, d, l2=False):
    T, Hk, dk = d["q"].shape
    Hv, dv = d["v"].shape[1], d["v"].shape[2]
    N = len(d["cu_seqlens"]) - 1
    q, k, v = bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"])
    a, b = dev(d["a"]), dev(d["b"])
    cu, has = dev(d["cu_seqlens"]), dev(d["has_initial_state"])
    S0 = dev(d["S0"].reshape(N, Hv, dv, dk))
    S_ref, S_na = S0.clone(), S0.clone()
    o_ref = torch.empty((T, Hv, dv), dtype=torch.bfloat16, device="cuda")
    o_na = torch.full((T, Hv, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.delta_rule_prefill_workspace_size(T, N, Hv, dk, dv), dtype=torch.uint8,
                     device="cuda")
    G.delta_rule_prefill_chunked(q, k, v, a, b, cu, S_ref, has, o_ref, ws, qk_l2norm=l2)
    G.delta_rule_prefill_chunked_noalloc(q, k, v, a, b, cu, S_na, has, o_na, qk_l2norm=l2)
    torch.cuda.synchronize()
    return o_na, o_ref, S_na, S_ref


def test_noalloc_matches_regular_entry_point_twice(G):
    first = synth.delta_case(71, [200, 63, 300], 16, 32, 128, 128, s0_std=0.05)
    second = synth.delta_case(72, [129, 64], 2, 4, 128, 128, s0_std=0.1)
    second["has_initial_state"] = np.array([0, 1], np.uint8)
    for d in (first, second):
        o_na, o_ref, S_na, S_ref = run_both(G, d)
        assert not torch.isnan(o_na.float()).any()
        assert rel(o_na.float(), o_ref.float()) < TOL_BF16
        assert rel(S_na, S_ref) < TOL_STATE


def test_noalloc_small_head_dim_and_size_limit(G):
    d = synth.delta_case(73, [70, 5], 2, 4, 64, 64, s0_std=0.05, normed_qk=False)
    o_na, o_ref, S_na, S_ref = run_both(G, d, l2=True)
    assert rel(o_na.float(), o_ref.float()) < TOL_BF16
    assert rel(S_na, S_ref) < TOL_STATE
    # A workspace larger than the fixed array is rejected before any launch.
    big = synth.delta_case(74, [1024, 1024], 16, 32, 128, 128)
    with pytest.raises(G.GdnError) as exc:
        run_both(G, big)
    assert exc.value.status == G.GDN_ERR_WORKSPACE


@pytest.mark.parametrize("d", [128, 64])
def test_noalloc_status_words(G, d):
    hk, hv, T = 2, 4, 100
    case = synth.delta_case(75, [T], hk, hv, d, d, s0_std=0.05)
    status = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    # a good call: both words GDN_OK
    q, k, v = bf16_dev(case["q"]), bf16_dev(case["k"]), bf16_dev(case["v"])
    a, b = dev(case["a"]), dev(case["b"])
    S = dev(case["S0"])
    o = torch.empty((T, hv, d), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_prefill_chunked_noalloc(q, k, v, a, b, dev(case["cu_seqlens"]), S,
                                         dev(case["has_initial_state"]), o)
    G.delta_rule_prefill_chunked_noalloc_status(status)
    torch.cuda.synchronize()
    assert status.tolist() == [G.GDN_OK, G.GDN_OK]
    # malformed cu_seqlens (the second entry decreases): reported, nothing touched
    N = 2
    S0 = (0.05 * np.random.default_rng(76).standard_normal((N, hv, d, d))).astype(np.float32)
    S = dev(S0)
    o = torch.full((T, hv, d), 3.0, dtype=torch.bfloat16, device="cuda")
    G.delta_rule_prefill_chunked_noalloc(q, k, v, a, b, dev(np.array([0, T, 50], np.int32)), S,
                                         dev(np.ones(N, np.uint8)), o)
    host = torch.full((2,), -7, dtype=torch.int32).pin_memory()
    G.delta_rule_prefill_chunked_noalloc_status(host)
    torch.cuda.synchronize()
    assert host[0].item() == G.GDN_ERR_INVALID_ARG
    assert host[1].item() == (G.GDN_ERR_INVALID_ARG if d == 128 else G.GDN_OK)
    assert torch.equal(S, dev(S0))
    assert bool((o.float() == 3.0).all())
