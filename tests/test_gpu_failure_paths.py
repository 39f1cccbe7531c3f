"""Failure detection on the GPU without a GPU fault.

* The bounded device-side wait that every kernel of the library uses on its
  mbarriers gives up by itself: a self-test CTA waits for a phase that nothing
  completes, reports GDN_ERR_TIMEOUT, and the context stays usable.
* The library's sticky device status (gdn_device_status) reads GDN_OK after a
  full pass of every kernel kind, GDN_ERR_TIMEOUT once a wait has given up
  (recorded by the self-test CTA through the same path the conv, decode and
  prefill kernels use), and GDN_OK again after a clear.
* Malformed cu_seqlens (a decreasing entry), which the host cannot see before
  launch, reach the device-side status words of the prefill workspace; the
  chunked prefill then leaves its outputs and the state untouched instead of
  reading records it never wrote.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, dev

pytestmark = pytest.mark.gpu

SENTINEL = 3.0


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


def test_bounded_wait_gives_up_and_context_survives(G):
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    G.selftest_bounded_wait(status, max_cycles=2_000_000)   # about a millisecond
    torch.cuda.synchronize()
    assert int(status.item()) == G.GDN_ERR_TIMEOUT
    # the context still runs kernels: a small decode step
    d = synth.delta_case(95, [1] * 4, 2, 4, 128, 128, s0_std=0.02, normed_qk=False)
    S = dev(d["S0"].reshape(4, 4, 128, 128))
    o = torch.empty((4, 4, 128), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_decode(bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"]), dev(d["a"]),
                        dev(d["b"]), S, o, qk_l2norm=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()


def run_every_kernel_kind(G):
    """Descriptors, conv prefill and update, decode (streaming and generic),
    chunked prefill (tensor-core and SIMT) and the fused decode step, small."""
    C = 2 * 2 * 128 + 4 * 128
    conv = synth.conv_case(97, [40, 9], C, initial_state=True)
    cu = dev(conv["cu_seqlens"])
    T = conv["x"].shape[0]
    chunks = torch.empty((T // 8 + 2, 4), dtype=torch.int32, device="cuda")
    count = torch.empty((1,), dtype=torch.int32, device="cuda")
    G.build_conv_chunks(cu, chunks, count, chunk_tokens=8)
    st = bf16_dev(conv["conv_state"])
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    w = bf16_dev(conv["w"])
    G.causal_conv1d_fwd(bf16_dev(conv["x"]), w, None, st, dev(conv["has_initial_state"]), cu, y,
                        chunks=chunks, num_chunks=count)
    yu = torch.empty((2, C), dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_update(y[:2].contiguous(), w, None, st, yu)
    for d in (128, 64):
        c = synth.delta_case(98 + d, [70, 5], 2, 4, d, d, s0_std=0.02)
        S = dev(c["S0"])
        o = torch.empty((c["T"], 4, d), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(G.delta_rule_prefill_workspace_size(c["T"], 2, 4, d, d),
                         dtype=torch.uint8, device="cuda")
        G.delta_rule_prefill_chunked(bf16_dev(c["q"]), bf16_dev(c["k"]), bf16_dev(c["v"]),
                                     dev(c["a"]), dev(c["b"]), dev(c["cu_seqlens"]), S,
                                     dev(c["has_initial_state"]), o, ws)
        od = torch.empty((2, 4, d), dtype=torch.bfloat16, device="cuda")
        G.delta_rule_decode(bf16_dev(c["q"][:2]), bf16_dev(c["k"][:2]), bf16_dev(c["v"][:2]),
                            dev(c["a"][:2]), dev(c["b"][:2]), S, od)
    Sd = torch.zeros((2, 4, 128, 128), device="cuda")
    st_out = torch.empty_like(st)
    G.decode_step_fused(y[:2].contiguous(), w, None, st, st_out, dev(c["a"][:2]),
                        dev(c["b"][:2]), Sd, torch.empty((2, 4, 128), dtype=torch.bfloat16,
                                                         device="cuda"), Hk=2)


def test_device_status_sticky_read_and_clear(G):
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    G.device_status(status, clear=True)           # start from a clean status
    run_every_kernel_kind(G)
    G.device_status(status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.GDN_OK
    word = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    G.selftest_bounded_wait(word, max_cycles=2_000_000)    # a wait that gives up
    G.device_status(status)
    torch.cuda.synchronize()
    assert int(word.item()) == G.GDN_ERR_TIMEOUT
    assert int(status.item()) == G.GDN_ERR_TIMEOUT
    G.device_status(status)                       # sticky: still there
    torch.cuda.synchronize()
    assert int(status.item()) == G.GDN_ERR_TIMEOUT
    G.device_status(status, clear=True)
    G.device_status(status)
    torch.cuda.synchronize()
    assert int(status.item()) == G.GDN_OK


@pytest.mark.parametrize("d", [128, 64])
def test_malformed_cu_seqlens_reported_on_device(G, d):
    hk, hv, T = 2, 4, 100
    case = synth.delta_case(96, [T], hk, hv, d, d, s0_std=0.05)
    cu = dev(np.array([0, T, 50], np.int32))          # the second entry decreases
    N = 2
    S0 = (0.05 * np.random.default_rng(97).standard_normal((N, hv, d, d))).astype(np.float32)
    S = dev(S0)
    has = dev(np.ones(N, np.uint8))
    o = torch.full((T, hv, d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = torch.full((G.delta_rule_prefill_workspace_size(T, N, hv, d, d),), 0x7f,
                    dtype=torch.uint8, device="cuda")
    G.delta_rule_prefill_chunked(bf16_dev(case["q"]), bf16_dev(case["k"]), bf16_dev(case["v"]),
                                 dev(case["a"]), dev(case["b"]), cu, S, has, o, ws,
                                 qk_l2norm=True)
    torch.cuda.synchronize()
    builder, state_pass = G.prefill_workspace_status(ws)
    assert builder == G.GDN_ERR_INVALID_ARG
    # the tensor-core state pass sees the missing chunks; the SIMT one (d < 128)
    # has no waits and reports GDN_OK
    assert state_pass == (G.GDN_ERR_INVALID_ARG if d == 128 else G.GDN_OK)
    # no chunk records exist, so the state pass touched neither S nor o
    assert torch.equal(S, dev(S0))
    assert bool((o.float() == SENTINEL).all())
