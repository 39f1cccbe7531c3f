"""Two follow-on engine cases on the GPU, through the C ABI.

Mixed step: one engine step that carries a prefill segment and decode tokens
together ("RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM",
Problem: the engine batches 2048 tokens per step across 32 concurrent
requests, so prefill chunks and decode tokens share steps). The decode tokens
ride the prefill calls as one-token sequences that continue from their state.
The mixed step is checked against the oracle (conv outputs elementwise, conv
state bytes exact, delta-rule outputs and states within the BF16 / float32
bars), and against separate prefill and decode calls on the GPU: conv outputs
and conv state bytes identical (the same arithmetic per element).

Other model shapes: the same kernels at other (q/k heads, v-heads) layouts of
width 128, checked against the oracle: 16 / 48 heads (conv width 10240, three
v-heads per q/k head) and 8 / 16 heads (conv width 4096).
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, bf16_host_bits, bf16_values, dev
from parity import assert_S, assert_conv_y, assert_o

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


def same_bits(x, y):
    return torch.equal(x.contiguous().view(torch.int16), y.contiguous().view(torch.int16))


def views(y, hk, hv):
    T = y.shape[0]
    return (y[:, :hk * D].view(T, hk, D), y[:, hk * D:2 * hk * D].view(T, hk, D),
            y[:, 2 * hk * D:].view(T, hv, D))


def test_mixed_prefill_and_decode_step(G):
    hk, hv = 16, 32
    C = 2 * hk * D + hv * D
    rng = np.random.default_rng(61)
    n_dec, L = 5, 200                                   # 5 decode tokens + a 200-token segment
    lens = [L] + [1] * n_dec
    cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu_h[-1])
    x = synth.normal_bf16(rng, (T, C))
    w = synth.normal_bf16(rng, (C, 4), std=0.5)
    st0 = synth.normal_bf16(rng, (len(lens), C, 3))
    a, b = synth.gates(rng, (T, hv))
    S0 = (0.02 * rng.standard_normal((len(lens), hv, D, D))).astype(np.float32)
    has = np.ones(len(lens), np.uint8)

    # --- one mixed step: conv over descriptors, then the chunked delta rule
    cu = dev(cu_h)
    st = bf16_dev(st0)
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    chunks = torch.empty((T // 8 + len(lens), 4), dtype=torch.int32, device="cuda")
    count = torch.empty((1,), dtype=torch.int32, device="cuda")
    G.build_conv_chunks(cu, chunks, count, chunk_tokens=8)
    G.causal_conv1d_fwd(bf16_dev(x), bf16_dev(w), None, st, dev(has), cu, y, chunks=chunks,
                        num_chunks=count)
    S = dev(S0)
    o = torch.empty((T, hv, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.delta_rule_prefill_workspace_size(T, len(lens), hv, D, D),
                     dtype=torch.uint8, device="cuda")
    q, k, v = views(y, hk, hv)
    G.delta_rule_prefill_chunked(q, k, v, dev(a), dev(b), cu, S, dev(has), o, ws, qk_l2norm=True)

    # --- the same work as separate calls: prefill of the segment, decode of the rest
    st_p = bf16_dev(st0[:1])
    y_p = torch.empty((L, C), dtype=torch.bfloat16, device="cuda")
    cu_p = dev(np.array([0, L], np.int32))
    G.causal_conv1d_fwd(bf16_dev(x[:L]), bf16_dev(w), None, st_p, dev(has[:1]), cu_p, y_p)
    S_p = dev(S0[:1])
    o_p = torch.empty((L, hv, D), dtype=torch.bfloat16, device="cuda")
    ws_p = torch.empty(G.delta_rule_prefill_workspace_size(L, 1, hv, D, D), dtype=torch.uint8,
                       device="cuda")
    qp, kp, vp = views(y_p, hk, hv)
    G.delta_rule_prefill_chunked(qp, kp, vp, dev(a[:L]), dev(b[:L]), cu_p, S_p, dev(has[:1]),
                                 o_p, ws_p, qk_l2norm=True)
    st_d = bf16_dev(st0[1:])
    y_d = torch.empty((n_dec, C), dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_update(bf16_dev(x[L:]), bf16_dev(w), None, st_d, y_d)
    S_d = dev(S0[1:])
    o_d = torch.empty((n_dec, hv, D), dtype=torch.bfloat16, device="cuda")
    qd, kd, vd = views(y_d, hk, hv)
    G.delta_rule_decode(qd, kd, vd, dev(a[L:]), dev(b[L:]), S_d, o_d, qk_l2norm=True)
    torch.cuda.synchronize()

    assert same_bits(y[:L], y_p) and same_bits(y[L:], y_d)
    assert same_bits(st[:1], st_p) and same_bits(st[1:], st_d)

    # --- the oracle on the mixed step's layout. The conv over the mixed batch
    # (decode tokens as one-token sequences with their state) on the same
    # inputs; the chunked delta-rule call over the same cu_seqlens (one
    # 200-token segment, five one-token sequences continuing from their
    # state) on seeded q / k / v, against the recurrence token by token. (The
    # oracle never takes the GPU's conv output as its input.)
    yr, sr = O.causal_conv1d_fwd(x, w, None, st0, has, cu_h)
    assert_conv_y(bf16_values(y), yr)
    assert np.array_equal(bf16_host_bits(st), O.to_bf16(sr))
    dm = synth.delta_case(62, lens, hk, hv, D, D, s0_std=0.02, normed_qk=False)
    dm["has_initial_state"][:] = 1
    S2 = dev(dm["S0"])
    o2 = torch.empty((T, hv, D), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_prefill_chunked(bf16_dev(dm["q"]), bf16_dev(dm["k"]), bf16_dev(dm["v"]),
                                 dev(dm["a"]), dev(dm["b"]), cu, S2, dev(dm["has_initial_state"]),
                                 o2, ws, qk_l2norm=True)
    torch.cuda.synchronize()
    o_r, S_r = O.delta_rule_prefill(dm["q"], dm["k"], dm["v"], dm["a"], dm["b"], cu_h, dm["S0"],
                                    dm["has_initial_state"], qk_l2norm=True)
    assert_o(bf16_values(o2), o_r)
    assert_S(S2.cpu().numpy(), S_r)
    # and the separate GPU calls agree with the mixed step within the same bars
    assert_o(bf16_values(o), torch.cat([o_p, o_d]).float().cpu().numpy())
    assert_S(S.cpu().numpy(), torch.cat([S_p, S_d]).cpu().numpy())


@pytest.mark.parametrize("hk,hv", [(16, 48), (8, 16)])
def test_other_model_shapes(G, hk, hv):
    C = 2 * hk * D + hv * D
    # conv prefill over exact chunks, two ragged sequences with initial state
    case = synth.conv_case(71 + hk, [203, 77], C, initial_state=True)
    x, w = bf16_dev(case["x"]), bf16_dev(case["w"])
    st = bf16_dev(case["conv_state"])
    cu = dev(case["cu_seqlens"])
    T = case["x"].shape[0]
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    chunks = torch.empty((T // 8 + 2, 4), dtype=torch.int32, device="cuda")
    count = torch.empty((1,), dtype=torch.int32, device="cuda")
    G.build_conv_chunks(cu, chunks, count, chunk_tokens=8)
    G.causal_conv1d_fwd(x, w, None, st, dev(case["has_initial_state"]), cu, y, chunks=chunks,
                        num_chunks=count)
    torch.cuda.synchronize()
    yr, sr = O.causal_conv1d_fwd(case["x"], case["w"], None, case["conv_state"],
                                 case["has_initial_state"], case["cu_seqlens"])
    assert_conv_y(bf16_values(y), yr)
    assert np.array_equal(bf16_host_bits(st), O.to_bf16(sr))

    # conv update + decode, 6 sequences
    cu_case = synth.conv_update_case(72 + hk, 6, C)
    x1 = bf16_dev(cu_case["x"])
    st1 = bf16_dev(cu_case["conv_state"])
    y1 = torch.empty_like(x1)
    G.causal_conv1d_update(x1, bf16_dev(cu_case["w"]), None, st1, y1)
    torch.cuda.synchronize()
    y1r, s1r = O.causal_conv1d_update(cu_case["x"], cu_case["w"], None, cu_case["conv_state"])
    assert_conv_y(bf16_values(y1), y1r)
    assert np.array_equal(bf16_host_bits(st1), O.to_bf16(s1r))

    d = synth.delta_case(73 + hk, [1] * 6, hk, hv, D, D, s0_std=0.02, normed_qk=False)
    q, k, v = bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"])
    S = dev(d["S0"].reshape(6, hv, D, D))
    o = torch.empty((6, hv, D), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_decode(q, k, v, dev(d["a"]), dev(d["b"]), S, o, qk_l2norm=True)
    torch.cuda.synchronize()
    o_r, S_r = O.delta_rule_decode(d["q"], d["k"], d["v"], d["a"], d["b"],
                                   d["S0"].reshape(6, hv, D, D), qk_l2norm=True)
    assert_o(bf16_values(o), o_r)
    assert_S(S.cpu().numpy(), S_r)

    # chunked prefill, two ragged sequences with initial state (all heads)
    d = synth.delta_case(74 + hk, [150, 70], hk, hv, D, D, s0_std=0.05)
    T = d["q"].shape[0]
    S = dev(d["S0"].reshape(2, hv, D, D))
    o = torch.empty((T, hv, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.delta_rule_prefill_workspace_size(T, 2, hv, D, D), dtype=torch.uint8,
                     device="cuda")
    G.delta_rule_prefill_chunked(bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"]),
                                 dev(d["a"]), dev(d["b"]), dev(d["cu_seqlens"]), S,
                                 dev(d["has_initial_state"]), o, ws)
    torch.cuda.synchronize()
    o_r, S_r = O.delta_rule_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu_seqlens"],
                                    d["S0"], d["has_initial_state"])
    assert_o(bf16_values(o), o_r)
    assert_S(S.cpu().numpy(), S_r)
