"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (``parity.py``; relative error = max|x - ref| / max|ref|):
  * descriptors and conv_state bytes: bit-exact;
  * conv outputs y: elementwise, one BF16 rounding of a float32 value;
  * delta-rule outputs o: 2e-2 over the tensor, over each v-head and over each
    (token, v-head) row;
  * float32 recurrent state S: 1e-4 over each (sequence, v-head) state.
Exact-chunk and whole-sequence conv dispatch must be byte-identical, and so must
a prefill split across steps against one longer prefill (same kernels, same
arithmetic per element).
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, bf16_host_bits, bf16_values, dev
from parity import assert_S, assert_conv_y, assert_o

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


# ----------------------------------------------------------------------------
# a1 descriptors
# ----------------------------------------------------------------------------

def run_chunks(G, cu, chunk=8, capacity=None):
    cu_d = dev(np.asarray(cu, np.int32))
    T, N = int(cu[-1]), len(cu) - 1
    cap = capacity if capacity is not None else T // chunk + N
    chunks = torch.full((max(cap, 1), 4), -7, dtype=torch.int32, device="cuda")[:cap]
    count = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    G.build_conv_chunks(cu_d, chunks, count, chunk_tokens=chunk, device_status=status)
    torch.cuda.synchronize()
    n = int(count.item())
    return chunks[:n].cpu().numpy(), int(status.item())


@pytest.mark.parametrize("cu,chunk", [
    ([0, 5, 18], 8),
    ([0, 1024, 2048], 8),
    ([0, 0, 3, 3, 20, 84, 85, 85], 8),
    ([0, 7, 7, 30, 31], 1 << 20),                 # whole-sequence descriptors
    ([0, 1024, 2048], 64),
    ([0], 8),                                     # no sequences
])
def test_chunks_bit_exact(G, cu, chunk):
    got, st = run_chunks(G, cu, chunk)
    assert st == 0
    assert np.array_equal(got, O.build_conv_chunks(cu, chunk))


def test_chunks_many_sequences_bit_exact(G):
    rng = np.random.default_rng(21)
    lengths = rng.integers(0, 40, size=3000)          # > one 1024-sequence tile
    cu = synth.packed_lengths_cu(lengths)
    got, st = run_chunks(G, cu.tolist(), 8)
    assert st == 0
    assert np.array_equal(got, O.build_conv_chunks(cu, 8))


def test_chunks_capacity_and_bad_offsets(G):
    got, st = run_chunks(G, [0, 5, 18], 8, capacity=2)
    assert st == -4 and len(got) == 0
    got, st = run_chunks(G, [0, 9, 4], 8, capacity=8)     # decreasing offsets
    assert st == -1 and len(got) == 0


# ----------------------------------------------------------------------------
# a2 / a3 conv
# ----------------------------------------------------------------------------

def conv_gpu(G, case, mode="chunks", silu=True, x_stride_pad=0):
    T, C = case["x"].shape
    x = bf16_dev(case["x"])
    if x_stride_pad:
        xb = torch.zeros((T, C + x_stride_pad), dtype=torch.bfloat16, device="cuda")
        xb[:, :C] = x
        x = xb[:, :C]
    w = bf16_dev(case["w"])
    bias = bf16_dev(case["bias"])
    st = bf16_dev(case["conv_state"])
    has = dev(case["has_initial_state"])
    cu = dev(case["cu_seqlens"])
    y = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    N = len(case["cu_seqlens"]) - 1
    if mode == "whole":
        G.causal_conv1d_fwd(x, w, bias, st, has, cu, y, silu=silu)
    else:
        cap = T // 8 + N
        chunks = torch.empty((cap, 4), dtype=torch.int32, device="cuda")
        count = torch.empty((1,), dtype=torch.int32, device="cuda")
        G.build_conv_chunks(cu, chunks, count, chunk_tokens=8)
        G.causal_conv1d_fwd(x, w, bias, st, has, cu, y, chunks=chunks, num_chunks=count, silu=silu)
    torch.cuda.synchronize()
    return y, st


def check_conv(case, y, st, silu=True):
    yr, sr = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], case["conv_state"],
                                 case["has_initial_state"], case["cu_seqlens"], apply_silu=silu)
    # Elementwise: one BF16 rounding of an fp32 value (plus fp32 rounding).
    assert_conv_y(bf16_values(y), yr)
    assert np.array_equal(bf16_host_bits(st), O.to_bf16(sr))


def test_conv_tiny(G):
    conv, _ = synth.tiny(0)
    y, st = conv_gpu(G, conv)
    check_conv(conv, y, st)


def test_conv_prefill_full_size(G):
    case = synth.conv_prefill(1)
    y, st = conv_gpu(G, case)
    check_conv(case, y, st)


@pytest.mark.parametrize("silu", [True, False])
def test_conv_varlen_edges(G, silu):
    lengths = [1, 2, 0, 3, 4, 7, 8, 9, 16, 17, 0, 31, 100]
    case = synth.conv_case(31, lengths, 64, bias=True)
    case["has_initial_state"] = (np.arange(len(lengths)) % 3 != 1).astype(np.uint8)
    y, st = conv_gpu(G, case, silu=silu, x_stride_pad=8)
    check_conv(case, y, st, silu=silu)


def test_conv_exact_chunks_equal_whole_sequence_bytes(G):
    lengths = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 0, 144, 1000]
    case = synth.conv_case(32, lengths, 256, bias=True)
    case["has_initial_state"] = (np.arange(len(lengths)) % 2).astype(np.uint8)
    y1, s1 = conv_gpu(G, case, "chunks")
    y2, s2 = conv_gpu(G, case, "whole")
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(s1.view(torch.int16), s2.view(torch.int16))


def test_conv_update_full_size(G):
    conv, _ = synth.decode(2)
    x, w, b = bf16_dev(conv["x"]), bf16_dev(conv["w"]), bf16_dev(conv["bias"])
    st = bf16_dev(conv["conv_state"])
    y = torch.empty_like(x)
    G.causal_conv1d_update(x, w, b, st, y)
    torch.cuda.synchronize()
    yr, sr = O.causal_conv1d_update(conv["x"], conv["w"], conv["bias"], conv["conv_state"])
    assert_conv_y(bf16_values(y), yr)
    assert np.array_equal(bf16_host_bits(st), O.to_bf16(sr))


def test_conv_prefill_then_updates_equals_longer_prefill(G):
    # Prefill 2 x 37 tokens, versus prefill 2 x 30 then 7 single-token updates:
    # identical bytes for y and conv_state.
    C = 512
    case = synth.conv_case(33, [37, 37], C, bias=True)
    y_full, st_full = conv_gpu(G, case)
    xs = case["x"].reshape(2, 37, C)
    part = dict(case)
    part["x"] = np.concatenate([xs[0, :30], xs[1, :30]])
    part["cu_seqlens"] = synth.packed_lengths_cu([30, 30])
    y_a, st = conv_gpu(G, part)
    w, b = bf16_dev(case["w"]), bf16_dev(case["bias"])
    ys = []
    for t in range(30, 37):
        x_t = bf16_dev(np.stack([xs[0, t], xs[1, t]]))
        y_t = torch.empty_like(x_t)
        G.causal_conv1d_update(x_t, w, b, st, y_t)
        ys.append(y_t)
    torch.cuda.synchronize()
    yf = y_full.view(2, 37, C)
    ya = y_a.view(2, 30, C)
    assert torch.equal(yf[:, :30].contiguous().view(torch.int16), ya.contiguous().view(torch.int16))
    for i, t in enumerate(range(30, 37)):
        assert torch.equal(yf[:, t].contiguous().view(torch.int16), ys[i].view(torch.int16))
    assert torch.equal(st.view(torch.int16), st_full.view(torch.int16))


# ----------------------------------------------------------------------------
# a5 decode
# ----------------------------------------------------------------------------

def decode_gpu(G, d, qk_l2norm=False, strided=False):
    N, Hk, dk = d["q"].shape
    Hv, dv = d["v"].shape[1], d["v"].shape[2]
    if strided:
        # q, k, v as column slices of one [N, 2*Hk*dk + Hv*dv] buffer (the conv
        # output layout of the Qwen3.5-style GDN layer).
        width = 2 * Hk * dk + Hv * dv
        buf = torch.zeros((N, width), dtype=torch.bfloat16, device="cuda")
        buf[:, :Hk * dk] = bf16_dev(d["q"]).reshape(N, -1)
        buf[:, Hk * dk:2 * Hk * dk] = bf16_dev(d["k"]).reshape(N, -1)
        buf[:, 2 * Hk * dk:] = bf16_dev(d["v"]).reshape(N, -1)
        q = buf[:, :Hk * dk].view(N, Hk, dk)
        k = buf[:, Hk * dk:2 * Hk * dk].view(N, Hk, dk)
        v = buf[:, 2 * Hk * dk:].view(N, Hv, dv)
    else:
        q, k, v = bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"])
    a, b = dev(d["a"]), dev(d["b"])
    S = dev(d["S0"].reshape(N, Hv, dv, dk))
    o = torch.empty((N, Hv, dv), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_decode(q, k, v, a, b, S, o, qk_l2norm=qk_l2norm)
    torch.cuda.synchronize()
    return o, S


def check_decode(d, o, S, qk_l2norm=False):
    N = d["q"].shape[0]
    Hv, dv, dk = d["v"].shape[1], d["v"].shape[2], d["q"].shape[2]
    orf, Sr = O.delta_rule_decode(d["q"], d["k"], d["v"], d["a"], d["b"],
                                  d["S0"].reshape(N, Hv, dv, dk), qk_l2norm=qk_l2norm)
    eo = assert_o(bf16_values(o), orf)
    es = assert_S(S.cpu().numpy(), Sr)
    return eo, es


def test_decode_full_size(G):
    _, d = synth.decode(2)
    o, S = decode_gpu(G, d)
    check_decode(d, o, S)


def test_decode_many_sequences(G):
    # 101 sequences: 6,464 state units of 64 rows over the persistent CTAs, so
    # each CTA walks its stage ring several times over (and the units do not
    # divide evenly among the CTAs).
    d = synth.delta_case(43, [1] * 101, 16, 32, 128, 128, s0_std=0.02)
    o, S = decode_gpu(G, d, qk_l2norm=True)
    check_decode(d, o, S, qk_l2norm=True)


@pytest.mark.parametrize("n", [1, 3])
def test_decode_small_batches(G, n):
    # 64 or 192 state units: fewer units than persistent CTAs, or one or two
    # per CTA.
    d = synth.delta_case(44 + n, [1] * n, 16, 32, 128, 128, s0_std=0.02)
    o, S = decode_gpu(G, d)
    check_decode(d, o, S)


def test_decode_strided_views_and_l2norm(G):
    d = synth.delta_case(41, [1] * 32, 16, 32, 128, 128, s0_std=0.02, normed_qk=False)
    o, S = decode_gpu(G, d, qk_l2norm=True, strided=True)
    check_decode(d, o, S, qk_l2norm=True)


@pytest.mark.parametrize("dk,dv,hk,hv", [(16, 16, 2, 2), (128, 64, 2, 4), (64, 128, 1, 3),
                                         (32, 16, 4, 4)])
def test_decode_head_shapes(G, dk, dv, hk, hv):
    d = synth.delta_case(42, [1] * 5, hk, hv, dk, dv, s0_std=0.5)
    o, S = decode_gpu(G, d)
    check_decode(d, o, S)


# ----------------------------------------------------------------------------
# a6-a8 chunked prefill
# ----------------------------------------------------------------------------

def prefill_gpu(G, d, qk_l2norm=False):
    T, Hk, dk = d["q"].shape
    Hv, dv = d["v"].shape[1], d["v"].shape[2]
    N = len(d["cu_seqlens"]) - 1
    q, k, v = bf16_dev(d["q"]), bf16_dev(d["k"]), bf16_dev(d["v"])
    a, b = dev(d["a"]), dev(d["b"])
    S = dev(d["S0"].reshape(N, Hv, dv, dk))
    cu = dev(d["cu_seqlens"])
    has = dev(d["has_initial_state"])
    o = torch.full((T, Hv, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(G.delta_rule_prefill_workspace_size(T, N, Hv, dk, dv), dtype=torch.uint8,
                     device="cuda")
    G.delta_rule_prefill_chunked(q, k, v, a, b, cu, S, has, o, ws, qk_l2norm=qk_l2norm)
    torch.cuda.synchronize()
    return o, S


def check_prefill(d, o, S, qk_l2norm=False, heads=None):
    orf, Sr = O.delta_rule_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu_seqlens"],
                                   d["S0"], d["has_initial_state"], qk_l2norm=qk_l2norm,
                                   heads=heads)
    og, Sg = bf16_values(o), S.cpu().numpy().astype(np.float64)
    if heads is not None:
        og, orf, Sg, Sr = og[:, heads], orf[:, heads], Sg[:, heads], Sr[:, heads]
    eo = assert_o(og, orf)
    es = assert_S(Sg, Sr)
    return eo, es


def test_prefill_tiny(G):
    _, d = synth.tiny(0)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_prefill_varlen_ragged(G, D):
    lengths = [1, 63, 64, 65, 0, 130, 3]
    d = synth.delta_case(51, lengths, 2, 4, D, D, s0_std=0.05)
    d["has_initial_state"] = np.array([1, 0, 1, 1, 0, 1, 0], np.uint8)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


def test_prefill_l2norm_flag(G):
    d = synth.delta_case(52, [70, 129], 2, 4, 128, 128, s0_std=0.02, normed_qk=False)
    o, S = prefill_gpu(G, d, qk_l2norm=True)
    check_prefill(d, o, S, qk_l2norm=True)


def test_prefill_full_size(G):
    # 2 x 1024 tokens, all 32 v-heads of both sequences against the oracle.
    d = synth.prefill(3)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


def test_prefill_then_decode_equals_longer_prefill(G):
    # GPU: prefill 2 x 100 tokens, versus prefill 2 x 90 then 10 decode steps.
    L, L0 = 100, 90
    d = synth.delta_case(53, [L, L], 2, 4, 128, 128, s0_std=0.1)
    o_full, S_full = prefill_gpu(G, d)
    idx = lambda lo, hi: np.concatenate([np.arange(lo, hi), L + np.arange(lo, hi)])
    head = {k: (d[k][idx(0, L0)] if k in ("q", "k", "v", "a", "b") else d[k]) for k in d}
    head["cu_seqlens"] = synth.packed_lengths_cu([L0, L0])
    o_a, S = prefill_gpu(G, head)
    for t in range(L0, L):
        rows = np.array([t, L + t])
        step = {k: d[k][rows] for k in ("q", "k", "v", "a", "b")}
        step["S0"] = S.cpu().numpy()
        o_t, S = decode_gpu(G, step)
        ref = bf16_values(o_full)[rows]
        assert_o(bf16_values(o_t), ref)
    assert_S(S.cpu().numpy(), S_full.cpu().numpy())


def test_prefill_slow_decay_state_precision(G):
    # Gates close to 1 (a = exp(-softplus(z - 4.5))): the state keeps a long
    # memory, so every float32 product that feeds it must keep its precision.
    d = synth.delta_case(54, [300, 1024], 16, 32, 128, 128, s0_std=0.05)
    rng = np.random.default_rng(55)
    z = rng.standard_normal(d["a"].shape) - 4.5
    d["a"] = np.exp(-np.logaddexp(0.0, z)).astype(np.float32)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


def test_prefill_large_step(G):
    # 8,192 tokens of 4 sequences, all 32 v-heads over 16 k-heads, d = 128: 128
    # chains of up to 47 chunk steps, a 130-record-per-head workspace.
    d = synth.delta_case(60, [3000, 2500, 2000, 692], 16, 32, 128, 128, s0_std=0.02)
    d["has_initial_state"] = np.array([1, 0, 1, 0], np.uint8)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_many_short_sequences(G, D):
    # 200 sequences of 1-9 tokens (and a few empty ones): 800 one-chunk chains,
    # several waves of state CTAs in longest-first order with many ties.
    rng = np.random.default_rng(58)
    lengths = [int(x) for x in rng.integers(0, 10, size=200)]
    d = synth.delta_case(59, lengths, 2, 4, D, D, s0_std=0.05)
    d["has_initial_state"] = (np.arange(len(lengths)) % 3 != 0).astype(np.uint8)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_long_sequences(G, D):
    # Chains of 79 and 50 chunk steps plus a one-token sequence (8,192 tokens),
    # with slowly decaying gates so that the state carries information across
    # the whole chain; few heads keep the float64 oracle within seconds.
    lengths = [5000, 3191, 1]
    d = synth.delta_case(56, lengths, 2, 4, D, D, s0_std=0.05)
    d["has_initial_state"] = np.array([1, 0, 1], np.uint8)
    rng = np.random.default_rng(57)
    z = rng.standard_normal(d["a"].shape) - 4.5
    d["a"] = np.exp(-np.logaddexp(0.0, z)).astype(np.float32)
    o, S = prefill_gpu(G, d)
    check_prefill(d, o, S)


def test_conv_prefill_large_step(G):
    # 16,384 tokens x 8192 channels in one call (2,048 descriptors of 8 tokens):
    # each persistent CTA walks several times the runs of the 2048-token step.
    case = synth.conv_case(34, [9000, 4000, 3000, 384], 8192, bias=True)
    case["has_initial_state"] = np.array([1, 0, 1, 1], np.uint8)
    y, st = conv_gpu(G, case)
    check_conv(case, y, st)


def test_conv_long_sequences(G):
    # 8,000-token sequence (1,000 exact 8-token chunks) beside short ones.
    lengths = [8000, 191, 1]
    case = synth.conv_case(33, lengths, 256, bias=True)
    case["has_initial_state"] = np.array([1, 0, 1], np.uint8)
    y, st = conv_gpu(G, case)
    check_conv(case, y, st)


@pytest.mark.parametrize("D", [128, 64])
def test_prefill_plan_reused_by_two_layers_equals_unplanned(G, D):
    """One chunk plan per engine step ("perf(gdn): dispatch exact causal-conv
    chunks", What changed: built once per step, reused by every layer): two
    calls with different inputs on one plan give the bytes of two calls that
    build their own, which the tests above hold against the oracle."""
    lengths = [130, 1, 64, 0, 257, 7]
    cases = [synth.delta_case(60 + i, lengths, 2, 4, D, D, s0_std=0.05) for i in range(2)]
    T, N = cases[0]["T"], cases[0]["N"]
    cu = dev(cases[0]["cu_seqlens"])
    ws_plan = torch.empty(G.delta_rule_prefill_workspace_size(T, N, 4, D, D), dtype=torch.uint8,
                          device="cuda")
    G.delta_rule_prefill_plan(cu, T, 4, D, D, ws_plan)
    for c in cases:
        ref_o, ref_S = prefill_gpu(G, c)
        S = dev(c["S0"].reshape(N, 4, D, D))
        o = torch.full((T, 4, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        G.delta_rule_prefill_chunked(bf16_dev(c["q"]), bf16_dev(c["k"]), bf16_dev(c["v"]),
                                     dev(c["a"]), dev(c["b"]), cu, S, dev(c["has_initial_state"]),
                                     o, ws_plan, planned=True)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(S.view(torch.int32), ref_S.view(torch.int32))
