"""State-slot indirection on the GPU, through the C ABI.

The serving engine of "RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps
vs vLLM" (Problem: 32 concurrent requests served out of a fixed block cache)
keeps recurrent states in a cache that outlives a batch. The *_slots calls take
that cache plus a per-sequence slot map. Checked here, for every kernel of the
path (conv prefill with exact chunks and whole-sequence dispatch, conv update,
decode with d = 128 and d = 64, chunked prefill with d = 128 and d = 64):

  * a valid entry matches the oracle run on the states gathered from the
    cache (conv outputs elementwise and conv state bytes exactly; delta-rule
    outputs and states within the BF16 / float32 bars);
  * a valid entry gives bit-identical outputs and new state to the call
    without the suffix on the gathered states (the same arithmetic runs);
  * slots that no sequence names keep their bytes;
  * padding entries (index -1, or one past the cache) leave their state and
    their output rows untouched.
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from gated_deltanet_linear_build_gb300 import synth

from devutil import bf16_dev, bf16_host_bits, bf16_values, dev
from parity import assert_S, assert_conv_y, assert_o

pytestmark = pytest.mark.gpu

SENTINEL = 3.0          # BF16-exact value left in output rows that must not be written


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from gated_deltanet_linear_build_gb300 import gdn
    return gdn


def same_bits(x, y):
    it = torch.int32 if x.dtype == torch.float32 else torch.int16
    return torch.equal(x.contiguous().view(it), y.contiguous().view(it))


def slot_map(seed, n, num_slots, pads):
    """Distinct slots for the n sequences, with the entries in ``pads`` made
    padding (alternately -1 and num_slots)."""
    rng = np.random.default_rng(seed)
    idx = rng.permutation(num_slots)[:n].astype(np.int32)
    for j, p in enumerate(pads):
        idx[p] = -1 if j % 2 == 0 else num_slots
    return idx


def gather(cache, idx):
    """Dense states of the batch: the slot's state, zeros for padding."""
    out = torch.zeros((len(idx),) + tuple(cache.shape[1:]), dtype=cache.dtype, device=cache.device)
    for n, s in enumerate(idx):
        if 0 <= s < cache.shape[0]:
            out[n] = cache[s]
    return out


def gather_np(cache, idx):
    """Host copy of the batch's states from the host cache (zeros for padding)."""
    out = np.zeros((len(idx),) + cache.shape[1:], dtype=cache.dtype)
    for n, s in enumerate(idx):
        if 0 <= s < cache.shape[0]:
            out[n] = cache[s]
    return out


def valid_entries(idx, num_slots):
    return [n for n, s in enumerate(idx) if 0 <= s < num_slots]


def check_cache(cache_after, cache_before, dense_after, idx):
    """Slots named by a valid entry hold the dense call's new state; every
    other slot keeps its bytes."""
    used = set()
    for n, s in enumerate(idx):
        if 0 <= s < cache_after.shape[0]:
            assert same_bits(cache_after[s], dense_after[n]), (n, s)
            used.add(int(s))
    for s in range(cache_after.shape[0]):
        if s not in used:
            assert same_bits(cache_after[s], cache_before[s]), s


def valid_rows(idx, num_slots, cu=None):
    """Token rows of the valid sequences (cu given) or the valid batch rows."""
    rows = []
    for n, s in enumerate(idx):
        if 0 <= s < num_slots:
            rows.extend(range(int(cu[n]), int(cu[n + 1])) if cu is not None else [n])
    return torch.tensor(rows, dtype=torch.long, device="cuda")


def pad_rows(idx, num_slots, cu=None):
    rows = []
    for n, s in enumerate(idx):
        if not 0 <= s < num_slots:
            rows.extend(range(int(cu[n]), int(cu[n + 1])) if cu is not None else [n])
    return torch.tensor(rows, dtype=torch.long, device="cuda")


@pytest.mark.parametrize("chunked", [True, False])
def test_conv_fwd_slots(G, chunked):
    lens = [203, 77, 1, 40, 9, 16]
    C, num_slots = 1024, 11
    case = synth.conv_case(81, lens, C, initial_state=True, bias=True)
    case["has_initial_state"][3] = 0
    cu_h = case["cu_seqlens"]
    T, N = case["x"].shape[0], len(lens)
    idx = slot_map(82, N, num_slots, pads=[2, 4])
    rng = np.random.default_rng(83)
    cache_h = synth.normal_bf16(rng, (num_slots, C, 3))
    cache0 = bf16_dev(cache_h)
    x, w, bias = bf16_dev(case["x"]), bf16_dev(case["w"]), bf16_dev(case["bias"])
    cu, has = dev(cu_h), dev(case["has_initial_state"])
    chunks = num = None
    if chunked:
        chunks = torch.empty((T // 8 + N, 4), dtype=torch.int32, device="cuda")
        num = torch.empty((1,), dtype=torch.int32, device="cuda")
        G.build_conv_chunks(cu, chunks, num, chunk_tokens=8)

    dense = gather(cache0, idx)
    y_d = torch.empty((T, C), dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_fwd(x, w, bias, dense, has, cu, y_d, chunks=chunks, num_chunks=num)

    cache = cache0.clone()
    y = torch.full((T, C), SENTINEL, dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_fwd_slots(x, w, bias, cache, has, cu, y, dev(idx), chunks=chunks,
                              num_chunks=num)
    torch.cuda.synchronize()
    vr, pr = valid_rows(idx, num_slots, cu_h), pad_rows(idx, num_slots, cu_h)
    assert same_bits(y[vr], y_d[vr])
    assert bool((y[pr].float() == SENTINEL).all())
    check_cache(cache, cache0, dense, idx)
    # the oracle on the gathered states
    yr, sr = O.causal_conv1d_fwd(case["x"], case["w"], case["bias"], gather_np(cache_h, idx),
                                 case["has_initial_state"], cu_h)
    vr_h = vr.cpu().numpy()
    assert_conv_y(bf16_values(y)[vr_h], yr[vr_h])
    for n in valid_entries(idx, num_slots):
        assert np.array_equal(bf16_host_bits(cache[int(idx[n])]), O.to_bf16(sr[n])), n


def test_conv_update_slots(G):
    C, N, num_slots = 1024, 9, 20
    case = synth.conv_update_case(84, N, C, bias=True)
    idx = slot_map(85, N, num_slots, pads=[0, 5])
    rng = np.random.default_rng(86)
    cache_h = synth.normal_bf16(rng, (num_slots, C, 3))
    cache0 = bf16_dev(cache_h)
    x, w, bias = bf16_dev(case["x"]), bf16_dev(case["w"]), bf16_dev(case["bias"])
    dense = gather(cache0, idx)
    y_d = torch.empty((N, C), dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_update(x, w, bias, dense, y_d)
    cache = cache0.clone()
    y = torch.full((N, C), SENTINEL, dtype=torch.bfloat16, device="cuda")
    G.causal_conv1d_update_slots(x, w, bias, cache, y, dev(idx))
    torch.cuda.synchronize()
    vr, pr = valid_rows(idx, num_slots), pad_rows(idx, num_slots)
    assert same_bits(y[vr], y_d[vr])
    assert bool((y[pr].float() == SENTINEL).all())
    check_cache(cache, cache0, dense, idx)
    yr, sr = O.causal_conv1d_update(case["x"], case["w"], case["bias"], gather_np(cache_h, idx))
    ok = valid_entries(idx, num_slots)
    assert_conv_y(bf16_values(y)[ok], yr[ok])
    for n in ok:
        assert np.array_equal(bf16_host_bits(cache[int(idx[n])]), O.to_bf16(sr[n])), n


@pytest.mark.parametrize("d,hk,hv", [(128, 4, 8), (64, 2, 4)])
def test_decode_slots(G, d, hk, hv):
    N, num_slots = 10, 23
    case = synth.delta_case(87 + d, [1] * N, hk, hv, d, d, normed_qk=False)
    idx = slot_map(88, N, num_slots, pads=[3, 9])
    rng = np.random.default_rng(89)
    cache_h = (0.02 * rng.standard_normal((num_slots, hv, d, d))).astype(np.float32)
    cache0 = dev(cache_h)
    q, k, v = bf16_dev(case["q"]), bf16_dev(case["k"]), bf16_dev(case["v"])
    a, b = dev(case["a"]), dev(case["b"])
    dense = gather(cache0, idx)
    o_d = torch.empty((N, hv, d), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_decode(q, k, v, a, b, dense, o_d, qk_l2norm=True)
    cache = cache0.clone()
    o = torch.full((N, hv, d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    G.delta_rule_decode_slots(q, k, v, a, b, cache, o, dev(idx), qk_l2norm=True)
    torch.cuda.synchronize()
    vr, pr = valid_rows(idx, num_slots), pad_rows(idx, num_slots)
    assert same_bits(o[vr], o_d[vr])
    assert bool((o[pr].float() == SENTINEL).all())
    check_cache(cache, cache0, dense, idx)
    o_r, S_r = O.delta_rule_decode(case["q"], case["k"], case["v"], case["a"], case["b"],
                                   gather_np(cache_h, idx), qk_l2norm=True)
    ok = valid_entries(idx, num_slots)
    assert_o(bf16_values(o)[ok], o_r[ok])
    assert_S(np.stack([cache[int(idx[n])].cpu().numpy() for n in ok]), S_r[ok])


@pytest.mark.parametrize("d,hk,hv", [(128, 4, 8), (64, 2, 4)])
def test_prefill_slots(G, d, hk, hv):
    lens = [150, 70, 1, 65, 33]
    N, num_slots = len(lens), 7
    case = synth.delta_case(90 + d, lens, hk, hv, d, d, s0_std=0.0)
    case["has_initial_state"][:] = 1
    case["has_initial_state"][1] = 0
    cu_h = case["cu_seqlens"]
    T = int(cu_h[-1])
    idx = slot_map(91, N, num_slots, pads=[3])
    rng = np.random.default_rng(92)
    cache_h = (0.05 * rng.standard_normal((num_slots, hv, d, d))).astype(np.float32)
    cache0 = dev(cache_h)
    q, k, v = bf16_dev(case["q"]), bf16_dev(case["k"]), bf16_dev(case["v"])
    a, b = dev(case["a"]), dev(case["b"])
    cu, has = dev(cu_h), dev(case["has_initial_state"])
    ws = torch.empty(G.delta_rule_prefill_workspace_size(T, N, hv, d, d), dtype=torch.uint8,
                     device="cuda")
    dense = gather(cache0, idx)
    o_d = torch.empty((T, hv, d), dtype=torch.bfloat16, device="cuda")
    G.delta_rule_prefill_chunked(q, k, v, a, b, cu, dense, has, o_d, ws)
    cache = cache0.clone()
    o = torch.full((T, hv, d), SENTINEL, dtype=torch.bfloat16, device="cuda")
    G.delta_rule_prefill_chunked_slots(q, k, v, a, b, cu, cache, has, o, ws, dev(idx))
    torch.cuda.synchronize()
    vr, pr = valid_rows(idx, num_slots, cu_h), pad_rows(idx, num_slots, cu_h)
    assert same_bits(o[vr], o_d[vr])
    assert bool((o[pr].float() == SENTINEL).all())
    check_cache(cache, cache0, dense, idx)
    o_r, S_r = O.delta_rule_prefill(case["q"], case["k"], case["v"], case["a"], case["b"], cu_h,
                                    gather_np(cache_h, idx), case["has_initial_state"])
    vr_h = vr.cpu().numpy()
    ok = valid_entries(idx, num_slots)
    assert_o(bf16_values(o)[vr_h], o_r[vr_h])
    assert_S(np.stack([cache[int(idx[n])].cpu().numpy() for n in ok]), S_r[ok])


def test_all_padding_touches_nothing(G):
    """num_slots = 0: every entry is padding; state and outputs keep their bytes."""
    N, C = 4, 1024
    case = synth.conv_update_case(93, N, C)
    rng = np.random.default_rng(94)
    cache0 = bf16_dev(synth.normal_bf16(rng, (2, C, 3)))
    cache = cache0.clone()
    y = torch.full((N, C), SENTINEL, dtype=torch.bfloat16, device="cuda")
    idx = dev(np.zeros(N, np.int32))
    G.causal_conv1d_update_slots(bf16_dev(case["x"]), bf16_dev(case["w"]), None, cache, y, idx,
                                 num_slots=0)
    torch.cuda.synchronize()
    assert same_bits(cache, cache0)
    assert bool((y.float() == SENTINEL).all())
