"""Plain CPU oracle of the Gated DeltaNet (GDN) token-mixer hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, links or runs this
file: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do. It shares no code with the CUDA path.

Everything here is written from the definitions, in float64, with numpy as the
only library. Inputs that the CUDA path stores as BF16 are handed in as their
``uint16`` bit patterns and widened exactly; float32 inputs are widened to
float64. Outputs are float64 (BF16 rounding happens only where a function says
so). Loops run over tokens and sequences exactly as the definitions step; the
only vectorisation is over independent channels or heads.

The method (the pages are engineering records of a serving engine; the
formulas below are the computation they optimise, as the benchmark spec of the
Qwen3.5 GDN path fixes it):

* Exact chunk descriptors: one record per (sequence, 8-token chunk), built once
  per engine step ("perf(gdn): dispatch exact causal-conv chunks", What
  changed; "RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps",
  Existing evidence).
* Depthwise causal conv1d, width 4, SiLU, rolling conv_state, over packed
  varlen sequences ("perf(gdn): dispatch exact causal-conv chunks", What
  changed; "RTX 5070 Ti ...", Existing evidence: the K=4 specialisation).
* Gated delta rule  S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
  o_t = S_t q_t, with S of shape [dv, dk] ("RTX 5070 Ti ...", Existing
  evidence: fused decode, register-resident decode state).

Readings where the pages are silent (each listed in the design notes):
S is [dv][dk] with dk contiguous; v-head h reads q/k-head h // (Hv // Hk); no
1/sqrt(dk) scale on q; the optional q/k L2 norm is x / sqrt(sum x^2 + 1e-6);
a sequence without initial state starts from zeros (conv halo and S); a
zero-length sequence leaves its states untouched.
"""
from __future__ import annotations

import numpy as np

L2NORM_EPS = 1e-6


# ----------------------------------------------------------------------------
# BF16 storage format (IEEE binary32 with the low 16 mantissa bits dropped)
# ----------------------------------------------------------------------------

def from_bf16(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def to_bf16(x) -> np.ndarray:
    """Round to BF16 bit patterns, round-to-nearest-even, through float32.

    The value is first rounded to float32 (numpy's cast is round-to-nearest-
    even), then the low 16 bits of the float32 pattern are rounded off: add
    0x7FFF plus the lowest kept bit, then shift. NaN inputs give a quiet NaN.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    kept_lsb = (u >> np.uint64(16)) & np.uint64(1)
    out = ((u + np.uint64(0x7FFF) + kept_lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out = np.where(nan, ((u >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16), out)
    return out


def round_bf16(x) -> np.ndarray:
    """x rounded to the nearest BF16 value, returned as float64."""
    return from_bf16(to_bf16(x))


# ----------------------------------------------------------------------------
# a1: exact (sequence, chunk) descriptors
# ----------------------------------------------------------------------------

def build_conv_chunks(cu_seqlens, chunk_tokens: int = 8) -> np.ndarray:
    """Descriptors of the exact (sequence, chunk) dispatch.

    For every sequence s with L = cu[s+1] - cu[s] tokens and every chunk j in
    [0, ceil(L / chunk_tokens)): the record (seq=s, tok_start=cu[s] +
    j*chunk_tokens, len=min(chunk_tokens, L - j*chunk_tokens),
    pos_in_seq=j*chunk_tokens). Sequence-major, chunks ascending; an empty
    sequence contributes nothing. Returns int32 [count, 4].

    Source: "perf(gdn): dispatch exact causal-conv chunks", What changed (one
    descriptor per (sequence, 8-token chunk), built once per step).
    """
    cu = [int(c) for c in cu_seqlens]
    out = []
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        j = 0
        while j * chunk_tokens < L:
            out.append((s, cu[s] + j * chunk_tokens,
                        min(chunk_tokens, L - j * chunk_tokens), j * chunk_tokens))
            j += 1
    return np.asarray(out, dtype=np.int32).reshape(-1, 4)


# ----------------------------------------------------------------------------
# a2 / a3: depthwise causal conv1d with SiLU and a rolling state
# ----------------------------------------------------------------------------

def silu(x):
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x))."""
    return x / (1.0 + np.exp(-x))


def causal_conv1d_fwd(x_bits, w_bits, bias_bits, state_bits, has_initial_state,
                      cu_seqlens, apply_silu: bool = True):
    """Varlen depthwise causal conv1d over packed sequences.

    For sequence s (tokens cu[s] .. cu[s+1]-1), channel c, and local position
    i, with K = w.shape[1] taps and the window source
        xw(m) = x[cu[s] + m, c]                 for m >= 0,
        xw(m) = state[s, c, (K-1) + m]          for m < 0 (initial state),
        xw(m) = 0                               for m < 0 (no initial state):
        y[cu[s]+i, c] = SiLU(bias[c] + sum_{j=0}^{K-1} w[c, j] * xw(i-(K-1)+j)).
    The new state of s is the last K-1 entries of (initial state ++ x_s); an
    empty sequence keeps its state.

    Args: BF16 bit arrays x [T, C], w [C, K], bias [C] or None, state
    [N, C, K-1]; has_initial_state [N] (0/1) or None (all 0); cu_seqlens
    [N+1]. Returns (y float64 [T, C], new_state float64 [N, C, K-1]).
    """
    x = from_bf16(x_bits)
    w = from_bf16(w_bits)
    T, C = x.shape
    K = w.shape[1]
    state = from_bf16(state_bits).reshape(-1, C, K - 1)
    N = len(cu_seqlens) - 1
    bias = np.zeros(C) if bias_bits is None else from_bf16(bias_bits)
    if has_initial_state is None:
        has_initial_state = np.zeros(N, dtype=np.uint8)
    y = np.zeros((T, C))
    new_state = state.copy()
    for s in range(N):
        start, end = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        if end == start:
            continue
        init = state[s] if has_initial_state[s] else np.zeros((C, K - 1))
        # ext[(K-1) + m] = xw(m) for m in [-(K-1), L)
        ext = np.concatenate([init.T, x[start:end]], axis=0)
        for i in range(end - start):
            acc = bias.copy()
            for j in range(K):
                acc = acc + w[:, j] * ext[i + j]
            y[start + i] = silu(acc) if apply_silu else acc
        new_state[s] = ext[-(K - 1):].T
    return y, new_state


def causal_conv1d_update(x_bits, w_bits, bias_bits, state_bits, apply_silu: bool = True):
    """One decode step of the conv for N sequences, one token each.

    The window is (state[n, c, 0], ..., state[n, c, K-2], x[n, c]);
    y[n, c] = SiLU(bias[c] + sum_j w[c, j] * window_j); the state rolls to
    (state[n, c, 1], ..., x[n, c]).

    Returns (y float64 [N, C], new_state float64 [N, C, K-1]).
    """
    x = from_bf16(x_bits)
    w = from_bf16(w_bits)
    N, C = x.shape
    K = w.shape[1]
    state = from_bf16(state_bits).reshape(N, C, K - 1)
    bias = np.zeros(C) if bias_bits is None else from_bf16(bias_bits)
    window = np.concatenate([state, x[:, :, None]], axis=2)  # [N, C, K]
    acc = np.broadcast_to(bias, (N, C)).copy()
    for j in range(K):
        acc = acc + w[None, :, j] * window[:, :, j]
    y = silu(acc) if apply_silu else acc
    return y, window[:, :, 1:].copy()


# ----------------------------------------------------------------------------
# a4: q/k L2 normalisation
# ----------------------------------------------------------------------------

def l2norm(x, eps: float = L2NORM_EPS):
    """x / sqrt(sum(x^2) + eps) over the last axis."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gate_activation(z_a, z_b):
    """Decay and write strength from raw gate logits (float64):
        a = exp(-softplus(z_a)) = 1 / (1 + e^{z_a}),   b = sigmoid(z_b) = 1 / (1 + e^{-z_b}),
    softplus(z) = log(1 + e^z) taken as logaddexp(0, z) so that large z does
    not overflow. The GDN gate prep between the conv and the recurrence
    ("RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM",
    Existing evidence: the post-conv tile).
    """
    z_a = np.asarray(z_a, np.float64)
    z_b = np.asarray(z_b, np.float64)
    a = np.exp(-np.logaddexp(0.0, z_a))
    b = np.exp(-np.logaddexp(0.0, -z_b))
    return a, b


def _head_map(hk: int, hv: int) -> np.ndarray:
    """q/k-head read by each v-head: contiguous groups of hv // hk v-heads."""
    return np.arange(hv) // (hv // hk)


# ----------------------------------------------------------------------------
# a5 / prefill: the gated delta rule, one token at a time
# ----------------------------------------------------------------------------

def delta_rule_step_literal(S, q, k, v, a, b):
    """One token of the gated delta rule, written as the matrix product.

    S [H, dv, dk], q/k [H, dk], v [H, dv], a/b [H]:
        S_new = a S (I - b k k^T) + b v k^T,   o = S_new q.
    O(dk^3) per head; used on small cases and to pin ``delta_rule_step``.
    """
    dk = k.shape[-1]
    eye = np.eye(dk)[None]
    P = eye - b[:, None, None] * k[:, :, None] * k[:, None, :]
    S_new = a[:, None, None] * (S @ P) + b[:, None, None] * v[:, :, None] * k[:, None, :]
    o = np.einsum("hij,hj->hi", S_new, q)
    return o, S_new


def delta_rule_step(S, q, k, v, a, b):
    """One token of the gated delta rule with the product expanded.

    S (I - b k k^T) = S - b (S k) k^T, so
        S_new = a S - a b (S k) k^T + b v k^T,   o = S_new q.
    Same value as ``delta_rule_step_literal`` up to rounding order, O(dv dk).
    """
    Sk = np.einsum("hij,hj->hi", S, k)
    S_new = (a[:, None, None] * S
             - (a * b)[:, None, None] * Sk[:, :, None] * k[:, None, :]
             + b[:, None, None] * v[:, :, None] * k[:, None, :])
    o = np.einsum("hij,hj->hi", S_new, q)
    return o, S_new


def _prep_qk(q_bits, k_bits, qk_l2norm):
    q = from_bf16(q_bits)
    k = from_bf16(k_bits)
    if qk_l2norm:
        q, k = l2norm(q), l2norm(k)
    return q, k


def delta_rule_decode(q_bits, k_bits, v_bits, a, b, S, qk_l2norm: bool = False,
                      literal: bool = False):
    """One decode token per sequence.

    q, k: BF16 bits [N, Hk, dk]; v: BF16 bits [N, Hv, dv]; a, b [N, Hv];
    S [N, Hv, dv, dk] (float32 or float64). Returns (o [N, Hv, dv],
    S_new [N, Hv, dv, dk]), both float64.
    """
    q, k = _prep_qk(q_bits, k_bits, qk_l2norm)
    v = from_bf16(v_bits)
    N, Hv = v.shape[0], v.shape[1]
    hmap = _head_map(q.shape[1], Hv)
    step = delta_rule_step_literal if literal else delta_rule_step
    S = np.asarray(S, dtype=np.float64)
    o = np.zeros(v.shape)
    S_new = np.empty_like(S)
    for n in range(N):
        o[n], S_new[n] = step(S[n], q[n, hmap], k[n, hmap], v[n],
                              np.asarray(a[n], np.float64), np.asarray(b[n], np.float64))
    return o, S_new


def delta_rule_prefill(q_bits, k_bits, v_bits, a, b, cu_seqlens, S0,
                       has_initial_state=None, qk_l2norm: bool = False,
                       literal: bool = False, heads=None):
    """The gated delta rule over packed sequences, token by token.

    q, k: BF16 bits [T, Hk, dk]; v: BF16 bits [T, Hv, dv]; a, b [T, Hv];
    S0 [N, Hv, dv, dk] (used where has_initial_state[s] is set, else zeros).
    ``heads`` restricts the work to a subset of v-heads (others are left as
    zeros in o and as S0 in S). Returns (o [T, Hv, dv], S_final [N, Hv, dv,
    dk]), float64. An empty sequence keeps S0 as its final state.
    """
    q, k = _prep_qk(q_bits, k_bits, qk_l2norm)
    v = from_bf16(v_bits)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    T, Hv, dv = v.shape
    dk = q.shape[-1]
    N = len(cu_seqlens) - 1
    hmap = _head_map(q.shape[1], Hv)
    hs = np.arange(Hv) if heads is None else np.asarray(heads)
    step = delta_rule_step_literal if literal else delta_rule_step
    S0 = np.asarray(S0, dtype=np.float64).reshape(N, Hv, dv, dk)
    if has_initial_state is None:
        has_initial_state = np.zeros(N, dtype=np.uint8)
    o = np.zeros((T, Hv, dv))
    S_final = S0.copy()
    for s in range(N):
        start, end = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        if end == start:
            continue
        S = S0[s, hs].copy() if has_initial_state[s] else np.zeros((len(hs), dv, dk))
        for t in range(start, end):
            o[t, hs], S = step(S, q[t, hmap[hs]], k[t, hmap[hs]], v[t, hs], a[t, hs], b[t, hs])
        S_final[s, hs] = S
    return o, S_final


# ----------------------------------------------------------------------------
# Chunked (WY / UT) form of the same recurrence -- used only to check, in
# float64, that the chunked algorithm reaches the sequential result.
# ----------------------------------------------------------------------------

def delta_rule_prefill_chunked(q_bits, k_bits, v_bits, a, b, cu_seqlens, S0,
                               has_initial_state=None, qk_l2norm: bool = False,
                               chunk: int = 64):
    """Chunkwise evaluation of the gated delta rule (one (seq, head) at a time).

    Within a chunk of C tokens r = 0..C-1 entering with state S0, with
    gamma_r = prod_{s<=r} a_s:
      u_r := b_r (v_r - a_r S_{r-1} k_r) so that S_r = a_r S_{r-1} + u_r k_r^T;
      A_rs = b_r (gamma_r / gamma_s) (k_r . k_s) for s < r (strictly lower);
      (I + A) Delta = diag(b) V - diag(b gamma) K S0^T, i.e. with
      Tm = (I + A)^{-1}, W = Tm diag(b gamma) K and U = Tm diag(b) V:
      Delta = U - W S0^T;
      O = diag(gamma) Q S0^T + (M o Q K^T) Delta with M_rs = gamma_r / gamma_s
      for s <= r, else 0;
      S_C = gamma_C S0 + Delta^T diag(gamma_C / gamma) K.
    Chunks start at each sequence's first token and never cross sequences.
    Tm is the explicit inverse of the unit lower-triangular (I + A).
    """
    q, k = _prep_qk(q_bits, k_bits, qk_l2norm)
    v = from_bf16(v_bits)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    T, Hv, dv = v.shape
    dk = q.shape[-1]
    N = len(cu_seqlens) - 1
    hmap = _head_map(q.shape[1], Hv)
    S0 = np.asarray(S0, dtype=np.float64).reshape(N, Hv, dv, dk)
    if has_initial_state is None:
        has_initial_state = np.zeros(N, dtype=np.uint8)
    o = np.zeros((T, Hv, dv))
    S_final = S0.copy()
    for s in range(N):
        start, end = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        if end == start:
            continue
        for h in range(Hv):
            S = S0[s, h].copy() if has_initial_state[s] else np.zeros((dv, dk))
            for c0 in range(start, end, chunk):
                c1 = min(c0 + chunk, end)
                Q = q[c0:c1, hmap[h]]
                Kc = k[c0:c1, hmap[h]]
                V = v[c0:c1, h]
                bc = b[c0:c1, h]
                gamma = np.cumprod(a[c0:c1, h])
                n = c1 - c0
                ratio = gamma[:, None] / gamma[None, :]          # gamma_r / gamma_s
                A = np.tril(bc[:, None] * ratio * (Kc @ Kc.T), -1)
                Tm = np.linalg.inv(np.eye(n) + A)
                W = Tm @ ((bc * gamma)[:, None] * Kc)
                U = Tm @ (bc[:, None] * V)
                Delta = U - W @ S.T
                M = np.tril(ratio)
                o[c0:c1, h] = gamma[:, None] * (Q @ S.T) + (M * (Q @ Kc.T)) @ Delta
                S = gamma[-1] * S + Delta.T @ ((gamma[-1] / gamma)[:, None] * Kc)
            S_final[s, h] = S
    return o, S_final


# ----------------------------------------------------------------------------
# Comparison metrics used by the parity checks
# ----------------------------------------------------------------------------

def rel_err(x, ref) -> float:
    """max |x - ref| / max |ref| over the tensor (0 when both are all zero).

    Both maxima are of absolute values, and the denominator is the
    reference's, not the candidate's. When the reference is all zero the
    absolute error max |x| is returned.
    """
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(x - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def rel_err_slices(x, ref, slice_ndim: int, floor: float = 0.0) -> float:
    """The largest ``rel_err`` over the slices formed by the last ``slice_ndim``
    axes (one slice per index of the leading axes).

    Each slice is measured against its own scale max |ref_slice|, floored at
    ``floor`` times the scale of the whole tensor, so that a slice whose
    reference is (nearly) zero is measured against the tensor's magnitude
    instead of being divided by zero. With ``floor = 0`` a slice whose
    reference is all zero contributes its absolute error, as ``rel_err``.
    Used with one output row per (token, head) and one state per
    (sequence, head), so that a small-magnitude head cannot hide behind a
    large one.
    """
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    lead = ref.shape[:ref.ndim - slice_ndim]
    n = int(np.prod(lead)) if lead else 1
    xs = x.reshape(n, -1)
    rs = ref.reshape(n, -1)
    num = np.max(np.abs(xs - rs), axis=1)
    den = np.max(np.abs(rs), axis=1)
    den = np.maximum(den, floor * float(np.max(np.abs(rs))))
    out = np.where(den > 0.0, num / np.where(den > 0.0, den, 1.0), num)
    return float(np.max(out))


# ----------------------------------------------------------------------------
# The synthetic GDN stack of the serving mix (greedy generation, one sequence)
# ----------------------------------------------------------------------------
#
# Readings (the pages name the model -- a Qwen3.5-style hybrid -- but give no
# definition of a synthetic stack): a residual stream h (float32 storage); per
# layer x = bf16(h / sqrt(mean(h^2) + 1e-6)); the conv over x (BF16 output);
# q, k, v split from it, q and k L2-normalised inside the delta rule; gates
# a = exp(-softplus(u_h . x_v[h] / sqrt(d))) and b = sigmoid(r_h . x_v[h] /
# sqrt(d)) from the pre-conv v slice of head h, stored as float32; the delta
# rule's BF16 output o; h <- h + s * [o, o] (the 4096-wide output repeated to
# the 8192-wide stream). Head: logits = bf16(rms-normalised h) . W, argmax
# with the lowest index winning ties. The first generated token comes from the
# last prompt position; each decode step consumes the previous token.

RMS_EPS = 1e-6


def rms_norm_bf16(h):
    """BF16 bit patterns of h / sqrt(mean(h^2) + 1e-6), row by row."""
    h = np.asarray(h, np.float64)
    return to_bf16(h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + RMS_EPS))


def _gate_logits(x_vals, u, r, hk, hv, d):
    """Gate logits of the synthetic stack: z_a[h] = u_h . x_v[h] / sqrt(d) and
    z_b[h] = r_h . x_v[h] / sqrt(d), with x_v[h] the pre-conv v slice of head h."""
    xv = x_vals[:, 2 * hk * d:].reshape(-1, hv, d)
    za = np.einsum("lhd,hd->lh", xv, np.asarray(u, np.float64)) / np.sqrt(d)
    zb = np.einsum("lhd,hd->lh", xv, np.asarray(r, np.float64)) / np.sqrt(d)
    return za, zb


def _gates(x_vals, u, r, hk, hv, d):
    za, zb = _gate_logits(x_vals, u, r, hk, hv, d)
    a, b = gate_activation(za, zb)
    return a.astype(np.float32), b.astype(np.float32)


def _stack_layer(stack, l, h, carry, first: bool):
    """Layer l of the synthetic stack on rows h [T, C] of ONE sequence.

    first: the rows are the whole prompt (conv prefill and the delta rule token
    by token from zero state); otherwise h holds one decode token. carry["conv"][l] and
    carry["S"][l] are read and replaced. Returns the new residual stream rows.
    """
    hk, hv, d = stack["hk"], stack["hv"], stack["d"]
    T = h.shape[0]
    xb = rms_norm_bf16(h)
    a, b = _gates(from_bf16(xb), stack["gate_u"][l], stack["gate_r"][l], hk, hv, d)
    if first:
        y, st = causal_conv1d_fwd(xb, stack["conv_w"][l], None, carry["conv"][l], [0], [0, T])
    else:
        y, st = causal_conv1d_update(xb, stack["conv_w"][l], None, carry["conv"][l])
    carry["conv"][l] = to_bf16(st)
    yb = to_bf16(y)
    q = yb[:, :hk * d].reshape(T, hk, d)
    k = yb[:, hk * d:2 * hk * d].reshape(T, hk, d)
    v = yb[:, 2 * hk * d:].reshape(T, hv, d)
    if first:
        o, carry["S"][l] = delta_rule_prefill(q, k, v, a, b, [0, T], carry["S"][l], [0],
                                              qk_l2norm=True)
    else:
        o, carry["S"][l] = delta_rule_decode(q, k, v, a, b, carry["S"][l], qk_l2norm=True)
    ob = round_bf16(o).reshape(T, hv * d)
    return h + np.asarray(stack["res_scale"][l], np.float64) * np.concatenate([ob, ob], axis=1)


def _new_carry(stack):
    C, hv, d = stack["C"], stack["hv"], stack["d"]
    return dict(conv=[np.zeros((1, C, 3), np.uint16) for _ in range(stack["layers"])],
                S=[np.zeros((1, hv, d, d)) for _ in range(stack["layers"])])


def stack_logits(stack, h_rows):
    """Head logits of residual rows: bf16(rms-normalised h) . W (float64)."""
    return from_bf16(rms_norm_bf16(h_rows)) @ from_bf16(stack["head"])


def serving_stack_sequence(stack, s: int, n_decode: int = 128):
    """Greedy generation of sequence s through the synthetic stack.

    Prompt: ``stack["prompts"][s]``; returns (ids, margins, logits_rows): the
    n_decode + 1 generated ids, the top-1 minus top-2 logit margin at each, and
    the logits rows (float64). The prompt goes through each layer at once, the
    delta rule token by token (the sequential recurrence, the definition);
    decode steps use the single-token forms.
    """
    embed = from_bf16(stack["embed"])
    carry = _new_carry(stack)
    h = embed[np.asarray(stack["prompts"][s])]
    for l in range(stack["layers"]):
        h = _stack_layer(stack, l, h, carry, True)
    ids, margins, rows = [], [], []
    lg = stack_logits(stack, h[-1:])[0]
    for step in range(n_decode + 1):
        top = int(np.argmax(lg))       # first index of the maximum
        srt = np.sort(lg)
        ids.append(top)
        margins.append(float(srt[-1] - srt[-2]))
        rows.append(lg)
        if step == n_decode:
            break
        h = embed[[top]]
        for l in range(stack["layers"]):
            h = _stack_layer(stack, l, h, carry, False)
        lg = stack_logits(stack, h)[0]
    return ids, margins, np.asarray(rows)


def serving_stack_prefill_logits(stack, tokens):
    """Logits at every position of ``tokens`` run through the stack as one prompt."""
    carry = _new_carry(stack)
    h = from_bf16(stack["embed"])[np.asarray(tokens)]
    for l in range(stack["layers"]):
        h = _stack_layer(stack, l, h, carry, True)
    return stack_logits(stack, h)
