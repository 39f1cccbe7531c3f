"""Seeded synthetic inputs for the GDN hot path.

This module is the one place that both the CUDA path's callers (tests, bench)
and the CPU oracle's callers draw their inputs from. It holds none of the
method's arithmetic: it only draws random numbers, shapes them into the
distributions the workloads name, and stores them in the storage formats the
path consumes (BF16 bit patterns as ``uint16``, ``float32`` gates, ``int32``
offsets). It imports numpy only.

Workloads (sizes as the Qwen3.5-style serving mix on the pages fixes them:
"Qwen3.5-4b BF16 optimization and correctness", Evidence / Problem sections;
"RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT, and VRAM gaps", Problem):

* ``tiny``: two packed sequences of 5 and 13 tokens, 64 conv channels,
  delta rule with 2 heads of width 16.
* ``conv_prefill``: 2 x 1024 tokens, 8192 conv channels.
* ``decode``: 32 sequences x 1 token, 32 v-heads over 16 k-heads, d = 128.
* ``prefill``: 2 x 1024 tokens, chunk 64, 32 v-heads over 16 k-heads, d = 128.
"""
from __future__ import annotations

import numpy as np

# Channel split of the 8192-wide conv output of the Qwen3.5-4B-shaped GDN
# layer: q (16 heads x 128), k (16 heads x 128), v (32 heads x 128).
QK_HEADS = 16
V_HEADS = 32
HEAD_DIM = 128
CONV_CHANNELS = 2 * QK_HEADS * HEAD_DIM + V_HEADS * HEAD_DIM  # 8192
CONV_K = 4


def bf16_bits(x) -> np.ndarray:
    """Round float values to bfloat16 (round-to-nearest-even from float32).

    Returns the 16-bit patterns as ``uint16``. NaN stays NaN (quiet).
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounding_bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + rounding_bias) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r = np.where(nan, ((u >> 16) | 0x40).astype(np.uint16), r)
    return r


def bf16_to_f32(bits) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples stored as BF16 bits (std is the standard deviation)."""
    return bf16_bits(rng.standard_normal(shape, dtype=np.float64) * std)


def unit_rows_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """Random directions: Gaussian rows scaled to unit length, stored as BF16.

    This is how the workloads' "L2-normed q, k" inputs are drawn (uniform on the
    sphere). After BF16 rounding the norm is 1 within about 2^-8.
    """
    g = rng.standard_normal(shape, dtype=np.float64)
    g /= np.sqrt(np.sum(g * g, axis=-1, keepdims=True))
    return bf16_bits(g)


def gate_logits(rng: np.random.Generator, shape, shift_a: float = 0.0, scale: float = 1.0):
    """Raw gate logits (z_a, z_b) in float32: scale * N(0,1), z_a shifted by
    ``shift_a`` (a negative shift makes the decay exp(-softplus(z_a)) close to 1)."""
    z1 = rng.standard_normal(shape, dtype=np.float64) * scale + shift_a
    z2 = rng.standard_normal(shape, dtype=np.float64) * scale
    return z1.astype(np.float32), z2.astype(np.float32)


def gates(rng: np.random.Generator, shape):
    """Gate inputs as the workloads define them, in float32.

    a = exp(-softplus(z1)) in (0, 1) and b = sigmoid(z2) in (0, 1) with z1, z2
    standard normal.
    """
    z1 = rng.standard_normal(shape, dtype=np.float64)
    z2 = rng.standard_normal(shape, dtype=np.float64)
    a = np.exp(-np.logaddexp(0.0, z1))
    b = 1.0 / (1.0 + np.exp(-z2))
    return a.astype(np.float32), b.astype(np.float32)


def packed_lengths_cu(lengths) -> np.ndarray:
    """Offsets of packed sequences: cu[0] = 0, cu[s+1] = cu[s] + lengths[s]."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


# ----------------------------------------------------------------------------
# Conv workloads
# ----------------------------------------------------------------------------

def conv_case(seed: int, lengths, channels: int, *, initial_state=True,
              bias=False, w_std: float = 0.5):
    """Inputs of a varlen causal-conv prefill call.

    x ~ N(0,1) [T, C], w ~ N(0, w_std^2) [C, 4], bias zero unless ``bias``
    (then N(0, 0.1^2)), conv_state ~ N(0,1) [N, C, 3], has_initial_state all
    ones if ``initial_state`` else all zeros.
    """
    rng = np.random.default_rng(seed)
    cu = packed_lengths_cu(lengths)
    T, N = int(cu[-1]), len(lengths)
    x = normal_bf16(rng, (T, channels))
    w = normal_bf16(rng, (channels, CONV_K), std=w_std)
    b = normal_bf16(rng, (channels,), std=0.1) if bias else np.zeros(channels, np.uint16)
    st = normal_bf16(rng, (N, channels, CONV_K - 1))
    has = np.full(N, 1 if initial_state else 0, dtype=np.uint8)
    return dict(x=x, w=w, bias=b, conv_state=st, has_initial_state=has,
                cu_seqlens=cu, T=T, N=N, C=channels)


def conv_update_case(seed: int, n: int, channels: int, *, bias=False):
    """Inputs of one decode conv update: x [N, C], rolling state [N, C, 3]."""
    rng = np.random.default_rng(seed)
    x = normal_bf16(rng, (n, channels))
    w = normal_bf16(rng, (channels, CONV_K), std=0.5)
    b = normal_bf16(rng, (channels,), std=0.1) if bias else np.zeros(channels, np.uint16)
    st = normal_bf16(rng, (n, channels, CONV_K - 1))
    return dict(x=x, w=w, bias=b, conv_state=st, N=n, C=channels)


# ----------------------------------------------------------------------------
# Delta-rule workloads
# ----------------------------------------------------------------------------

def delta_case(seed: int, lengths, hk: int, hv: int, dk: int, dv: int, *,
               s0_std: float = 0.0, normed_qk: bool = True, initial_state=None):
    """Inputs of a delta-rule call over packed sequences.

    q, k [T, hk, dk] BF16 (unit rows when ``normed_qk``, else N(0,1)),
    v [T, hv, dv] BF16 N(0,1), gates a, b [T, hv] float32, initial state
    S0 [N, hv, dv, dk] float32 ~ N(0, s0_std^2) (zeros when s0_std == 0).
    ``initial_state`` defaults to "has state" exactly when s0_std > 0.
    """
    rng = np.random.default_rng(seed)
    cu = packed_lengths_cu(lengths)
    T, N = int(cu[-1]), len(lengths)
    if normed_qk:
        q = unit_rows_bf16(rng, (T, hk, dk))
        k = unit_rows_bf16(rng, (T, hk, dk))
    else:
        q = normal_bf16(rng, (T, hk, dk))
        k = normal_bf16(rng, (T, hk, dk))
    v = normal_bf16(rng, (T, hv, dv))
    a, b = gates(rng, (T, hv))
    if s0_std > 0:
        S0 = (rng.standard_normal((N, hv, dv, dk)) * s0_std).astype(np.float32)
    else:
        S0 = np.zeros((N, hv, dv, dk), np.float32)
    if initial_state is None:
        initial_state = s0_std > 0
    has = np.full(N, 1 if initial_state else 0, dtype=np.uint8)
    return dict(q=q, k=k, v=v, a=a, b=b, S0=S0, has_initial_state=has,
                cu_seqlens=cu, T=T, N=N, Hk=hk, Hv=hv, dk=dk, dv=dv)


# ----------------------------------------------------------------------------
# The named workloads
# ----------------------------------------------------------------------------

def tiny(seed: int = 0):
    """Two packed sequences (5 and 13 tokens), 64 channels, 2 heads of 16."""
    conv = conv_case(seed, [5, 13], 64, initial_state=True)
    delta = delta_case(seed + 100, [5, 13], 2, 2, 16, 16)
    return conv, delta


def conv_prefill(seed: int = 1):
    """2 x 1024 packed tokens over 8192 channels, fresh prompts (zero halo)."""
    return conv_case(seed, [1024, 1024], CONV_CHANNELS, initial_state=False)


def decode(seed: int = 2):
    """32 sequences x 1 token: conv update over 8192 channels, then the delta
    rule with 32 v-heads over 16 k-heads, d = 128, S ~ N(0, 0.02^2)."""
    conv = conv_update_case(seed, 32, CONV_CHANNELS)
    delta = delta_case(seed + 100, [1] * 32, QK_HEADS, V_HEADS, HEAD_DIM, HEAD_DIM,
                       s0_std=0.02)
    return conv, delta


def prefill(seed: int = 3):
    """2 x 1024 tokens, 32 v-heads over 16 k-heads, d = 128, S0 = 0."""
    return delta_case(seed, [1024, 1024], QK_HEADS, V_HEADS, HEAD_DIM, HEAD_DIM)


# ----------------------------------------------------------------------------
# Serving mix
# ----------------------------------------------------------------------------

SERVING_LAYERS = 24
SERVING_SEQS = 32
SERVING_STEP_TOKENS = 2048
SERVING_DECODE_STEPS = 128


def serving_mix_lengths(seed: int = 4, n: int = SERVING_SEQS, lo: int = 512, hi: int = 1024):
    """Prompt lengths of the serving mix: n integers uniform on [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


SERVING_VOCAB = 4096


def serving_stack(seed: int = 4, layers: int = SERVING_LAYERS, n_seqs: int = SERVING_SEQS,
                  vocab: int = SERVING_VOCAB, hk: int = QK_HEADS, hv: int = V_HEADS,
                  d: int = HEAD_DIM, len_lo: int = 512, len_hi: int = 1024):
    """Weights and prompts of the synthetic GDN stack used by the serving mix.

    embed [vocab, C] BF16 ~ N(0,1); per layer: conv taps [C, 4] BF16 ~ N(0, 0.5^2),
    gate projections u, r [hv, d] float32 ~ N(0,1), residual scales [C] float32 ~
    N(0, 0.5^2); head [C, vocab] BF16 ~ N(0, 1/C); prompts: lengths U[len_lo,
    len_hi] (seed ``seed``) and token ids U[0, vocab) (seed ``seed + 1000``).
    """
    C = 2 * hk * d + hv * d
    rng = np.random.default_rng(seed + 500)
    embed = normal_bf16(rng, (vocab, C))
    conv_w = [normal_bf16(rng, (C, CONV_K), std=0.5) for _ in range(layers)]
    gate_u = [rng.standard_normal((hv, d)).astype(np.float32) for _ in range(layers)]
    gate_r = [rng.standard_normal((hv, d)).astype(np.float32) for _ in range(layers)]
    res_scale = [(0.5 * rng.standard_normal(C)).astype(np.float32) for _ in range(layers)]
    head = normal_bf16(rng, (C, vocab), std=1.0 / np.sqrt(C))
    lengths = [int(x) for x in serving_mix_lengths(seed, n_seqs, len_lo, len_hi)]
    ids_rng = np.random.default_rng(seed + 1000)
    prompts = [ids_rng.integers(0, vocab, size=L).astype(np.int64) for L in lengths]
    return dict(embed=embed, conv_w=conv_w, gate_u=gate_u, gate_r=gate_r, res_scale=res_scale,
                head=head, prompts=prompts, lengths=lengths, layers=layers, hk=hk, hv=hv, d=d,
                C=C, vocab=vocab)
