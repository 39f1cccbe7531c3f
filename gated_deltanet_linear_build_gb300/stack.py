"""Engine-step executor for a stack of GDN token-mixer layers.

This is the host side of the hot path as the serving engine on the pages runs
it ("perf(gdn): dispatch exact causal-conv chunks", What changed; "RTX 5070 Ti:
close Qwen3.5-4B TTFT, TPOT, and VRAM gaps vs vLLM", Problem: 2048 batched
tokens per step, 32 concurrent sequences):

* a scheduler that packs prompts, in arrival order, into prefill steps of at
  most ``budget`` tokens (a prompt may be split across steps; its later part
  then continues from the carried conv_state and S);
* per prefill step: the exact 8-token conv descriptors and the chunked
  prefill's 64-token chunk plan are built ONCE and reused by every layer; per
  layer, the conv prefill over the descriptors and
  the chunked delta-rule prefill on q/k/v read in place from the conv output
  (q/k L2-normalised and the gates activated from their logits inside the
  kernel);
* per decode step: per layer, the conv update and the delta-rule decode.

Every step of the path runs in the CUDA library; this module only allocates
buffers (through PyTorch), slices them and calls the C ABI.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List

import torch

from . import gdn

# Kernels enqueued by one gdn_delta_rule_prefill_chunked call on a planned
# workspace (chunk kernel and state kernel); the plan itself is one more
# launch per engine step.
PREFILL_LAUNCHES = 2


@dataclass
class Segment:
    seq: int        # sequence slot
    start: int      # first prompt position of this segment
    length: int     # tokens in this step


@dataclass
class PrefillStep:
    segments: List[Segment] = field(default_factory=list)

    @property
    def tokens(self) -> int:
        return sum(s.length for s in self.segments)


def pack_prefill_steps(lengths, budget: int = 2048) -> List[PrefillStep]:
    """Pack prompts in order into steps of at most ``budget`` tokens.

    Greedy: fill the current step with the next unprocessed tokens of the
    current prompt; a prompt that does not fit is split and continues at the
    start of the next step.
    """
    steps: List[PrefillStep] = []
    cur = PrefillStep()
    room = budget
    for s, L in enumerate(lengths):
        pos = 0
        while pos < L:
            if room == 0:
                steps.append(cur)
                cur, room = PrefillStep(), budget
            take = min(room, L - pos)
            cur.segments.append(Segment(s, pos, take))
            pos += take
            room -= take
    if cur.segments:
        steps.append(cur)
    return steps


class GdnLayerStack:
    """Weights and carried states of ``layers`` GDN layers for ``n_seqs`` slots.

    Shapes follow the Qwen3.5-4B-style layer: conv over C = 2*Hk*d + Hv*d
    channels (q | k | v), Hk q/k heads and Hv v-heads of width d.
    Per layer: conv weights [C, 4] BF16, conv_state [n_seqs, C, 3] BF16 and
    S [n_seqs, Hv, d, d] float32. The conv weights are drawn N(0, w_std^2)
    from ``seed`` unless ``conv_weights`` (one [C, 4] tensor per layer) is
    given. With ``gate_logits`` (the default) the layers' gate inputs are the
    raw logits z_a, z_b and the delta-rule kernels compute a = exp(-softplus(z_a)),
    b = sigmoid(z_b) themselves; otherwise they are the activated gates.
    """

    def __init__(self, layers: int, n_seqs: int, *, hk: int = 16, hv: int = 32, d: int = 128,
                 max_step_tokens: int = 2048, device="cuda", seed: int = 0,
                 w_std: float = 0.5, conv_weights=None, gate_logits: bool = True):
        self.layers, self.n_seqs = layers, n_seqs
        self.hk, self.hv, self.d = hk, hv, d
        self.C = 2 * hk * d + hv * d
        self.device = torch.device(device)
        g = torch.Generator(device=self.device)
        g.manual_seed(seed)
        C = self.C
        if conv_weights is not None:
            assert len(conv_weights) == layers
            self.w = [w.to(device=self.device, dtype=torch.bfloat16).contiguous()
                      for w in conv_weights]
            assert all(tuple(w.shape) == (C, 4) for w in self.w)
        else:
            self.w = [(torch.randn((C, 4), generator=g, device=self.device) * w_std)
                      .to(torch.bfloat16) for _ in range(layers)]
        self.conv_state = [torch.zeros((n_seqs, C, 3), dtype=torch.bfloat16, device=self.device)
                           for _ in range(layers)]
        self.S = [torch.zeros((n_seqs, hv, d, d), dtype=torch.float32, device=self.device)
                  for _ in range(layers)]
        self.gate_logits = gate_logits
        self.max_step_tokens = max_step_tokens
        self.chunks = torch.empty((max_step_tokens // 8 + n_seqs, 4), dtype=torch.int32,
                                  device=self.device)
        self.num_chunks = torch.empty((1,), dtype=torch.int32, device=self.device)
        ws = gdn.delta_rule_prefill_workspace_size(max_step_tokens, n_seqs, hv, d, d)
        self.workspace = torch.empty((ws,), dtype=torch.uint8, device=self.device)
        self.launches = 0      # kernels enqueued so far (for the launch count)

    # -- views of the conv output ------------------------------------------
    def qkv(self, y):
        T, hk, hv, d = y.shape[0], self.hk, self.hv, self.d
        q = y[:, :hk * d].view(T, hk, d)
        k = y[:, hk * d:2 * hk * d].view(T, hk, d)
        v = y[:, 2 * hk * d:].view(T, hv, d)
        return q, k, v

    def step_meta(self, step: PrefillStep):
        """cu_seqlens, has_initial_state and first slot of a prefill step."""
        lens = [s.length for s in step.segments]
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        has = [1 if s.start > 0 else 0 for s in step.segments]
        slots = [s.seq for s in step.segments]
        assert slots == list(range(slots[0], slots[0] + len(slots))), "slots are contiguous"
        return cu, has, slots[0]

    # -- one call per kernel family -------------------------------------------
    def build_chunks(self, cu_d, T: int):
        """Exact 8-token conv descriptors and the chunked prefill's plan of one
        prefill step of T tokens (built once per step, reused by every layer)."""
        gdn.build_conv_chunks(cu_d, self.chunks, self.num_chunks, chunk_tokens=8)
        gdn.delta_rule_prefill_plan(cu_d, T, self.hv, self.d, self.d, self.workspace)
        self.launches += 2

    def conv_prefill_layer(self, l: int, cu_d, has_d, first_slot: int, n: int, x, y,
                           chunks=None, num_chunks=None):
        """Layer l's conv prefill over a step's descriptors (the stack's own
        buffer unless ``chunks``/``num_chunks`` are given)."""
        sl = slice(first_slot, first_slot + n)
        gdn.causal_conv1d_fwd(x, self.w[l], None, self.conv_state[l][sl], has_d, cu_d, y,
                              chunks=self.chunks if chunks is None else chunks,
                              num_chunks=self.num_chunks if num_chunks is None else num_chunks)
        self.launches += 1

    def delta_prefill_layer(self, l: int, cu_d, has_d, first_slot: int, n: int, y, a, b, out):
        """Layer l's chunked delta rule on q/k/v read in place from the conv output
        y, with the step's plan (build_chunks) already in the workspace."""
        sl = slice(first_slot, first_slot + n)
        q, k, v = self.qkv(y)
        gdn.delta_rule_prefill_chunked(q, k, v, a, b, cu_d, self.S[l][sl], has_d, out,
                                       self.workspace, qk_l2norm=True,
                                       gate_logits=self.gate_logits, planned=True)
        self.launches += PREFILL_LAUNCHES

    def conv_update_layer(self, l: int, x, y):
        gdn.causal_conv1d_update(x, self.w[l], None, self.conv_state[l], y)
        self.launches += 1

    def delta_decode_layer(self, l: int, y, a, b, out):
        q, k, v = self.qkv(y)
        gdn.delta_rule_decode(q, k, v, a, b, self.S[l], out, qk_l2norm=True,
                              gate_logits=self.gate_logits)
        self.launches += 1

    def prefill_layer(self, l: int, cu_d, has_d, first_slot: int, n: int, x, a, b, y, out,
                      tick=None):
        """Layer l of a prefill step: conv prefill over the step's descriptors,
        then the chunked delta rule on q/k/v read in place from the conv output."""
        tick = tick if tick is not None else (lambda kind, edge: None)
        tick("conv_prefill", "start")
        self.conv_prefill_layer(l, cu_d, has_d, first_slot, n, x, y)
        tick("conv_prefill", "end")
        tick("delta_prefill", "start")
        self.delta_prefill_layer(l, cu_d, has_d, first_slot, n, y, a, b, out)
        tick("delta_prefill", "end")

    def decode_layer(self, l: int, x, a, b, y, out, tick=None):
        """Layer l of a decode step: conv update, then the delta-rule decode."""
        tick = tick if tick is not None else (lambda kind, edge: None)
        tick("conv_update", "start")
        self.conv_update_layer(l, x, y)
        tick("conv_update", "end")
        tick("delta_decode", "start")
        self.delta_decode_layer(l, y, a, b, out)
        tick("delta_decode", "end")

    # -- whole engine steps over precomputed layer inputs ------------------------
    def prefill_step(self, cu_d, has_d, first_slot: int, n: int, xs, gates, ys, outs,
                     timer=None):
        """One prefill engine step over all layers.

        cu_d: int32 [n+1] on the device; has_d: uint8 [n]; xs[l]: BF16 [T, C]
        inputs; gates[l]: (a, b) float32 [T, Hv]; ys[l]: BF16 [T, C] conv
        outputs; outs[l]: BF16 [T, Hv, d] delta outputs. ``timer(kind, edge)``,
        if given, is called before ("start") and after ("end") every call.
        """
        tick = timer if timer is not None else (lambda kind, edge: None)
        tick("build_chunks", "start")
        self.build_chunks(cu_d, int(xs[0].shape[0]))
        tick("build_chunks", "end")
        for l in range(self.layers):
            a, b = gates[l]
            self.prefill_layer(l, cu_d, has_d, first_slot, n, xs[l], a, b, ys[l], outs[l], tick)

    def decode_step(self, xs, gates, ys, outs, timer=None):
        """One decode engine step (one token for every slot) over all layers."""
        for l in range(self.layers):
            a, b = gates[l]
            self.decode_layer(l, xs[l], a, b, ys[l], outs[l], timer)
