"""Greedy generation through a stack of synthetic GDN layers.

The serving mix the pages measure ("RTX 5070 Ti: close Qwen3.5-4B TTFT, TPOT,
and VRAM gaps vs vLLM", Problem: 32 concurrent sequences, 2048 batched tokens
per step) runs whole models; here the model around the GDN token mixer is a
synthetic one, the same for every layer:

    x = bf16(h / sqrt(mean(h^2) + 1e-6))                       (per token)
    a = exp(-softplus(u_h . x_v[h] / sqrt(d))),  b = sigmoid(r_h . x_v[h] / sqrt(d))
                                             (activated inside the delta-rule kernels)
    y = causal conv1d + SiLU of x (BF16);   q | k | v = y
    o = gated delta rule (q, k L2-normalised; BF16 output)
    h = h + s * [o, o]                       (o repeated to the stream width)

with x_v[h] the slice of x that feeds v-head h, and a head
logits = bf16(rms-normalised h) . W, argmax with the lowest index on ties.

The conv and the delta rule run in the CUDA library through ``GdnLayerStack``;
the glue above (norms, gates, residual, embedding, head) is plain PyTorch on
the device: it is the model around the token mixer, not part of it.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .stack import GdnLayerStack, pack_prefill_steps

RMS_EPS = 1e-6


def _bf16(bits, device):
    """BF16 bit patterns (uint16 numpy) as a BF16 tensor on ``device``."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def _rms_bf16(h):
    return (h * torch.rsqrt(h.pow(2).mean(dim=-1, keepdim=True) + RMS_EPS)).to(torch.bfloat16)


class SyntheticServingStack:
    """The synthetic stack on one GPU, with state slots for every sequence.

    ``weights`` holds numpy arrays: embed [V, C] and head [C, V] (BF16 bits),
    conv_w[l] [C, 4] (BF16 bits), gate_u[l], gate_r[l] [Hv, d] and
    res_scale[l] [C] (float32), prompts (token id arrays), and the sizes
    layers, hk, hv, d, C, vocab.
    """

    def __init__(self, weights, device="cuda", budget: int = 2048):
        dev = torch.device(device)
        self.device = dev
        self.layers = int(weights["layers"])
        self.hk, self.hv, self.d = int(weights["hk"]), int(weights["hv"]), int(weights["d"])
        self.C, self.vocab = int(weights["C"]), int(weights["vocab"])
        self.prompts = [np.asarray(p, np.int64) for p in weights["prompts"]]
        self.n_seqs = len(self.prompts)
        self.budget = budget
        self.embed = _bf16(weights["embed"], dev)
        self.head = _bf16(weights["head"], dev).float()
        self.gate_u = torch.stack([torch.from_numpy(np.asarray(u, np.float32))
                                   for u in weights["gate_u"]]).to(dev)
        self.gate_r = torch.stack([torch.from_numpy(np.asarray(r, np.float32))
                                   for r in weights["gate_r"]]).to(dev)
        self.res_scale = torch.stack([torch.from_numpy(np.asarray(s, np.float32))
                                      for s in weights["res_scale"]]).to(dev)
        self.conv_w = [_bf16(w, dev) for w in weights["conv_w"]]

    def _gates(self, l, x):
        """Gate logits z_a, z_b (the projections of the model glue); the
        delta-rule kernels turn them into a = exp(-softplus(z_a)) and
        b = sigmoid(z_b)."""
        T = x.shape[0]
        xv = x[:, 2 * self.hk * self.d:].float().reshape(T, self.hv, self.d)
        scale = 1.0 / math.sqrt(self.d)
        za = ((xv * self.gate_u[l]).sum(-1) * scale).contiguous()
        zb = ((xv * self.gate_r[l]).sum(-1) * scale).contiguous()
        return za, zb

    def _residual(self, l, h, o):
        o2 = o.reshape(o.shape[0], -1).float()
        return h + self.res_scale[l] * torch.cat([o2, o2], dim=1)

    def _logits(self, h_rows):
        return _rms_bf16(h_rows).float() @ self.head

    @torch.no_grad()
    def generate(self, n_decode: int = 128, forced=None, keep_logits=()):
        """Prefill every prompt in steps of at most ``budget`` tokens, then run
        ``n_decode`` decode steps over all sequences.

        Returns (ids [n_seqs, n_decode + 1] int64, {s: logits [n_decode + 1, V]}
        for s in ``keep_logits``). ``forced`` maps a sequence to the ids it is
        fed during decode (teacher forcing: at step t it consumes forced[s][t]
        instead of its own previous argmax); other sequences run free.
        """
        dev, C = self.device, self.C
        forced = forced or {}
        lengths = [len(p) for p in self.prompts]
        stack = GdnLayerStack(self.layers, self.n_seqs, hk=self.hk, hv=self.hv, d=self.d,
                              max_step_tokens=self.budget, device=dev,
                              conv_weights=self.conv_w)
        n_out = n_decode + 1
        ids = torch.zeros((self.n_seqs, n_out), dtype=torch.int64, device=dev)
        kept = {s: [] for s in keep_logits}

        for step in pack_prefill_steps(lengths, self.budget):
            cu, has, first = stack.step_meta(step)
            n, T = len(step.segments), cu[-1]
            toks = np.concatenate([self.prompts[sg.seq][sg.start:sg.start + sg.length]
                                   for sg in step.segments])
            cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
            has_d = torch.tensor(has, dtype=torch.uint8, device=dev)
            h = self.embed[torch.from_numpy(toks).to(dev)].float()
            y = torch.empty((T, C), dtype=torch.bfloat16, device=dev)
            o = torch.empty((T, self.hv, self.d), dtype=torch.bfloat16, device=dev)
            stack.build_chunks(cu_d, T)
            for l in range(self.layers):
                x = _rms_bf16(h).contiguous()
                a, b = self._gates(l, x)
                stack.prefill_layer(l, cu_d, has_d, first, n, x, a, b, y, o)
                h = self._residual(l, h, o)
            for i, sg in enumerate(step.segments):
                if sg.start + sg.length == lengths[sg.seq]:
                    lg = self._logits(h[cu[i + 1] - 1:cu[i + 1]])[0]
                    ids[sg.seq, 0] = torch.argmax(lg)
                    if sg.seq in kept:
                        kept[sg.seq].append(lg)

        N = self.n_seqs
        forced_rows = torch.tensor(sorted(forced), dtype=torch.int64, device=dev)
        forced_ids = (torch.tensor(np.stack([np.asarray(forced[s][:n_out]) for s in sorted(forced)]),
                                   dtype=torch.int64, device=dev) if forced else None)
        y = torch.empty((N, C), dtype=torch.bfloat16, device=dev)
        o = torch.empty((N, self.hv, self.d), dtype=torch.bfloat16, device=dev)
        for t in range(n_decode):
            cur = ids[:, t].clone()
            if forced:
                cur[forced_rows] = forced_ids[:, t]
            h = self.embed[cur].float()
            for l in range(self.layers):
                x = _rms_bf16(h).contiguous()
                a, b = self._gates(l, x)
                stack.decode_layer(l, x, a, b, y, o)
                h = self._residual(l, h, o)
            lg = self._logits(h)
            ids[:, t + 1] = torch.argmax(lg, dim=1)
            for s in kept:
                kept[s].append(lg[s])
        logits = {s: torch.stack(v).double().cpu().numpy() for s, v in kept.items()}
        return ids.cpu().numpy(), logits
