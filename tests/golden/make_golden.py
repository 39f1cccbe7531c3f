"""Writes the oracle's results on the tiny workload to ``tiny_oracle.json``.

The stored values come from the CPU oracle only (inputs from the seeded
generators); they guard the oracle against silent drift between commits. Run
from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import gdn_oracle as O  # noqa: E402
from gated_deltanet_linear_build_gb300 import synth  # noqa: E402


def tiny_expectations():
    conv, d = synth.tiny(0)
    chunks = O.build_conv_chunks(conv["cu_seqlens"], 8)
    y, st = O.causal_conv1d_fwd(conv["x"], conv["w"], conv["bias"], conv["conv_state"],
                                conv["has_initial_state"], conv["cu_seqlens"])
    o, S = O.delta_rule_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["cu_seqlens"],
                                d["S0"], d["has_initial_state"])
    return {
        "source": "CPU oracle on the tiny workload (cu_seqlens [0,5,18], 64 channels, "
                  "2 heads of 16), seeds 0 and 100; written by tests/golden/make_golden.py",
        "chunks": chunks.tolist(),
        "conv_y_bf16": O.to_bf16(y).astype(int).tolist(),
        "conv_state_bf16": O.to_bf16(st).astype(int).tolist(),
        "delta_o_bf16": O.to_bf16(o).astype(int).tolist(),
        "delta_S_sum": float(S.sum()),
        "delta_S_abs_sum": float(abs(S).sum()),
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(out, "w") as f:
        json.dump(tiny_expectations(), f)
    print("wrote", out)
