"""Write ``oracle_small_cases.json``: stored inputs and oracle outputs of two
small layer-core cases, a fixed record of what the oracle computes.

The pages print no worked example with numbers, so every stored expected
value here comes from the oracle (``oracle/``) and from nothing else; the
inputs come from the seeded recipe (``mamba_selective_scan_gb300.inputs``).
``tests/test_golden_oracle.py`` re-runs the oracle on the stored inputs and
compares: any later change to the oracle's arithmetic shows up there and has
to be justified by the passage it follows before this file is regenerated.

What the stored values follow (mamba-rs docs.rs source pages):
  forward -- mamba-rs 0.3.1 ``src/mamba_ssm/gpu/forward_mixed.rs``, the
    per-layer loop of ``gpu_forward_mamba_backbone_mixed``: F4a conv1d and
    SiLU, F4c softplus of delta_raw plus dt_bias, F4d the selective scan
    with the D skip, F4e gated = y * silu(z); A = -exp(a_log) and the zero
    initial state from mamba-rs 0.7.3 ``src/mamba_ssm/gpu/trainer.rs``
    (``recompute_a_neg_all``, ``reset_state``).
  backward -- the gradients the same forward page's
    ``GpuMambaMixedTrainScratch`` lists (d_delta, d_u, d_B, d_C reduced over
    d_inner, d_D, d_a_log, softplus and conv1d backward), as the exact
    derivative of L = sum(gated * d_gated).

Run from the repository root: ``python tests/golden/make_oracle_golden.py``.
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mamba_selective_scan_gb300.inputs import make_inputs  # noqa: E402

OUT = os.path.join(HERE, "oracle_small_cases.json")

# (name, batch, seq_len, d_inner, act, seed, random_params, chunk of the backward)
CASES = [
    ("f32_b1_t6_d2_random_params", 1, 6, 2, "f32", 11, True, 0),
    ("bf16_b2_t4_d2_recipe_params_chunk2", 2, 4, 2, "bf16", 12, False, 2),
]
INPUT_KEYS = ("x", "delta_raw", "z", "B", "C", "d_gated", "conv_w", "conv_b", "dt_bias",
              "a_log", "D")


def _arr(a):
    """An array as its shape and its values in row-major order (exact float64 repr)."""
    a = np.asarray(a, dtype=np.float64)
    return {"shape": list(a.shape), "data": [float(v) for v in a.ravel()]}


def _case(name, batch, T, D, act, seed, random_params, chunk):
    inp = make_inputs(batch, T, D, act=act, seed=seed, random_params=random_params)
    f = oracle.forward(inp)
    g = oracle.backward(inp, chunk=chunk)
    return {
        "name": name,
        "shape": {"batch": batch, "seq_len": T, "d_inner": D, "d_state": inp.d_state,
                  "d_conv": inp.d_conv},
        "act": act,
        "seed": seed,
        "random_params": random_params,
        "chunk": chunk,
        "inputs": {k: _arr(inp[k]) for k in INPUT_KEYS},
        "forward": {k: _arr(f[k]) for k in ("gated", "y", "u", "delta", "ssm_state_out")},
        "backward": {k: _arr(g[k]) for k in oracle.GRAD_NAMES},
    }


def main():
    doc = {
        "about": "inputs and float64 oracle outputs of small Mamba-1 layer-core cases; "
                 "written by tests/golden/make_oracle_golden.py from oracle/ only",
        "cases": [_case(*c) for c in CASES],
    }
    # one array per line
    text = json.dumps(doc, separators=(",", ":"))
    text = text.replace('{"shape":', '\n{"shape":')
    with open(OUT, "w", encoding="utf-8") as fh:
        fh.write(text + "\n")
    print("wrote", OUT)


if __name__ == "__main__":
    main()
