"""Writes linear_small.json: a small W8A8 linear (seeded synthetic input,
the video-projection recipe at M=4, K=32, N=8) with the oracle's codes,
scales and bf16 outputs.  Calls only the oracle and the seeded input
generator.  Run from the repository root:  python tests/golden/make_golden.py"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import w8a8_workloads as wl  # noqa: E402


def bits(t):
    return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)


def main():
    X, W, b = wl.make("video", M=4, N=8, K=32, seed=2024)
    xb, wb, bb = bits(X), bits(W), bits(b)
    wq, sw = oracle.quantize_rows(wb)
    xq, sx = oracle.quantize_rows(xb)
    ref = oracle.linear(xb, wq, sw, oracle.bf16_bits_to_f32(bb), exact_f64=True)
    out = {
        "what": "W8A8 linear, M=4 K=32 N=8, bf16 X, W, bias; video-projection recipe, seed 2024",
        "written_by": "tests/golden/make_golden.py (oracle only)",
        "X_bf16_bits": xb.tolist(), "W_bf16_bits": wb.tolist(), "bias_bf16_bits": bb.tolist(),
        "Xq": xq.tolist(), "sx_f32_bits": sx.view(np.uint32).tolist(),
        "Wq": wq.tolist(), "sw_f32_bits": sw.view(np.uint32).tolist(),
        "acc": oracle.gemm_s32_f64(xq, wq).tolist(),
        "Y_bf16_bits": ref["y"].tolist(),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "linear_small.json"), "w") as f:
        f.write("{\n" + ",\n".join("%s: %s" % (json.dumps(k), json.dumps(v)) for k, v in out.items()) + "\n}\n")


if __name__ == "__main__":
    main()
