"""Writes tests/golden/nf4_oracle_small.json from the CPU oracle alone.

The input is a closed-form rational pattern (no random generator, no libm), so it
is identical on every machine; the stored values pin the oracle's results across
machines and compilers.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import codebooks  # noqa: E402

N, K, M = 16, 192, 5


def pattern_weight():
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    num = ((n * 37 + k * 101 + (n * k) % 13) % 1009 - 504).astype(np.float32)
    return num / np.float32(504.0) * np.float32(0.05)


def pattern_x():
    m = np.arange(M)[:, None]
    k = np.arange(K)[None, :]
    num = ((m * 53 + k * 29) % 31 - 15).astype(np.float32)
    return oracle.f32_to_bf16_bits(num / np.float32(8.0))


def main():
    code4 = codebooks.nf4_code4()
    code8 = codebooks.dynamic_code8()
    w = pattern_weight()
    st = oracle.quantize(w, code4, 64, True, code8, 256)
    wb = oracle.dequantize(st, "bf16")
    x = pattern_x()
    y = oracle.linear_fwd(x, wb)
    out = {
        "what": "oracle outputs for the closed-form pattern of make_golden.py (N=16, K=192, M=5)",
        "packed_hex": st.packed.tobytes().hex(),
        "absmax_f32_hex": st.absmax.tobytes().hex(),
        "absmax_q_hex": st.absmax_q.tobytes().hex(),
        "nested_absmax_f32_hex": st.nested_absmax.tobytes().hex(),
        "nested_offset_f32_hex": st.nested_offset.tobytes().hex(),
        "dequant_bf16_hex": wb.tobytes().hex(),
        "y_f64_hex": y.tobytes().hex(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "nf4_oracle_small.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
