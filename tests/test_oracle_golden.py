"""The oracle reproduces its stored outputs (tests/golden/nf4_oracle_small.json,
written by tests/golden/make_golden.py from the oracle alone) on this machine."""
import json
import os

import numpy as np

import oracle
from oracle import codebooks
from tests.golden import make_golden

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "nf4_oracle_small.json")


def test_oracle_matches_stored_golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    st = oracle.quantize(make_golden.pattern_weight(), codebooks.nf4_code4(), 64, True,
                         codebooks.dynamic_code8(), 256)
    assert st.packed.tobytes().hex() == g["packed_hex"]
    assert st.absmax.tobytes().hex() == g["absmax_f32_hex"]
    assert st.absmax_q.tobytes().hex() == g["absmax_q_hex"]
    assert st.nested_absmax.tobytes().hex() == g["nested_absmax_f32_hex"]
    assert st.nested_offset.tobytes().hex() == g["nested_offset_f32_hex"]
    wb = oracle.dequantize(st, "bf16")
    assert wb.tobytes().hex() == g["dequant_bf16_hex"]
    y = oracle.linear_fwd(make_golden.pattern_x(), wb)
    np.testing.assert_array_equal(y, np.frombuffer(bytes.fromhex(g["y_f64_hex"]), np.float64).reshape(y.shape))
