"""The library derives its codebooks with its own code (torch); they must equal the
oracle's (numpy/scipy) bit for bit, for every table a user can select."""
import numpy as np
import pytest

from oracle import codebooks as ocb
import bit_nf4_quantized_linear_gb300 as nf4


@pytest.mark.parametrize("name", ["nf4_code4", "fp4_code4", "dynamic_code8", "e4m3_code8"])
def test_library_codebooks_equal_oracle_bits(name):
    lib = getattr(nf4, name)().numpy()
    ref = getattr(ocb, name)()
    assert lib.dtype == np.float32 and lib.shape == ref.shape
    np.testing.assert_array_equal(lib.view(np.uint32), ref.view(np.uint32))


def test_code4_for_quant_type():
    np.testing.assert_array_equal(nf4.code4_for("nf4").numpy(), ocb.nf4_code4())
    np.testing.assert_array_equal(nf4.code4_for("fp4").numpy().view(np.uint32),
                                  ocb.fp4_code4().view(np.uint32))
    with pytest.raises(ValueError):
        nf4.code4_for("int4")


def test_code_for_every_quant_type():
    for qt, ref in (("nf4", ocb.nf4_code4()), ("fp4", ocb.fp4_code4()),
                    ("int8", ocb.dynamic_code8()), ("fp8", ocb.e4m3_code8())):
        np.testing.assert_array_equal(nf4.code_for(qt).numpy().view(np.uint32), ref.view(np.uint32))
    with pytest.raises(ValueError):
        nf4.code_for("nf8")
