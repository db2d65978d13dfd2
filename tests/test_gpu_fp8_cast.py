"""The library's E4M3 conversion against the oracle's encoder, value by value.

Every FP8 quantiser of the library (queries, pooled keys, the paged append) applies one conversion to its scaled
values (magnitudes up to 448 by construction).  This sweeps every fp32 value of both signs in the binades
[2^-12, 2^9), which hold every rounding transition of E4M3 including the subnormal steps, the ties and the
saturation above 448, plus a strided sample of smaller and larger finite values, and compares the codes with the
oracle's encoder (written from the OCP E4M3 definition) bit for bit."""
import numpy as np
import pytest
import torch

from oracle import kpool_oracle as O
from pooled_key_dsa_gb300 import build as B
from pooled_key_dsa_gb300 import kpooldsa as K

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    K.lib()


def _compare(bits: np.ndarray):
    x = bits.view(np.float32)
    got = K.cast_e4m3(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = O.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[k]), int(got[k]), int(ref[k])) for k in bad[:8]]


@pytest.mark.parametrize("sign", [0, 1])
def test_every_value_of_the_rounding_binades(sign):
    mant = np.arange(1 << 23, dtype=np.uint32)
    for e in range(127 - 12, 127 + 9):                 # binades 2^-12 .. [256, 512)
        _compare((np.uint32(sign) << 31) | (np.uint32(e) << 23) | mant)


def test_strided_sample_of_tiny_and_large_values():
    step = 7919                                          # a prime stride through the bit patterns
    lo = np.arange(0, (127 - 12) << 23, step, dtype=np.uint32)          # zero, subnormals .. 2^-12
    hi = np.arange((127 + 9) << 23, 0x7F800000, step, dtype=np.uint32)   # 512 .. the largest finite value
    for part in (lo, hi):
        _compare(part)
        _compare(part | np.uint32(1 << 31))
