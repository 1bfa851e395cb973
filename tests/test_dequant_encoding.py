"""The 16-bit encodings the grouped GEMM's packed dequantisation relies on,
checked on the host (no GPU): a 4-bit code q placed in the low mantissa bits
of M (128 in bf16, 1024 in fp16) is exactly the number M + q; subtracting M
is exact; and the word layout -- codes i and i + 4 of a 32-bit word share a
pair until two byte permutes put (2i, 2i + 1) together -- yields the codes in
order.  The int4 affine format itself (code q of group g is s_g * q + b_g) is
pinned against the oracle in tests/test_oracle_pins.py; this file covers only
the bit arithmetic of the kernel's fast path, restated in NumPy."""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

MAGIC = {"bf16": 0x4300, "fp16": 0x6400}
BASE = {"bf16": 128.0, "fp16": 1024.0}


def decode16(bits, dt):
    bits = np.asarray(bits, dtype=np.uint32)
    if dt == "fp16":
        return (bits.astype(np.uint16)).view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_magic_number_holds_every_code_exactly(dt):
    q = np.arange(16, dtype=np.uint32)
    v = decode16(MAGIC[dt] | q, dt)
    assert np.array_equal(v, BASE[dt] + q)            # M + q, exactly
    assert np.array_equal(v - BASE[dt], q.astype(np.float64))


def byte_perm(a, b, sel):
    """Byte permute of the pair (b:a): result byte i is byte sel_i of the 8."""
    src = np.concatenate([np.array([a], dtype=np.uint32).view(np.uint8),
                          np.array([b], dtype=np.uint32).view(np.uint8)])
    out = [src[(sel >> (4 * i)) & 7] for i in range(4)]
    return int(np.array(out, dtype=np.uint8).view(np.uint32)[0])


def test_pairing_and_permutes_give_codes_in_order():
    rng = np.random.default_rng(3)
    for _ in range(200):
        v = int(rng.integers(0, 2**32, dtype=np.uint64))
        # the kernel's four pairs: nibbles (i, i + 4) of v >> 4i
        y = [((v >> (4 * i)) & 0x000F000F) | 0x43004300 for i in range(4)]
        o = [byte_perm(y[0], y[1], 0x5410), byte_perm(y[2], y[3], 0x5410),
             byte_perm(y[0], y[1], 0x7632), byte_perm(y[2], y[3], 0x7632)]
        got = []
        for w in o:                                    # low half = lower K index
            got += [w & 0xFFFF, w >> 16]
        codes = [int(x) - 0x4300 for x in got]
        want = [(v >> (4 * c)) & 0xF for c in range(8)]  # code c in bits 4c..4c+3
        assert codes == want
