"""The seeded input generator: storage formats and determinism (CPU only)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi


def test_bf16_rounding_matches_torch():
    rng = np.random.Generator(np.random.PCG64(0))
    v = np.concatenate([rng.normal(0, 1, 4096), rng.normal(0, 1e-30, 64), [0.0, -0.0, 1e30, -3.0]])
    v = v.astype(np.float32)
    ours = mi.round_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(mi.bf16_bits_to_f32(ours), torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_pack_unpack_roundtrip():
    rng = np.random.Generator(np.random.PCG64(1))
    q = rng.integers(0, 16, size=(3, 5, 64), dtype=np.uint8)
    p = mi.pack_int4(q)
    assert p.shape == (3, 5, 8) and p.dtype == np.uint32
    assert np.array_equal(mi.unpack_int4(p), q)
    assert mi.pack_int4(np.arange(8, dtype=np.uint8))[0] == 0x76543210


def test_layer_is_deterministic_and_shaped():
    for name in ("tiny",):
        sp = mi.SPECS[name]
        a, b = mi.make_layer(sp, 3), mi.make_layer(sp, 3)
        for k, v in a.arrays().items():
            assert np.array_equal(v, b.arrays()[k]), k
        assert a.up_q.shape == (sp.n_experts, sp.expert_ffn, sp.k_in // 8)
        assert a.up_s.shape == (sp.n_experts, sp.expert_ffn, sp.k_in // sp.group_size)
        assert a.down_q.shape == (sp.n_experts, sp.k_in, sp.expert_ffn // 8)
        c = mi.make_layer(sp, 4)
        assert not np.array_equal(a.up_q, c.up_q)


def test_direct_codes_statistics():
    """Large layers draw codes directly; reconstructed weights keep mean ~0 and
    std ~weight_std."""
    sp = mi.SPECS["tiny"].with_(n_experts=4)
    rng = np.random.Generator(np.random.PCG64(2))
    words, s, b = mi._quant_expert_direct(rng, 4, 256, 512, sp)
    q = mi.unpack_int4(words).astype(np.float64)
    w = q * np.repeat(mi.bf16_bits_to_f32(s), 64, -1) + np.repeat(mi.bf16_bits_to_f32(b), 64, -1)
    assert abs(w.mean()) < 2e-3 and abs(w.std() - 0.02) < 2e-3


def test_zipf_bias_is_a_ranking():
    b = mi.zipf_router_bias(496, 0)
    assert b.shape == (496,) and b.max() == 0.0 and len(np.unique(b)) == 496


def test_fp4_codecs_round_trip():
    """The generator's encoders and the oracle's decoders (written apart) agree
    on every representable value: each finite non-negative E4M3 value encodes
    to its own byte, each E2M1 value to its own code, and values between two
    grid points go to the nearer one (E4M3 ties to the even mantissa)."""
    import numpy as np
    import moe_inputs as mi
    from oracle import moe_oracle as ora
    b = np.arange(0x7F)                     # 0x00..0x7E: every non-negative finite E4M3 byte
    v = ora.e4m3_values(b)
    eb, ev = mi.e4m3_round(v)
    assert np.array_equal(eb, b) and np.array_equal(ev, v)
    mid = (v[1:] + v[:-1]) / 2              # exact midpoints: ties to the even mantissa
    mb, _ = mi.e4m3_round(mid)
    assert np.all((mb == b[:-1]) | (mb == b[1:]))
    assert np.all(mb % 2 == 0)
    above, _ = mi.e4m3_round(mid * (1 + 2.0 ** -20))
    assert np.array_equal(above, b[1:])
    codes = np.arange(16)
    vals = ora.e2m1_values(codes)
    got = mi.e2m1_round(vals)
    # +0 and -0 both encode as code 0 (the encoder keeps no sign for zero)
    assert np.array_equal(ora.e2m1_values(got), vals) and got[8] == 0
    e8 = np.arange(0xFF)
    assert np.array_equal(np.log2(ora.e8m0_values(e8)), e8 - 127.0)


def test_e4m3_codecs_match_torch_float8():
    """A third implementation: PyTorch's float8_e4m3fn decodes every byte to the
    oracle's value (NaN where the oracle has NaN) and rounds the generator's
    inputs to the same bytes."""
    import numpy as np
    import moe_inputs as mi
    from oracle import moe_oracle as ora
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this PyTorch")
    b = np.arange(256, dtype=np.uint8)
    tv = torch.from_numpy(b).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ov = ora.e4m3_values(b)
    nan = np.isnan(ov)
    assert np.array_equal(np.isnan(tv), nan)
    assert np.array_equal(tv[~nan], ov[~nan])
    rng = np.random.Generator(np.random.PCG64(3))
    x = np.abs(rng.normal(0, 30, 4096)) + rng.uniform(0, 2.0 ** -7, 4096)
    x = np.minimum(x, 448.0)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    x32 = x.astype(np.float32).astype(np.float64)
    ours32, _ = mi.e4m3_round(x32)
    assert np.array_equal(ours32, ref)
