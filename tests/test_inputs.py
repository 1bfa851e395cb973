"""The seeded input generator: storage formats and determinism (CPU only)."""
import numpy as np
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
