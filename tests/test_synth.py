"""The seeded input generators: determinism, ranges, and the stated distributions (CPU only)."""
import numpy as np

from quantized_moe_expert_dequant_gb300 import synth


def test_mix64_matches_python_int_and_published_first_outputs():
    # SplitMix64 seeded with 0: the first outputs of the published generator
    first = [synth.mix64_int(synth.G * (i + 1)) for i in range(3)]
    assert first == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    z = np.array([synth.G * (i + 1) & synth.M64 for i in range(3)], dtype=np.uint64)
    assert [int(v) for v in synth.mix64(z)] == first


def test_codes_deterministic_and_uniform():
    a = synth.code_bytes(1, 2, synth.GATE, 5, 64, 2048, 4)
    b = synth.code_bytes(1, 2, synth.GATE, 5, 64, 2048, 4)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, synth.code_bytes(1, 2, synth.GATE, 6, 64, 2048, 4))
    nib = np.concatenate([a.reshape(-1) & 15, a.reshape(-1) >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()


def test_expert_slices_are_independent_of_the_stack():
    one = synth.expert_proj(3, 0, synth.DOWN, 7, 128, 768, 6)
    stack = synth.stacked_proj(3, 0, synth.DOWN, 8, 128, 768, 6)
    for i in range(3):
        assert np.array_equal(stack[i][7], one[i])


def test_scales_and_biases_ranges():
    for bits in (4, 6, 8):
        c, s, b = synth.expert_proj(4, 0, synth.UP, 0, 256, 2048, bits)
        sf = s.view(np.float16).astype(np.float64)
        bf = b.view(np.float16).astype(np.float64)
        assert sf.min() >= 0.005 - 1e-5 and sf.max() <= 0.02 + 1e-5
        ratio = -bf / sf
        half = 2 ** (bits - 1)
        slack = 0.5 + half * 2.0 ** -10  # the +-0.5 spread plus fp16 rounding of the bias
        assert ratio.min() >= half - slack and ratio.max() <= half + slack
        assert abs(ratio.mean() - half) < 0.05


def test_activations_and_router_outputs():
    x = synth.bf16_bits_to_f32(synth.activations(0, 0, 0, 1 << 16)).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    g = synth.bf16_bits_to_f32(synth.gate_vector(0, 0, 1 << 16)).astype(np.float64)
    assert abs(g.std() - 0.02) < 0.001
    for E, K in ((128, 8), (60, 4), (512, 10), (4, 4)):
        ids = synth.topk_ids(9, 1, 0, E, K)
        assert len(set(ids.tolist())) == K and ids.min() >= 0 and ids.max() < E
        sc = synth.scores(9, 1, 0, K)
        assert sc.dtype == np.float32 and abs(float(sc.sum()) - 1) < 1e-6 and (sc > 0).all()
    assert not np.array_equal(synth.topk_ids(9, 1, 0, 128, 8), synth.topk_ids(9, 2, 0, 128, 8))


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]
