"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one part of the oracle to a library routine, a closed form, an invariant of the
block's definition, or a brute-force dense computation on a tiny shape.  Together they are chosen
so that a dropped term, a wrong sign, a wrong group or row index, or a transposed operand fails at
least one of them (tests/test_oracle_mutants.py plants such mistakes and checks that).

Block definition pinned here: kernel A of "two-kernel decode-MoE that beats gather_qmm" (What
changed, step 2: gate/up + swiglu into act_g[K, Dff]), kernel B of the same step (down * score,
summed over K) and the tail of "Red Lite dev39 -- fused expert tail" (Change: x = resid +
(routed + shared * scalar)), with affine dequantisation w = scale * q + bias per group of 64.
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle import oracle as O
from quantized_moe_expert_dequant_gb300 import synth
from tests import helpers as H

ONE_F16 = 0x3C00


def f16_bits(v):
    return np.asarray(v, dtype=np.float16).view(np.uint16)


# ------------------------------------------------------------------ exact conversions

def test_f16_every_pattern_matches_numpy():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([O.f16(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_every_pattern_matches_fp32_upper_half():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = (pats.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([O.bf16(int(b)) for b in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------------ unpacking

@pytest.mark.parametrize("bits", [4, 6, 8])
def test_unpack_every_value_at_every_phase(bits):
    # code c = (c // phases) mod 2^b puts each value at every bit phase a code can start on
    phases = {4: 2, 6: 4, 8: 1}[bits]
    n = (1 << bits) * phases
    n = -(-n // 64) * 64
    codes = np.array([(c // phases) % (1 << bits) for c in range(n)])
    row = H.pack_bigint(codes, bits)
    assert np.array_equal(O.unpack_row(row, bits, n), codes)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_unpack_random_rows(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=256)
    row = H.pack_bigint(codes, bits)
    assert np.array_equal(O.unpack_row(row, bits, 256), codes)
    # and the synthetic code bytes read back the same through both readers
    cb = synth.code_bytes(7, 0, synth.GATE, 3, 2, 128, bits)
    for r in range(2):
        assert np.array_equal(O.unpack_row(cb[r], bits, 128), H.unpack_bigint(cb[r], bits, 128))


def test_unpack_matches_uint32_word_layout():
    # the canonical layout packs 8 nibbles per little-endian uint32, nibble n at bits 4n
    rng = np.random.default_rng(0)
    q = rng.integers(0, 16, size=64).astype(np.uint32)
    words = np.zeros(8, dtype=np.uint32)
    for i in range(8):
        for n in range(8):
            words[i] |= q[8 * i + n] << np.uint32(4 * n)
    row = words.astype("<u4").view(np.uint8)
    assert np.array_equal(row, H.pack_bigint(q, 4))
    assert np.array_equal(O.unpack_row(row, 4, 64), q)


# ------------------------------------------------------------------ dequantisation

def _proj(Q, scales, biases, bits):
    return H.packed_from_codes(Q, f16_bits(scales), f16_bits(biases), bits)


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_weight_unit_scale_zero_bias_is_the_code(bits):
    rng = np.random.default_rng(1)
    Q = rng.integers(0, 1 << bits, size=(3, 128))
    p = _proj(Q, np.ones((3, 2)), np.zeros((3, 2)), bits)
    for r in range(3):
        for c in range(0, 128, 5):
            assert O.weight(p, r, c) == Q[r, c]


def test_weight_zero_scale_reads_the_bias_of_its_row_and_group():
    Q = np.full((3, 192), 5)
    biases = np.arange(9, dtype=np.float64).reshape(3, 3) - 4.0
    p = _proj(Q, np.zeros((3, 3)), biases, 4)
    for r in range(3):
        for c in range(192):
            assert O.weight(p, r, c) == biases[r, c // 64]


def test_weight_scale_of_its_row_and_group():
    Q = np.full((2, 128), 3)
    scales = np.array([[0.5, 2.0], [-4.0, 0.25]])
    p = _proj(Q, scales, np.full((2, 2), -1.0), 4)
    for r in range(2):
        for c in (0, 63, 64, 127):
            assert O.weight(p, r, c) == scales[r, c // 64] * 3 - 1.0


def test_weight_centred_codes():
    Q = np.arange(16).repeat(4).reshape(1, 64)
    p = _proj(Q, np.ones((1, 1)), np.full((1, 1), -8.0), 4)
    assert [O.weight(p, 0, c) for c in range(0, 64, 4)] == list(range(-8, 8))


# ------------------------------------------------------------------ matvec

def test_matvec_one_hot_picks_a_column_and_ones_sum_rows():
    rng = np.random.default_rng(2)
    Q = rng.integers(0, 16, size=(5, 128))
    p = _proj(Q, np.ones((5, 2)), np.zeros((5, 2)), 4)
    for c in (0, 1, 63, 64, 127):
        e = np.zeros(128)
        e[c] = 1.0
        assert np.array_equal(O.matvec(p, e), Q[:, c].astype(np.float64))
    assert np.array_equal(O.matvec(p, np.ones(128)), Q.sum(axis=1).astype(np.float64))
    assert np.array_equal(O.matvec(p, np.ones(128), rows=[4, 1]), Q.sum(axis=1)[[4, 1]])


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_matvec_brute_force_dense(bits):
    p = H.synth_packed(11, 0, synth.DOWN, 2, 96, 192, bits)
    v = np.random.default_rng(3).standard_normal(192)
    ref = H.dense(p) @ v
    got = O.matvec(p, v)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


# ------------------------------------------------------------------ activations

def test_silu_and_sigmoid_against_expit():
    assert O.silu(0.0) == 0.0
    assert O.sigmoid(0.0) == 0.5
    for z in np.linspace(-30, 30, 61):
        assert O.sigmoid(z) == pytest.approx(float(expit(z)), rel=1e-14, abs=1e-300)
        assert O.silu(z) == pytest.approx(z * float(expit(z)), rel=1e-14, abs=1e-300)
        assert O.silu(z) - O.silu(-z) == pytest.approx(z, rel=1e-14, abs=1e-14)


def test_expert_act_zero_gate_is_zero_and_brute_force():
    din, dff = 128, 64
    x = H.bf16_to_f64(synth.activations(1, 0, 0, din))
    zero_gate = _proj(np.zeros((dff, din), dtype=int), np.ones((dff, 2)), np.zeros((dff, 2)), 4)
    up = H.synth_packed(1, 0, synth.UP, 0, dff, din, 4)
    assert np.array_equal(O.expert_act(zero_gate, up, x), np.zeros(dff))
    gate = H.synth_packed(1, 0, synth.GATE, 0, dff, din, 4)
    ref = H.dense_expert_act(gate, up, x)
    assert np.allclose(O.expert_act(gate, up, x), ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_expert_act_is_silu_gate_times_up_not_swapped():
    # gate . x = 2 and up . x = -3 exactly: act = silu(2) * -3, and silu(-3) * 2 if swapped
    din, dff = 64, 64
    x = np.ones(din)
    Qg = np.zeros((dff, din), dtype=int)
    Qg[:, :2] = 1
    Qu = np.zeros((dff, din), dtype=int)
    Qu[:, :3] = 1
    gate = _proj(Qg, np.ones((dff, 1)), np.zeros((dff, 1)), 4)
    up = _proj(Qu, -np.ones((dff, 1)), np.zeros((dff, 1)), 4)
    act = O.expert_act(gate, up, x)
    assert np.allclose(act, 2 * expit(2.0) * -3.0, rtol=1e-15)


def test_shared_scalar_closed_forms():
    din = 64
    x = H.bf16_to_f64(synth.activations(2, 0, 0, din))
    assert O.shared_scalar(x, np.zeros(din, dtype=np.uint16)) == 0.5
    g = synth.f32_to_bf16_bits(np.full(din, 1.0 / 64, dtype=np.float32))  # exact in bf16
    ones = np.ones(din)
    assert O.shared_scalar(ones, g) == pytest.approx(float(expit(1.0)), rel=1e-15)
    assert O.shared_scalar(-ones, g) == pytest.approx(float(expit(-1.0)), rel=1e-15)


# ------------------------------------------------------------------ the whole block

def _tiny_layer(seed=5, din=64, dff=64, E=4, bits=(4, 4, 4), n_sh=0, dff_sh=64, bits_sh=4):
    mk = lambda proj, e, r, c, b: H.synth_packed(seed, 0, proj, e, r, c, b)
    gate = [mk(synth.GATE, e, dff, din, bits[0]) for e in range(E)]
    up = [mk(synth.UP, e, dff, din, bits[1]) for e in range(E)]
    down = [mk(synth.DOWN, e, din, dff, bits[2]) for e in range(E)]
    shg = [mk(synth.SH_GATE, s, dff_sh, din, bits_sh) for s in range(n_sh)]
    shu = [mk(synth.SH_UP, s, dff_sh, din, bits_sh) for s in range(n_sh)]
    shd = [mk(synth.SH_DOWN, s, din, dff_sh, bits_sh) for s in range(n_sh)]
    return gate, up, down, shg, shu, shd


def _sel(lst, ids):
    return [lst[i] for i in ids]


@pytest.mark.parametrize("bits", [(4, 4, 4), (8, 8, 8), (4, 4, 6), (6, 6, 8)])
def test_block_brute_force_tiny(bits):
    # Din=64, Dff=64 (down's groups run along Dff, so Dff is at least one group), E=4, K=2, plus
    # a gated shared expert
    din, dff, E, K = 64, 64, 4, 2
    gate, up, down, shg, shu, shd = _tiny_layer(din=din, dff=dff, E=E, bits=bits, n_sh=1)
    x = synth.activations(5, 0, 0, din)
    resid = synth.residual(5, 0, 0, din)
    ids = synth.topk_ids(5, 0, 0, E, K)
    sc = synth.scores(5, 0, 0, K)
    gv = synth.gate_vector(5, 0, din)
    got = O.moe_token(x, resid, sc, _sel(gate, ids), _sel(up, ids), _sel(down, ids), shg, shu, shd,
                      gate_vec_bf16=gv)
    ref = H.dense_block(x, H.bf16_to_f64(resid), sc, _sel(gate, ids), _sel(up, ids),
                        _sel(down, ids), shg, shu, shd, gate_vec=gv)
    assert H.rel_l2(got, ref) < 1e-13


def test_block_single_expert_unit_score_is_the_expert_mlp():
    din, dff = 128, 64
    gate, up, down, *_ = _tiny_layer(din=din, dff=dff, E=2)
    x = synth.activations(6, 0, 0, din)
    resid = np.zeros(din, dtype=np.float32)
    got = O.moe_token(x, resid, np.ones(1, np.float32), [gate[1]], [up[1]], [down[1]])
    ref = H.dense(down[1]) @ H.dense_expert_act(gate[1], up[1], H.bf16_to_f64(x))
    assert H.rel_l2(got, ref) < 1e-13


def test_block_zero_scores_leave_resid_plus_shared_term():
    din, dff = 64, 64
    gate, up, down, shg, shu, shd = _tiny_layer(din=din, dff=dff, n_sh=2, dff_sh=128)
    x = synth.activations(7, 0, 0, din)
    resid = synth.residual(7, 0, 0, din)
    gv = synth.gate_vector(7, 0, din)
    zero = np.zeros(3, np.float32)
    got = O.moe_token(x, resid, zero, gate[:3], up[:3], down[:3], shg, shu, shd, gate_vec_bf16=gv)
    xf = H.bf16_to_f64(x)
    sh = sum(H.dense(shd[s]) @ H.dense_expert_act(shg[s], shu[s], xf) for s in range(2))
    ref = H.bf16_to_f64(resid) + float(expit(xf @ H.bf16_to_f64(gv))) * sh
    assert H.rel_l2(got - H.bf16_to_f64(resid), ref - H.bf16_to_f64(resid)) < 1e-13
    # and with no routed slots at all
    got0 = O.moe_token(x, resid, np.zeros(0, np.float32), [], [], [], shg, shu, shd, gate_vec_bf16=gv)
    assert np.allclose(got0, got, rtol=0, atol=1e-12)


def test_block_ungated_shared_scalar_is_one():
    din, dff = 64, 64
    _, _, _, shg, shu, shd = _tiny_layer(din=din, dff=dff, n_sh=1)
    x = synth.activations(8, 0, 0, din)
    resid = np.zeros(din, np.float32)
    got1 = O.moe_token(x, resid, np.zeros(0, np.float32), [], [], [], shg, shu, shd)
    gzero = np.zeros(din, dtype=np.uint16)
    got_half = O.moe_token(x, resid, np.zeros(0, np.float32), [], [], [], shg, shu, shd,
                           gate_vec_bf16=gzero)
    assert np.allclose(got_half, 0.5 * got1, rtol=1e-14, atol=1e-14)


def test_block_slot_permutation_invariant_and_scores_follow_their_slot():
    din, dff, E = 64, 64, 4
    gate, up, down, *_ = _tiny_layer(din=din, dff=dff, E=E)
    x = synth.activations(9, 0, 0, din)
    resid = synth.residual(9, 0, 0, din)
    ids = np.array([2, 0, 3])
    sc = np.array([0.5, 0.3, 0.2], np.float32)
    base = O.moe_token(x, resid, sc, _sel(gate, ids), _sel(up, ids), _sel(down, ids))
    perm = [2, 0, 1]
    got = O.moe_token(x, resid, sc[perm], _sel(gate, ids[perm]), _sel(up, ids[perm]),
                      _sel(down, ids[perm]))
    assert np.allclose(got, base, rtol=1e-12, atol=1e-12)
    # permuting the scores alone changes the output
    bad = O.moe_token(x, resid, sc[perm], _sel(gate, ids), _sel(up, ids), _sel(down, ids))
    assert not np.allclose(bad, base, rtol=1e-6, atol=1e-6)


def test_block_linear_in_scores_and_duplicate_slots_merge():
    din, dff = 64, 64
    gate, up, down, *_ = _tiny_layer(din=din, dff=dff, E=3)
    x = synth.activations(10, 0, 0, din)
    resid = np.zeros(din, np.float32)
    sc = np.array([0.25, 0.75], np.float32)
    one = O.moe_token(x, resid, sc, gate[:2], up[:2], down[:2])
    two = O.moe_token(x, resid, 2 * sc, gate[:2], up[:2], down[:2])
    assert np.allclose(two, 2 * one, rtol=1e-13, atol=1e-13)
    dup = O.moe_token(x, resid, np.array([0.25, 0.5, 0.25], np.float32), [gate[0], gate[1], gate[1]],
                      [up[0], up[1], up[1]], [down[0], down[1], down[1]])
    assert np.allclose(dup, one, rtol=1e-13, atol=1e-13)


def test_block_resid_is_added_once_in_either_dtype():
    din, dff = 64, 64
    gate, up, down, *_ = _tiny_layer(din=din, dff=dff, E=2)
    x = synth.activations(11, 0, 0, din)
    r16 = synth.residual(11, 0, 0, din)
    r32 = synth.bf16_bits_to_f32(r16)
    sc = np.array([1.0], np.float32)
    a = O.moe_token(x, r16, sc, gate[:1], up[:1], down[:1])
    b = O.moe_token(x, r32, sc, gate[:1], up[:1], down[:1])
    z = O.moe_token(x, np.zeros(din, np.float32), sc, gate[:1], up[:1], down[:1])
    assert np.array_equal(a, b)
    assert np.allclose(a - z, r32.astype(np.float64), rtol=0, atol=1e-12)


def test_block_row_subset_equals_full_rows():
    din, dff = 128, 64
    gate, up, down, shg, shu, shd = _tiny_layer(din=din, dff=dff, E=2, n_sh=1)
    x = synth.activations(12, 0, 0, din)
    resid = synth.residual(12, 0, 0, din)
    sc = np.array([0.6, 0.4], np.float32)
    gv = synth.gate_vector(12, 0, din)
    full = O.moe_token(x, resid, sc, gate, up, down, shg, shu, shd, gate_vec_bf16=gv)
    rows = [127, 0, 64, 63, 5]
    part = O.moe_token(x, resid, sc, gate, up, down, shg, shu, shd, gate_vec_bf16=gv, rows=rows)
    assert np.array_equal(part, full[rows])


def test_block_rejects_mismatched_shapes():
    gate, up, down, *_ = _tiny_layer(din=64, dff=64, E=1)
    x = synth.activations(13, 0, 0, 128)
    with pytest.raises(ValueError):
        O.moe_token(x, np.zeros(128, np.float32), np.ones(1, np.float32), gate, up, down)


# ---------------------------------------------------------------- route inversion (batches of tokens)

def _brute_invert(ids, n_experts):
    """Independent restatement: a dict from expert to its pairs, built in one scan."""
    groups = {}
    for p, e in enumerate(np.asarray(ids).reshape(-1).tolist()):
        if 0 <= e < n_experts:
            groups.setdefault(e, []).append(p)
    return groups


@pytest.mark.parametrize("m,k,E,seed", [(1, 8, 128, 1), (8, 6, 128, 2), (32, 6, 128, 3),
                                        (4, 4, 5, 4), (16, 10, 512, 5)])
def test_route_invert_matches_brute_force(m, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(m)]).astype(np.int32)
    uniq, offs, pairs = O.route_invert(ids, E)
    groups = _brute_invert(ids, E)
    assert uniq.tolist() == sorted(groups)
    for u, e in enumerate(uniq):
        assert pairs[offs[u]:offs[u + 1]].tolist() == groups[e]
    # every pair appears exactly once, and each names its expert
    assert sorted(pairs.tolist()) == list(range(m * k))
    for u, e in enumerate(uniq):
        assert all(ids.reshape(-1)[p] == e for p in pairs[offs[u]:offs[u + 1]])


def test_route_invert_special_cases():
    # one token: every slot its own expert, experts ascending, pairs follow the ids' order
    ids = np.array([[7, 3, 9]], np.int32)
    uniq, offs, pairs = O.route_invert(ids, 10)
    assert uniq.tolist() == [3, 7, 9] and offs.tolist() == [0, 1, 2, 3]
    assert pairs.tolist() == [1, 0, 2]
    # every token picks the same experts: one group per expert with all tokens in order
    ids = np.array([[2, 0]] * 4, np.int32)
    uniq, offs, pairs = O.route_invert(ids, 3)
    assert uniq.tolist() == [0, 2]
    assert pairs[offs[0]:offs[1]].tolist() == [1, 3, 5, 7]
    assert pairs[offs[1]:offs[2]].tolist() == [0, 2, 4, 6]
    # invalid ids belong to no group; a repeated id inside one token gives two pairs
    ids = np.array([[-1, 4, 4], [5, 9, 0]], np.int32)
    uniq, offs, pairs = O.route_invert(ids, 5)
    assert uniq.tolist() == [0, 4] and pairs.tolist() == [5, 1, 2]
    # nothing valid
    uniq, offs, pairs = O.route_invert(np.array([[-3, 7]], np.int32), 5)
    assert len(uniq) == 0 and offs.tolist() == [0] and len(pairs) == 0


# ---------------------------------------------------------------- router (top-k pool with softmax weights)

def _brute_router(logits, k):
    """Independent restatement: a stable sort on (-logit, id), softmax with numpy in float64."""
    order = sorted(range(len(logits)), key=lambda e: (-float(logits[e]), e))[:k]
    z = np.array([float(logits[e]) for e in order])
    w = np.exp(z - z.max())
    return np.array(order, np.int32), (w / w.sum()).astype(np.float32)


@pytest.mark.parametrize("E,k,seed", [(128, 8, 1), (60, 4, 2), (512, 10, 3), (128, 6, 4), (5, 5, 5),
                                      (1024, 64, 6)])
def test_router_matches_brute_force(E, k, seed):
    logits = np.random.default_rng(seed).standard_normal(E).astype(np.float32)
    ids, scores = O.router(logits, k)
    bi, bs = _brute_router(logits, k)
    assert np.array_equal(ids, bi)
    np.testing.assert_allclose(scores, bs, rtol=1e-6, atol=0)
    assert abs(float(np.sum(scores.astype(np.float64))) - 1.0) < 1e-6
    assert np.all(np.diff(logits[ids]) <= 0)          # larger logits first


def test_router_ties_and_special_cases():
    logits = np.array([0.5, 2.0, 2.0, -1.0, 2.0, 0.5], np.float32)
    ids, scores = O.router(logits, 4)
    assert ids.tolist() == [1, 2, 4, 0]                  # equal logits: lower id first
    assert np.allclose(scores[:3], scores[0]) and scores[3] < scores[0]
    ids, scores = O.router(logits, 1)
    assert ids.tolist() == [1] and scores.tolist() == [1.0]   # one slot: weight exactly 1
    # k = E: every expert, ordered; the weights are the full softmax
    z = np.array([3.0, -2.0, 0.0], np.float32)
    ids, scores = O.router(z, 3)
    assert ids.tolist() == [0, 2, 1]
    e = np.exp(np.array([3.0, 0.0, -2.0]) - 3.0)
    np.testing.assert_allclose(scores, e / e.sum(), rtol=1e-7)
    # shifting every logit by a constant changes no id and no weight (beyond rounding)
    logits = np.random.default_rng(9).standard_normal(64).astype(np.float32)
    i1, s1 = O.router(logits, 8)
    i2, s2 = O.router(logits + np.float32(4.0), 8)
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(s1, s2, rtol=1e-5)


# ------------------------------------------------------------------ the folded RMSNorm (chained stack)
# "Red Lite dev39 -- fused expert tail", Measurements: a tail that also folded in the next layer's
# RMSNorm.  The page gives no formula; the oracle takes the usual RMSNorm, rounded to bf16.

def test_round_bf16_ties_to_even_and_edges():
    one = 0x3F80
    assert O.round_bf16(1.0) == one
    assert O.round_bf16(1 + 2.0 ** -8) == one              # halfway to 1 + 2^-7: the even one
    assert O.round_bf16(1 + 3 * 2.0 ** -8) == 0x3F82       # halfway to 1 + 2^-6: the even one
    assert O.round_bf16(1 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert O.round_bf16(-(1 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81
    assert O.round_bf16(2.0 ** -133) == 0x0001             # smallest subnormal
    assert O.round_bf16(2.0 ** -134) == 0x0000             # halfway to zero: even
    assert O.round_bf16(3 * 2.0 ** -134) == 0x0002
    assert O.round_bf16(3.39e38) == 0x7F7F                 # largest finite bf16 is 3.3895e38
    assert O.round_bf16(3.4e38) == 0x7F80 and O.round_bf16(-3.4e38) == 0xFF80
    assert O.round_bf16(float("inf")) == 0x7F80 and O.round_bf16(float("-inf")) == 0xFF80
    assert O.round_bf16(0.0) == 0 and O.round_bf16(-0.0) == 0x8000
    nan = O.round_bf16(float("nan"))
    assert nan & 0x7F80 == 0x7F80 and nan & 0x7F


def test_round_bf16_matches_an_independent_fp32_rounding():
    v = np.random.default_rng(3).standard_normal(4000).astype(np.float32)
    v *= np.float32(2.0) ** np.random.default_rng(4).integers(-60, 60, 4000).astype(np.float32)
    got = np.array([O.round_bf16(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, synth.f32_to_bf16_bits(v))


def rne_bf16_f64(y: np.ndarray) -> np.ndarray:
    """y (fp64) rounded once to the nearest bf16 value, ties to even: a test-side restatement
    of round-to-nearest at the bf16 spacing (8 significant bits), normal range only."""
    _, e = np.frexp(y)
    sp = np.ldexp(1.0, e - 8)
    return np.rint(y / sp) * sp


def test_rmsnorm_matches_torch_rms_norm():
    """The norm is gamma * v / sqrt(mean v^2 + eps) rounded once to bf16: the oracle's codes equal
    torch's fp64 rms_norm rounded to nearest even, except where torch's value lies within 1e-12
    (relative) of a rounding tie, where the two fp64 evaluation orders may fall either side."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    for n, eps, scale in ((2048, 1e-6, 1.0), (4096, 1e-5, 30.0), (64, 1e-6, 1e-3), (192, 0.0, 1.0)):
        v = (rng.standard_normal(n) * scale).astype(np.float32)
        g = synth.f32_to_bf16_bits((1 + 0.2 * rng.standard_normal(n)).astype(np.float32))
        x = synth.bf16_bits_to_f32(O.rmsnorm_bf16(v, g, eps)).astype(np.float64)
        w = torch.from_numpy(synth.bf16_bits_to_f32(g).astype(np.float64))
        ref = torch.nn.functional.rms_norm(torch.from_numpy(v.astype(np.float64))[None], (n,),
                                           weight=w, eps=eps)[0].numpy()
        _, e = np.frexp(ref)
        frac = ref / np.ldexp(1.0, e - 8)
        near_tie = np.abs(np.abs(frac - np.floor(frac)) - 0.5) < 1e-12 * np.abs(frac)
        same = x == rne_bf16_f64(ref)
        assert np.all(same | near_tie), (n, eps, int(np.sum(~same)))
        assert np.all(np.abs(x - ref) <= np.ldexp(1.0, e - 9) * (1 + 1e-12)), (n, eps)


def test_rmsnorm_is_one_rounding_of_the_fp64_value():
    """On a million elements some products lie so close to a bf16 rounding tie that rounding
    v * r and gamma * (v * r) to fp32 first would send them the other way: the oracle follows the
    single rounding of the fp64 value at every one of them."""
    n = 1 << 20
    rng = np.random.default_rng(11)
    v = rng.standard_normal(n).astype(np.float32)
    g = synth.f32_to_bf16_bits((1 + 0.2 * rng.standard_normal(n)).astype(np.float32))
    gf = synth.bf16_bits_to_f32(g)
    r = 1.0 / np.sqrt(np.mean(v.astype(np.float64) ** 2) + 1e-6)
    exact = rne_bf16_f64(gf.astype(np.float64) * (v.astype(np.float64) * r))
    via_f32 = rne_bf16_f64((gf * (v * np.float32(r))).astype(np.float64))
    differ = exact != via_f32
    assert differ.sum() >= 5                      # the case this pin exists for does occur
    got = synth.bf16_bits_to_f32(O.rmsnorm_bf16(v, g, 1e-6)).astype(np.float64)
    assert np.array_equal(got, exact)


def test_rmsnorm_closed_forms_and_scale_invariance():
    n = 256
    unit = np.full(n, 0x3F80, np.uint16)
    for c in (3.0, -0.125, 7e30, 1e-20):
        x = O.rmsnorm_bf16(np.full(n, c, np.float32), unit, 0.0)
        assert np.all(x == (0x3F80 if c > 0 else 0xBF80)), c   # v / rms(v) = sign(v)
    x = O.rmsnorm_bf16(np.zeros(n, np.float32), unit, 1e-6)
    assert np.all(x & 0x7FFF == 0)
    rng = np.random.default_rng(6)
    v = rng.standard_normal(n).astype(np.float32)
    g = synth.f32_to_bf16_bits((1 + 0.2 * rng.standard_normal(n)).astype(np.float32))
    base = O.rmsnorm_bf16(v, g, 0.0)
    for k in (-20, -1, 7):                                    # powers of two scale exactly
        assert np.array_equal(O.rmsnorm_bf16(v * np.float32(2.0 ** k), g, 0.0), base)
    assert np.all(O.rmsnorm_bf16(v, np.zeros(n, np.uint16), 1e-6) & 0x7FFF == 0)
    # mean of x^2 / gamma^2 is 1 up to bf16 rounding (eps 0)
    xf = synth.bf16_bits_to_f32(base).astype(np.float64) / synth.bf16_bits_to_f32(g)
    assert abs(np.mean(xf ** 2) - 1.0) < 2 ** -7


# ------------------------------------------------------------------ dense bf16 decode GEMV
# "Measure attention projections instead of serving them, and record the amortisation trap": the
# q/k/v/o projections of a decode token, y = x W^T with bf16 W and x, measured at 1, 8, 32 rows.

def test_gemv_matches_numpy_matmul():
    rng = np.random.default_rng(8)
    for m, n_out, n_in in ((1, 48, 64), (8, 33, 72), (32, 17, 40), (3, 1, 8)):
        W = synth.f32_to_bf16_bits(rng.standard_normal((n_out, n_in)).astype(np.float32))
        x = synth.f32_to_bf16_bits(rng.standard_normal((m, n_in)).astype(np.float32))
        ref = (synth.bf16_bits_to_f32(x).astype(np.float64)
               @ synth.bf16_bits_to_f32(W).astype(np.float64).T)
        np.testing.assert_allclose(O.gemv_bf16(W, x), ref, rtol=1e-12, atol=1e-12)


def test_gemv_one_hot_inputs_pick_columns_and_rows_stay_apart():
    rng = np.random.default_rng(9)
    n_out, n_in = 12, 24
    W = synth.f32_to_bf16_bits(rng.standard_normal((n_out, n_in)).astype(np.float32))
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    one = synth.f32_to_bf16_bits(np.float32(1.0))
    for i in (0, 7, n_in - 1):
        x = np.zeros((2, n_in), np.uint16)
        x[1, i] = one                                    # token 1 picks column i, token 0 is zero
        y = O.gemv_bf16(W, x)
        assert np.all(y[0] == 0.0)
        assert np.array_equal(y[1], Wf[:, i])
    # a unit row of W returns the matching input element for every token
    Wi = np.zeros((n_in, n_in), np.uint16)
    Wi[np.arange(n_in), np.arange(n_in)] = one
    x = synth.f32_to_bf16_bits(rng.standard_normal((3, n_in)).astype(np.float32))
    assert np.array_equal(O.gemv_bf16(Wi, x), synth.bf16_bits_to_f32(x).astype(np.float64))
