"""Pins of the CPU oracle against something other than itself.

Each test checks one oracle function against values the pages print (fixtures in
tests/golden, each with its citation), a closed form, a library routine, brute force
on tiny inputs, or an invariant the method fixes.  They are chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ================================================================ formats
def test_bf16_decoder_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, 20000, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_to_f64(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_decoder_exhaustive_vs_torch_and_spec_points():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])
    # OCP E4M3 landmarks: largest finite, smallest normal, smallest subnormal, one, NaN codes
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])


def test_e2m1_levels_are_the_pages_magnitudes():
    g = gold("fp4_course_lesson.json")
    pos = O.e2m1_to_f64(np.arange(8))
    neg = O.e2m1_to_f64(np.arange(8, 16))
    assert pos.tolist() == g["e2m1_magnitudes"]
    assert (-neg).tolist() == g["e2m1_magnitudes"]


def test_fp4_dequant_page_examples_and_layout():
    g = gold("fp4_course_lesson.json")
    level3 = 0b0101  # e=2, m=1 -> 3
    for scale, expect in g["level3_times_scale"]:
        scode = int(torch.tensor([scale]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
        codes = np.array([[level3 | (level3 << 4)] * 8], np.uint8)  # 16 channels
        vals = O.fp4_to_f64(codes, np.array([[scode]], np.uint8), 16)
        assert np.all(vals == expect)
    # nibble order (low nibble = even channel) and one scale per group
    codes = np.zeros((1, 16), np.uint8)  # 32 channels
    codes[0, 0] = 0x2 | (0xB << 4)  # ch0 = +1.0, ch1 = -1.5
    codes[0, 8] = 0x7  # ch16 = +6
    s_half = 0x30  # E4M3 0.5
    s_two = 0x40  # E4M3 2.0
    v16 = O.fp4_to_f64(codes, np.array([[s_half, s_two]], np.uint8), 16)
    assert v16[0, 0] == 0.5 and v16[0, 1] == -0.75 and v16[0, 16] == 12.0
    v32 = O.fp4_to_f64(codes, np.array([[s_two]], np.uint8), 32)
    assert v32[0, 0] == 2.0 and v32[0, 1] == -3.0 and v32[0, 16] == 12.0
    # record size at group 16: 4.5 bits per channel, 288 B per 512-channel latent
    assert (512 // 2 + 512 // 16) == g["bytes_per_512_latent_group16"]
    assert (16 * 4 + 8) / 16 == g["bits_per_channel_group16"]


def test_generator_fp4_encoder_page_example():
    g = gold("fp4_course_lesson.json")
    x = torch.zeros(1, 32)
    x[0, 0] = 3.2
    x[0, 1] = 6.0  # makes the group scale exactly 1
    codes, scales = synth.fp4_groups(x, 32)
    vals = O.fp4_to_f64(codes, scales, 32)
    assert vals[0, 0] == g["store_3p2_scale1_level"] and vals[0, 1] == 6.0


def test_mxfp4_decoder_spec_points():
    # OCP MX: UE8M0 scale 2^(e - 127) per block of 32 E2M1 elements; e = 255 is NaN
    codes = np.zeros((1, 64), np.uint8)  # 128 elements
    codes[0, 0] = 0x7 | (0xA << 4)       # el 0 = +6, el 1 = -1.0
    codes[0, 16] = 0x1                    # el 32 = +0.5
    codes[0, 63] = 0x30                   # el 127 = +1.5
    v = O.mxfp4_to_f64(codes, np.array([[127, 130, 0, 255]], np.uint8))
    assert v[0, 0] == 6.0 and v[0, 1] == -1.0 and v[0, 2:32].tolist() == [0.0] * 30
    assert v[0, 32] == 0.5 * 8.0  # the second block scales by 2^3
    assert v[0, 64] == 0.0 and np.all(np.isnan(v[0, 96:]))  # 2^-127 * 0; the NaN block
    # every code with a unit scale is its E2M1 level (low nibble = even element)
    allc = np.arange(256, dtype=np.uint8)[None, :32].repeat(2, 0).reshape(1, 64)
    vv = O.mxfp4_to_f64(allc, np.array([[127, 127, 127, 127]], np.uint8))
    assert np.array_equal(vv[0, 0::2], O.e2m1_to_f64(allc[0] & 0xF)) and np.array_equal(vv[0, 1::2], O.e2m1_to_f64(allc[0] >> 4))


def test_fp8_row_scale():
    codes = np.array([[0x38, 0xB8, 0x7E]], np.uint8)
    v = O.fp8_rows_to_f64(codes, np.array([0.25], np.float32))
    assert v.tolist() == [[0.25, -0.25, 112.0]]


# ================================================================ cache writer
def test_writer_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(100_000) * rng.choice([1e-3, 1.0, 100.0], 100_000)).astype(np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, -(2.0 ** -10), 464.0, 1000.0])])
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_round(x), ref)


def test_writer_e2m1_page_example_levels_and_ties():
    g = gold("fp4_course_lesson.json")
    # the lesson's example: 3.2 at scale 1 stores level 3 and reads back 3.0 (error -0.2)
    c = O.e2m1_round(np.float32([3.2]))
    assert O.e2m1_to_f64(c)[0] == g["store_3p2_scale1_level"]
    assert abs(float(O.e2m1_to_f64(c)[0]) - 3.2 - (-0.2)) < 1e-6
    # every level is its own code, with either sign
    lev = np.float32(g["e2m1_magnitudes"])
    assert np.array_equal(O.e2m1_to_f64(O.e2m1_round(lev)), lev)
    assert np.array_equal(O.e2m1_to_f64(O.e2m1_round(-lev[1:])), -lev[1:])
    # midpoints go to the even code; beyond 6 saturates
    mids = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 9.0])
    assert O.e2m1_to_f64(O.e2m1_round(mids)).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0]
    # nearest level off the midpoints (brute force)
    q = np.linspace(-7, 7, 2801).astype(np.float32)
    q = q[~np.isin(np.abs(q), mids)]
    got = O.e2m1_to_f64(O.e2m1_round(q))
    allv = np.concatenate([lev, -lev])
    ref = allv[np.argmin(np.abs(q[:, None].astype(np.float64) - allv[None, :]), axis=1)]
    assert np.array_equal(got, ref)


def test_writer_fp4_scale_rule_and_error_bound():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((64, 512)) * np.exp2(rng.integers(-12, 8, (64, 1)))).astype(np.float32)
    x[3] = 0.0
    for group in (16, 32):
        codes, scodes = O.fp4_quantize(x, group)
        assert codes.shape == (64, 256) and scodes.shape == (64, 512 // group)
        amax = np.abs(x.reshape(64, -1, group)).max(-1).astype(np.float64)
        sval = O.e4m3_to_f64(scodes)
        prev = O.e4m3_to_f64(np.maximum(scodes.astype(np.int64) - 1, 0).astype(np.uint8))
        s = (amax.astype(np.float32) / np.float32(6.0)).astype(np.float64)
        # the smallest E4M3 value at or above amax / 6
        assert np.all(sval >= s) and np.all((scodes == 0) | (prev < s))
        deq = O.fp4_to_f64(codes, scodes, group)
        # no clipping; every value within half a level step of the scaled grid (step <= 2)
        err = np.abs(deq - x.astype(np.float64)).reshape(64, -1, group)
        assert np.all(err <= sval[..., None] * 1.0 + 1e-30)
        assert np.all(deq[3] == 0.0)
        # groups on an exact grid (level x scale, one element at +-6 x scale, so the group's
        # scale is that scale) come back code for code
        sc = rng.integers(8, 110, (64, 512 // group)).astype(np.uint8)
        lv = rng.integers(0, 16, (64, 512)).astype(np.uint8)
        lv[lv == 8] = 0  # no negative zero
        lv.reshape(64, -1, group)[..., 0] = rng.choice([7, 15], (64, 512 // group))
        grid = (O.e2m1_to_f64(lv) * np.repeat(O.e4m3_to_f64(sc), group, -1)).astype(np.float32)
        c2, s2 = O.fp4_quantize(grid, group)
        assert np.array_equal(s2, sc)
        assert np.array_equal(c2, (lv[:, 0::2] | (lv[:, 1::2] << 4)).astype(np.uint8))


def test_writer_fp8_rows_round_trip():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((32, 512)) * 3).astype(np.float32)
    x[5] = 0.0
    codes, scale = O.fp8_quantize_rows(x)
    assert np.array_equal(scale[5:6], np.float32([1.0]))
    assert np.allclose(scale[:5], np.abs(x[:5]).max(-1) / 448, rtol=1e-7)
    deq = O.fp8_rows_to_f64(codes, scale)
    # relative error of E4M3 (3 mantissa bits) at most 2^-4 of each value, plus the subnormal step
    assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0 ** -4 + scale[:, None] * 2.0 ** -10)
    assert np.all((codes[:5] & 0x7F).max(-1) == 0x7E)  # each row's largest magnitude is 448


def test_writer_rotation_is_rope_in_float32():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((8, 512)).astype(np.float32)
    pos = np.array([0, 1, 7, 100, 4095, 65536, 1_000_000, 2_000_000])
    r = O.rotate_f32(x, pos, 10000.0)
    ref = np.stack([O.rope(x[i].astype(np.float64), int(pos[i]), 10000.0, 64) for i in range(8)])
    assert np.array_equal(r[:, :448], x[:, :448])
    assert np.allclose(r, ref, rtol=0, atol=1e-5)
    assert np.array_equal(r[0], x[0])  # position 0 turns nothing
    # float32 products and sums exactly as written
    c = np.cos(np.float64(100) * 10000.0 ** (-2.0 * 3 / 64)).astype(np.float32)
    sn = np.sin(np.float64(100) * 10000.0 ** (-2.0 * 3 / 64)).astype(np.float32)
    assert r[3, 454] == (x[3, 454] * c) - (x[3, 455] * sn)


# ================================================================ compressor
def test_compressor_special_cases_and_invariants():
    rng = np.random.default_rng(21)
    kv = rng.standard_normal((10, 512))
    gate = rng.standard_normal((10, 512)) * 3
    # ratio 1: no pooling (softmax over one token is 1)
    assert np.allclose(O.compress(kv, gate, 1), kv, rtol=0, atol=0)
    # equal gates: the mean of the pair; an odd tail yields no entry
    e = O.compress(kv[:9], np.zeros((9, 512)), 2)
    assert e.shape == (4, 512) and np.allclose(e, (kv[0:8:2] + kv[1:8:2]) / 2, rtol=0, atol=1e-15)
    # per channel, the entry lies between its two tokens (a convex combination) ...
    e2 = O.compress(kv, gate, 2)
    lo = np.minimum(kv[0::2], kv[1::2]); hi = np.maximum(kv[0::2], kv[1::2])
    assert np.all(e2 >= lo - 1e-12) and np.all(e2 <= hi + 1e-12)
    # ... with the two-token softmax weight, channel by channel
    w0 = 1.0 / (1.0 + np.exp(gate[1::2] - gate[0::2]))
    assert np.allclose(e2, w0 * kv[0::2] + (1 - w0) * kv[1::2], rtol=1e-12, atol=1e-12)
    # a dominant gate picks its token
    g = np.zeros((2, 512)); g[1, :256] = 60.0; g[0, 256:] = 60.0
    one = O.compress(kv[:2], g, 2)[0]
    assert np.allclose(one[:256], kv[1, :256]) and np.allclose(one[256:], kv[0, 256:])
    # adding a per-channel constant to both gates changes nothing
    assert np.allclose(O.compress(kv, gate + rng.standard_normal(512), 2), e2, rtol=1e-12, atol=1e-12)


def test_compressor_causal_visibility():
    # an entry is visible once both its tokens are: positions 0 1 2 3 4 -> 0 1 1 2 2 entries
    assert O.visible_entries(np.arange(5), 2).tolist() == [0, 1, 1, 2, 2]
    assert O.visible_entries(np.arange(4), 1).tolist() == [1, 2, 3, 4]


# ================================================================ indexer score
def test_index_score_hand_case():
    q = np.array([[1.0, 2.0], [-1.0, 0.0]])
    k = np.array([[3.0, 1.0], [1.0, -1.0], [-2.0, -1.0]])
    w = np.array([0.5, 2.0])
    # head 0 dots 5, -1, -4; head 1 dots -3, -1, 2 -> 0.5*5, 0, 2*2
    assert O.index_scores(q, w, k).tolist() == [2.5, 0.0, 4.0]


def test_index_score_one_hot_weight_is_relu_dot():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((50, 128))
    for h in (0, 7, 31):
        w = np.zeros(32)
        w[h] = 1.0
        ref = np.array([max(0.0, float(np.dot(q[h], kj))) for kj in k])
        assert np.allclose(O.index_scores(q, w, k), ref, rtol=1e-13, atol=1e-13)


def test_index_score_all_negative_dots_give_zero():
    q = np.ones((4, 8))
    k = -np.ones((3, 8))
    assert np.all(O.index_scores(q, np.ones(4), k) == 0.0)


# ================================================================ top-K
def test_topk_select_values_cases():
    for c in gold("select_values_course06.json")["cases"]:
        order = O.topk_order(c["scores"], c["k"])
        assert order.tolist() == c["positions_desc"]
        assert [c["values"][i] for i in order] == c["values_read"]
        assert O.topk_set(c["scores"], c["k"]).tolist() == sorted(c["positions_desc"])


def test_topk_matches_rank_definition_bruteforce():
    rng = np.random.default_rng(2)
    for trial in range(300):
        n = int(rng.integers(1, 24))
        k = int(rng.integers(1, 30))
        s = rng.integers(-3, 4, n).astype(np.float64)  # many ties
        # j is selected iff fewer than k entries precede it in (score desc, index asc)
        expect = [j for j in range(n)
                  if sum(1 for i in range(n) if s[i] > s[j] or (s[i] == s[j] and i < j)) < k]
        assert O.topk_set(s, k).tolist() == expect


def test_topk_special_cases():
    assert O.topk_set(np.zeros(10), 4).tolist() == [0, 1, 2, 3]
    assert O.topk_set(np.array([1.0, 5.0]), 8).tolist() == [0, 1]
    assert O.topk_set(np.array([0.0, -0.0, -1.0]), 1).tolist() == [0]
    assert O.topk_set(np.array([-0.0, 0.0, -1.0]), 1).tolist() == [0]


# ================================================================ block pool
def test_block_pool_course_toy():
    g = gold("hierarchical_toy_course07.json")
    s = np.full(g["n_positions"], 0.1)
    s[6] = 0.9   # block [5-8] (1-based)
    s[17] = 0.8  # block [17-20]
    s[0] = 0.5
    s[23] = 0.4
    pool, bm, kept = O.block_pool(s, g["block_size"], g["n_keep"])
    assert (pool + 1).tolist() == g["pool_1based"]
    assert kept.tolist() == [1, 4]


def test_block_pool_invariants():
    rng = np.random.default_rng(3)
    for trial in range(100):
        n = int(rng.integers(1, 300))
        bs = int(rng.integers(1, 17))
        nk = int(rng.integers(1, 12))
        s = rng.integers(-5, 6, n).astype(np.float64)
        pool, bm, kept = O.block_pool(s, bs, nk)
        nb = (n + bs - 1) // bs
        assert len(bm) == nb
        for c in range(nb):
            assert bm[c] == s[c * bs:min(n, (c + 1) * bs)].max()
        dropped = np.setdiff1d(np.arange(nb), kept)
        if len(dropped) and len(kept):
            assert bm[kept].min() >= bm[dropped].max()
        assert int(np.argmax(bm)) in kept.tolist()
        assert np.all(np.diff(pool) > 0) and pool.max() < n
        if nk * bs >= n:
            assert pool.tolist() == list(range(n))
    s = rng.standard_normal(200)
    pool, _, _ = O.block_pool(s, 1, 17)
    assert pool.tolist() == O.topk_set(s, 17).tolist()


def test_hierarchy_scored_positions_count():
    g = gold("hierarchy_count_v41.json")
    assert g["n_keep_blocks"] * g["block_size"] == g["pool_positions"]
    got = O.scored_positions(g["n_visible"], g["n_later"], g["n_keep_blocks"], g["block_size"])
    assert got == g["scored"]
    assert round(g["five_full_scans"] / got, 2) == g["ratio_printed"]


# ================================================================ RoPE
def test_rope_page_pair():
    g = gold("rope_v4_pair_toy.json")
    x = np.array([0.0, 0.0] + g["pair"])  # D=4, rotary on the last 2
    y = O.rope(x, 3, 1e4, 2)
    assert abs(y[2] - g["rotated"][0]) <= g["tol"] and abs(y[3] - g["rotated"][1]) <= g["tol"]
    assert y[0] == 0.0 and y[1] == 0.0


def test_rope_frequencies_and_placement():
    # theta^(-2i/64) at theta=1e4: pair 24 turns 1e-3 rad per position, pair 8 turns 0.1
    D, R = 512, 64
    x = np.zeros(D)
    x[:D - R] = 7.0
    x[D - R + 2 * 24] = 1.0
    x[D - R + 2 * 8 + 1] = 1.0
    y = O.rope(x, 1000, 1e4, R)
    assert np.all(y[:D - R] == 7.0)
    assert abs(y[D - R + 48] - math.cos(1.0)) < 1e-12 and abs(y[D - R + 49] - math.sin(1.0)) < 1e-12
    # (0, 1) turned by 100 rad -> (-sin 100, cos 100)
    assert abs(y[D - R + 16] + math.sin(100.0)) < 1e-10 and abs(y[D - R + 17] - math.cos(100.0)) < 1e-10


def test_rope_inverse_norm_and_relative_position():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(512)
    k = rng.standard_normal(512)
    for p in (0, 5, 2047, 1048576):
        qp = O.rope(q, p, 1e4, 64)
        assert np.allclose(O.rope(qp, p, 1e4, 64, sign=-1), q, atol=1e-9)
        assert abs(np.linalg.norm(qp) - np.linalg.norm(q)) < 1e-9
    d1 = O.rope(q, 100, 1e4, 64) @ O.rope(k, 40, 1e4, 64)
    d2 = O.rope(q, 1100, 1e4, 64) @ O.rope(k, 1040, 1e4, 64)
    assert abs(d1 - d2) < 1e-9
    assert abs(d1 - q @ k) > 1e-3  # the rotation is not the identity


# ================================================================ sink softmax and attention
@pytest.mark.parametrize("name", ["sink_softmax_v4_swa_toy.json", "sink_softmax_v4_csa_toy.json"])
def test_sink_softmax_page_values(name):
    g = gold(name)
    z = np.array(g["logits"]) if "logits" in g else g["scale"] * np.array(g["qk"])
    p, sm = O.sink_softmax(z, g["sink"])
    assert np.all(np.abs(p - np.array(g["weights"])) <= g["tol"])
    assert abs(sm - g["sink_mass"]) <= g["tol"]
    assert p.sum() + sm == pytest.approx(1.0, abs=1e-15)
    if "denominator" in g:
        assert abs(np.exp(z).sum() + math.exp(g["sink"]) - g["denominator"]) <= g["tol"]


def test_sink_lowers_mass_below_one():
    rng = np.random.default_rng(5)
    z = rng.standard_normal(640)
    p, sm = O.sink_softmax(z, 0.3)
    assert 0.0 < sm < 1.0 and p.sum() < 1.0
    p, sm = O.sink_softmax(z, -np.inf)
    assert sm == 0.0 and abs(p.sum() - 1.0) < 1e-14


def test_attend_course_two_query_example():
    g = gold("reuse_two_query_course06.json")
    K, V = np.array(g["keys"], float), np.array(g["values"], float)
    q = np.array([g["query_A"], g["query_B"]], float)
    o, sm = O.attend(q, K, V, g["scale"], np.array([-np.inf, -np.inf]))
    z = g["scale"] * (q[0] @ K.T)
    pA, _ = O.sink_softmax(z, -np.inf)
    assert np.all(np.abs(pA - g["weights_A"]) <= g["tol"])
    assert np.all(np.abs(o[0] - g["output_A"]) <= g["tol"])
    assert np.all(np.abs(o[1] - g["output_B"]) <= g["tol"])
    assert np.all(sm == 0.0)


def test_attend_dense_special_case_matches_torch_sdpa():
    rng = np.random.default_rng(6)
    H, D, n = 8, 64, 37
    q = rng.standard_normal((H, D))
    kv = rng.standard_normal((n, D)) / 8
    o, _ = O.attend(q, kv, kv, D ** -0.5, np.full(H, -np.inf))
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(kv), torch.from_numpy(kv), scale=D ** -0.5)
    assert np.allclose(o, t.numpy(), rtol=1e-12, atol=1e-12)


def test_attention_row_closed_form_constant_rows():
    # all rows equal c with a zero rotary part: o_h = (1 - sigma_h) c
    H, D, R = 4, 512, 64
    rng = np.random.default_rng(7)
    c = rng.standard_normal(D) / 16
    c[D - R:] = 0.0
    q = rng.standard_normal((H, D))
    sink = rng.standard_normal(H)
    sel = np.tile(c, (5, 1))
    swa = np.tile(c, (3, 1))
    o, sm = O.csa2_attention_row(q, 1234, sel, swa, sink, 1e4, R, D ** -0.5)
    z = D ** -0.5 * (q @ c)
    sigma = np.exp(sink) / (8 * np.exp(z) + np.exp(sink))
    assert np.allclose(sm, sigma, rtol=1e-12)
    assert np.allclose(o, (1 - sigma)[:, None] * c[None, :], rtol=1e-12, atol=1e-15)


def test_attention_row_is_rope_sdpa_inverse_rope_without_sink():
    rng = np.random.default_rng(8)
    H, D, R = 6, 512, 64
    q = rng.standard_normal((H, D))
    sel = rng.standard_normal((9, D)) / 20
    swa = rng.standard_normal((4, D)) / 20
    pos = 777
    o, sm = O.csa2_attention_row(q, pos, sel, swa, np.full(H, -np.inf), 1e4, R, D ** -0.5)
    kv = np.concatenate([sel, swa])
    qr = O.rope(q, pos, 1e4, R)
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr), torch.from_numpy(kv), torch.from_numpy(kv), scale=D ** -0.5).numpy()
    assert np.allclose(o, O.rope(t, pos, 1e4, R, sign=-1), rtol=1e-11, atol=1e-13)
    assert not np.allclose(o, t, atol=1e-6)  # the output rotation is applied


# ================================================================ drivers: invariants of the step
def _small(name, **kw):
    return synth.make_inputs(synth.scaled(synth.WORKLOADS[name], **kw), seed=11)


def test_causality_future_records_and_window_do_not_matter():
    inp = _small("tiny_decode", N=700)
    inp["rows"]["n_visible"][:] = 600
    base = O.csa2_group(inp)[0]
    c = inp["cache"]
    c["k_idx"][:, 600:] = c["k_idx"][:, 600:][:, ::-1]
    c["lat"][:, 600:] ^= np.uint16(0x0101)
    again = O.csa2_group(inp)[0]
    assert np.array_equal(base["idx"], again["idx"])
    assert np.array_equal(base["o"], again["o"])
    assert base["idx"].max() < 600


def test_window_rows_outside_the_window_do_not_matter():
    wl = synth.scaled(synth.WORKLOADS["prefill_chunk"], N=900, T=20, P0=880)
    inp = synth.make_inputs(wl, seed=3)
    rows = [0, 5, 19]
    base = O.csa2_group(inp, rows=rows)[0]
    swa = inp["layers"][0]["swa"]
    # row t=0 (position 880) sees window positions 753..880 = buffer rows 0..127
    swa[0, 128:] ^= np.uint16(0x1111)
    r0 = O.csa2_layer(inp, 0, rows=[0])
    assert np.array_equal(r0["o"][0], base["o"][0])


def test_reuse_same_indices_different_queries_differ():
    inp = _small("hierarchical", N=3000, B=2)
    res = O.csa2_group(inp)
    r4, r5 = res[4], res[5]
    assert r4["mode"] == "reuse" and r5["mode"] == "reuse"
    assert np.array_equal(r4["idx"], r5["idx"]) and np.array_equal(r4["idx"], res[3]["idx"])
    rms = np.sqrt(np.mean(r4["o"] ** 2))
    assert np.max(np.abs(r4["o"] - r5["o"])) > 0.1 * rms
    # same query, same indices -> identical output
    inp["layers"][5]["q"] = inp["layers"][4]["q"]
    inp["layers"][5]["swa"] = inp["layers"][4]["swa"]
    inp["layers"][5]["sink"] = inp["layers"][4]["sink"]
    again = O.csa2_layer(inp, 5, res[4])
    assert np.array_equal(again["o"], r4["o"])


def test_pool_covering_everything_makes_reindex_equal_full():
    inp = _small("hierarchical", N=1000, B=2, n_keep=16, block_size=64)
    inp["layers"][1]["q_idx"] = inp["layers"][0]["q_idx"]
    inp["layers"][1]["w"] = inp["layers"][0]["w"]
    res = O.csa2_group(inp)
    assert np.array_equal(res[0]["pool"][:, :1000], np.tile(np.arange(1000), (2, 1)))
    assert np.array_equal(res[1]["idx"], res[0]["idx"])


def test_grid_mode_scores_are_exact_integers_over_16():
    inp = _small("tiny_decode", N=500)
    g = synth.make_inputs(synth.scaled(synth.WORKLOADS["tiny_decode"], N=500), seed=2, mode="grid")
    s = O.index_scores_rows(g, 0)
    assert np.all(s * 16 == np.round(s * 16))
    assert np.all(np.abs(s) < 2 ** 16)
    assert inp["params"]["mode"] == "gauss"


# ================================================================ projections
def test_rms_norm_closed_form():
    # [3, 4]: mean square 12.5
    y = O.rms_norm([3.0, 4.0], eps=0.0)
    assert np.allclose(y, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    assert np.allclose(O.rms_norm([3.0, 4.0], [2.0, 0.5], eps=0.0), [0.8485281374238570 * 2, 1.1313708498984760 * 0.5])
    # eps enters under the root: mean square 12.5 + eps 12.5 -> divide by 5
    assert np.allclose(O.rms_norm([3.0, 4.0], eps=12.5), [0.6, 0.8], rtol=0, atol=1e-15)
    # normalized over the last axis only
    v = np.array([[3.0, 4.0], [30.0, 40.0]])
    assert np.allclose(O.rms_norm(v, eps=0.0)[0], O.rms_norm(v, eps=0.0)[1])


def _toy_query_weights():
    # hidden 3 -> rank 2 -> 2 heads of 2
    w_dq = np.array([[1.0, 0.0, 0.0], [0.0, 1.0, 1.0]])
    w_uq = np.array([[1.0, 0.0], [0.0, 1.0],      # head 0 = c
                     [2.0, 0.0], [0.0, 0.0]])     # head 1 = (2 c0, 0)
    return w_dq, w_uq


def test_query_proj_hand_worked():
    w_dq, w_uq = _toy_query_weights()
    x = np.array([[1.0, 2.0, 2.0]])               # c = (1, 4), mean square 8.5
    q = O.query_proj(x, w_dq, None, w_uq, None, n_heads=2, eps=0.0)
    assert q.shape == (1, 2, 2)
    assert np.allclose(q[0, 0], [1 / math.sqrt(8.5), 4 / math.sqrt(8.5)], atol=1e-14)
    assert np.allclose(q[0, 1], [math.sqrt(2.0), 0.0], atol=1e-14)
    # the rank gain acts before the up-projection: c * g = (1, 8) -> head 0 = (1, 8) / sqrt(32.5)
    q = O.query_proj(x, w_dq, [1.0, 2.0], w_uq, None, n_heads=2, eps=0.0)
    assert np.allclose(q[0, 0], [1 / math.sqrt(32.5), 8 / math.sqrt(32.5)], atol=1e-14)
    # the head gain acts last, per coordinate of every head
    q = O.query_proj(x, w_dq, None, w_uq, [1.0, -3.0], n_heads=2, eps=0.0)
    assert np.allclose(q[0, 0], [1 / math.sqrt(8.5), -12 / math.sqrt(8.5)], atol=1e-14)
    # eps in both norms: c / sqrt(8.5 + 8.5) = (1, 4) / sqrt(17); head 0 has mean square 1/2,
    # so it is divided by sqrt(0.5 + 8.5) = 3
    q = O.query_proj(x, w_dq, None, w_uq, None, n_heads=2, eps=8.5)
    assert np.allclose(q[0, 0], [1 / math.sqrt(17) / 3, 4 / math.sqrt(17) / 3], atol=1e-14)


def test_query_proj_invariants():
    rng = np.random.default_rng(5)
    T, d, r, H, D = 4, 64, 32, 3, 16
    x = rng.standard_normal((T, d))
    w_dq = rng.standard_normal((r, d))
    w_uq = rng.standard_normal((H * D, r))
    g_q = rng.uniform(0.5, 1.5, r)
    q = O.query_proj(x, w_dq, g_q, w_uq, None, H, eps=0.0)
    # every head has unit RMS; a per-token scale of x and a scale of either weight cancel
    assert np.allclose(np.sqrt(np.mean(q ** 2, -1)), 1.0, atol=1e-12)
    assert np.allclose(O.query_proj(7.0 * x, w_dq, g_q, w_uq, None, H, eps=0.0), q, atol=1e-12)
    assert np.allclose(O.query_proj(x, 0.25 * w_dq, g_q, 3.0 * w_uq, None, H, eps=0.0), q, atol=1e-12)
    # heads are independent: head 1's rows of w_uq do not change head 0
    w2 = w_uq.copy()
    w2[D:2 * D] = rng.standard_normal((D, r))
    q2 = O.query_proj(x, w_dq, g_q, w2, None, H, eps=0.0)
    assert np.allclose(q2[:, 0], q[:, 0], atol=1e-12) and not np.allclose(q2[:, 1], q[:, 1])
    # with eps 0 and unit gains the path is the normalized product of the two matrices
    ref = x @ w_dq.T
    ref = ref / np.linalg.norm(ref, axis=-1, keepdims=True)
    ref = (ref @ w_uq.T).reshape(T, H, D)
    ref = ref / np.linalg.norm(ref, axis=-1, keepdims=True) * math.sqrt(D)
    assert np.allclose(O.query_proj(x, w_dq, None, w_uq, None, H, eps=0.0), ref, atol=1e-12)


def test_out_proj_hand_worked():
    o = np.array([[[1.0], [2.0], [3.0], [4.0]]])  # 4 heads of 1, groups {0,1} and {2,3}
    w_oa = np.array([[[1.0, 1.0]], [[1.0, -1.0]]])  # group 0 -> 1 + 2 = 3, group 1 -> 3 - 4 = -1
    w_ob = np.array([[1.0, 0.0], [2.0, 3.0]])
    assert np.allclose(O.out_proj(o, w_oa, w_ob), [[3.0, 3.0]], atol=0)


def test_out_proj_is_a_block_diagonal_product():
    import scipy.linalg
    rng = np.random.default_rng(9)
    T, H, D, G, r, d = 3, 8, 4, 4, 5, 6
    o = rng.standard_normal((T, H, D))
    w_oa = rng.standard_normal((G, r, H // G * D))
    w_ob = rng.standard_normal((d, G * r))
    dense = scipy.linalg.block_diag(*list(w_oa))   # [G r, H D]
    ref = (o.reshape(T, H * D) @ dense.T) @ w_ob.T
    assert np.allclose(O.out_proj(o, w_oa, w_ob), ref, atol=1e-12)
    # one group: a plain two-stage low-rank product
    w_oa1 = rng.standard_normal((1, r, H * D))
    assert np.allclose(O.out_proj(o, w_oa1, w_ob[:, :r]), (o.reshape(T, H * D) @ w_oa1[0].T) @ w_ob[:, :r].T)
    # a head only reaches the hidden state through its own group's rank slice
    o2 = o.copy()
    o2[:, 5] += 1.0                                 # head 5 is in group 2 (heads 4, 5)
    w_ob2 = w_ob.copy()
    w_ob2[:, 2 * r:3 * r] = 0.0
    assert np.allclose(O.out_proj(o2, w_oa, w_ob2), O.out_proj(o, w_oa, w_ob2), atol=1e-12)


def test_bf16_round_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(50000) * np.exp2(rng.integers(-30, 30, 50000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_round(x), ref)
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1); 1 + 3 * 2^-8 -> 1 + 2^-6
    t = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], np.float32)
    assert list(O.bf16_round(t)) == [0x3F80, 0x3F82, 0xBF80]


def test_bf16_round_f64_rounds_once():
    rng = np.random.default_rng(22)
    x = rng.standard_normal(20000).astype(np.float32).astype(np.float64)  # float32 values: no double rounding
    assert np.array_equal(O.bf16_round_f64(x), O.bf16_round(x.astype(np.float32)))
    # just above a bf16 tie: float32 would round to the tie first and then to even
    y = np.array([1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8 + 2 ** -30), 1 + 2 ** -8])
    assert list(O.bf16_round_f64(y)) == [0x3F81, 0xBF81, 0x3F80]
    assert list(O.bf16_round(y.astype(np.float32))) == [0x3F80, 0xBF80, 0x3F80]


def test_encoder_memory_positions_causality_and_parts():
    rng = np.random.default_rng(23)
    T = 41  # 20 entries of two tokens; the last token forms no entry
    kv = rng.standard_normal((T, 512)).astype(np.float32)
    gate = rng.standard_normal((T, 512)).astype(np.float32)
    w_ik = (rng.standard_normal((128, 512)) / np.sqrt(512)).astype(np.float32)
    m = O.encoder_memory(kv, gate, 2, w_ik)
    assert m["lat"].shape == (20, 512) and m["k_idx"].shape == (20, 128)
    assert list(m["pos"][:3]) == [1, 3, 5] and int(m["pos"][-1]) == 39
    # an entry becomes visible with its last token
    assert [int(O.visible_entries(p, 2)) for p in (0, 1, 2, 3, 39, 40)] == [0, 1, 1, 2, 20, 20]
    # entries depend only on their own tokens: changing tokens 10.. leaves entries 0..4 alone
    kv2, gate2 = kv.copy(), gate.copy()
    kv2[10:] += 1.0
    gate2[10:] -= 2.0
    m2 = O.encoder_memory(kv2, gate2, 2, w_ik)
    assert np.array_equal(m2["lat"][:5], m["lat"][:5]) and np.array_equal(m2["k_idx"][:5], m["k_idx"][:5])
    assert not np.array_equal(m2["lat"][5], m["lat"][5])
    # the latent row is the entry rotated at its position, within bf16 rounding
    lat = O.bf16_to_f64(m["lat"])
    rot = O.rotate_f32(m["entries"], m["pos"], 10000.0).astype(np.float64)
    assert np.all(np.abs(lat - rot) <= 2.0 ** -8 * np.abs(rot))
    assert np.array_equal(lat[:, :448], O.bf16_to_f64(O.bf16_round(m["entries"][:, :448])))
    # the key is W_IK times the unrotated bf16 entry, within bf16 rounding
    plain = O.bf16_to_f64(O.bf16_round(m["entries"]))
    ref = plain @ w_ik.astype(np.float64).T
    assert np.all(np.abs(O.bf16_to_f64(m["k_idx"]) - ref) <= 2.0 ** -8 * np.abs(ref))
