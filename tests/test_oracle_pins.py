"""Pins of the fp64 oracle against facts the pages and plain mathematics fix.

Nothing here compares the oracle with itself retyped: each check is a closed form, an invariant,
an identity stated on the pages, a special case with a known answer, or a relation between two
differently-shaped computations (paged vs contiguous, permuted vs not). Together they are chosen so
that a dropped term, a flipped sign, a wrong index (head map, token, block) or a transposed operand
in the oracle fails at least one of them.

Sources: opt.ai.kr "FlashDecoding++ async softmax -- theory" s1 and s3 (definition, phi form,
fallback), hwan-h-heo.github.io "Optimizing sparse 3D generation inference" s2.2 (A 1 = 1).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _prob(B, Hq, Hkv, d, scale, L, phi=0.0, lo=-30.0, hi=10.0, dtype=oracle.F32, **kw):
    return oracle.make_problem(batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                               dtype=dtype, scale=scale, phi=phi, lo=lo, hi=hi, max_seq_len=L,
                               **kw)


def _rand_problem(seed, B=2, Hq=4, Hkv=2, d=8, L=37, dtype=oracle.F32):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    sl = rng.integers(1, L + 1, size=B).astype(np.int32)
    return q, k, v, sl


# ------------------------------------------------------------------------------------------
# golden closed forms
# ------------------------------------------------------------------------------------------

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    assert case["cite"]
    if "q_by_head" in case:
        Hq, Hkv = case["num_q_heads"], case["num_kv_heads"]
        q = np.array(case["q_by_head"], dtype=np.float32)[None]          # [1][Hq][d]
        k = np.array(case["k_by_token_head"], dtype=np.float32)[None]    # [1][L][Hkv][d]
        v = np.array(case["v_by_token_head"], dtype=np.float32)[None]
        expected = np.array(case["expected_by_head"], dtype=np.float64)
    else:
        Hq = Hkv = 1
        q = np.array(case["q"], dtype=np.float32)[None]                  # [1][1][d]
        k = np.array(case["k"], dtype=np.float32).reshape(1, -1, 1, q.shape[-1])
        v = np.array(case["v"], dtype=np.float32).reshape(1, -1, 1, q.shape[-1])
        if "expected" in case:
            expected = np.array(case["expected"], dtype=np.float64)
        else:
            e = math.e
            expected = np.array([[eval(case["expected_formula"], {"e": e})]], dtype=np.float64)
    L = k.shape[1]
    d = q.shape[-1]
    prob = _prob(1, Hq, Hkv, d, case["scale"], L)
    out, _ = oracle.attention(prob, q, k, v, np.array([L], np.int32))
    np.testing.assert_allclose(out, expected, rtol=1e-14, atol=1e-14)
    # the method's own steps (any split length, normal and forced-online) reach the same value
    for S in (1, 2, L):
        for mode in (oracle.MODE_NORMAL, oracle.MODE_FORCE_ONLINE):
            res = oracle.split_method(prob, q, k, v, np.array([L], np.int32), S,
                                      (L + S - 1) // S, mode=mode)
            np.testing.assert_allclose(res["out"], expected, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------------------------------------
# closed forms computed independently of the oracle's loop
# ------------------------------------------------------------------------------------------

def test_two_tokens_is_a_logistic_mix():
    """L = 2: w_1 = 1 / (1 + exp(s_2 - s_1)), a closed form with no sum over exponentials."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        qv = float(rng.integers(-4, 5))
        k1, k2 = (float(x) for x in rng.integers(-4, 5, size=2))
        v1, v2 = (float(x) for x in rng.standard_normal(2).astype(np.float32))
        scale = 0.5
        s1, s2 = scale * qv * k1, scale * qv * k2      # exact in binary
        expected = v1 / (1.0 + math.exp(s2 - s1)) + v2 / (1.0 + math.exp(s1 - s2))
        q = np.array([[[qv]]], np.float32)
        k = np.array([[[[k1]], [[k2]]]], np.float32)
        v = np.array([[[[v1]], [[v2]]]], np.float32)
        out, _ = oracle.attention(_prob(1, 1, 1, 1, scale, 2), q, k, v, np.array([2], np.int32))
        assert abs(out[0, 0] - expected) <= 1e-15 * max(1.0, abs(expected))


def test_identity_values_expose_weights():
    """With V rows = unit vectors e_t, out = the weight vector: non-negative, sums to 1, and
    orders like the scores (softmax is monotone)."""
    rng = np.random.default_rng(11)
    L = d = 16
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    k = rng.standard_normal((1, L, 1, d)).astype(np.float32)
    v = np.eye(L, dtype=np.float32).reshape(1, L, 1, d)
    out, _ = oracle.attention(_prob(1, 1, 1, d, 0.25, L), q, k, v, np.array([L], np.int32))
    w = out[0]
    assert (w > 0).all()
    assert abs(w.sum() - 1.0) < 1e-14
    scores = (q[0, 0].astype(np.float64) @ k[0, :, 0].astype(np.float64).T)
    assert (np.argsort(w) == np.argsort(scores)).all()


# ------------------------------------------------------------------------------------------
# invariants
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_convex_hull_and_permutation(seed):
    q, k, v, sl = _rand_problem(seed)
    B, L, Hkv, d = k.shape
    prob = _prob(B, q.shape[1], Hkv, d, 0.3, L)
    out, _ = oracle.attention(prob, q, k, v, sl)
    out = out.reshape(B, q.shape[1], d)
    G = q.shape[1] // Hkv
    for b in range(B):
        for h in range(q.shape[1]):
            vv = v[b, :sl[b], h // G].astype(np.float64)
            assert (out[b, h] >= vv.min(0) - 1e-12).all()
            assert (out[b, h] <= vv.max(0) + 1e-12).all()
    # permuting (k_t, v_t) pairs inside each valid prefix leaves the result unchanged
    rng = np.random.default_rng(100 + seed)
    k2, v2 = k.copy(), v.copy()
    for b in range(B):
        p = rng.permutation(sl[b])
        k2[b, :sl[b]] = k[b, p]
        v2[b, :sl[b]] = v[b, p]
    out2, _ = oracle.attention(prob, q, k2, v2, sl)
    np.testing.assert_allclose(out2.reshape(out.shape), out, rtol=1e-12, atol=1e-14)


def test_head_map_is_floor_division():
    """GQA: query head h reads kv head floor(h / G). Each kv head gets constant V = g + 1, so
    out[h] must equal floor(h / G) + 1 exactly (A 1 = 1 per row)."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, d, L = 2, 8, 2, 4, 9
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    v = np.zeros((B, L, Hkv, d), np.float32)
    for g in range(Hkv):
        v[:, :, g, :] = g + 1
    out, _ = oracle.attention(_prob(B, Hq, Hkv, d, 0.5, L), q, k, v, np.full(B, L, np.int32))
    out = out.reshape(B, Hq, d)
    for h in range(Hq):
        assert np.all(out[:, h] == h // (Hq // Hkv) + 1)


def test_masking_ignores_everything_past_seq_len():
    """Tokens t >= L_b never enter: NaN there changes nothing, and the result equals the same
    problem stored with a cache exactly L_b long."""
    q, k, v, sl = _rand_problem(5, B=3, L=20)
    B, L, Hkv, d = k.shape
    prob = _prob(B, q.shape[1], Hkv, d, 0.4, L)
    kp, vp = k.copy(), v.copy()
    for b in range(B):
        kp[b, sl[b]:] = np.nan
        vp[b, sl[b]:] = np.nan
    out_p, _ = oracle.attention(prob, q, kp, vp, sl)
    assert np.isfinite(out_p).all()
    for b in range(B):
        Lb = int(sl[b])
        pb = _prob(1, q.shape[1], Hkv, d, 0.4, Lb)
        ob, _ = oracle.attention(pb, q[b:b + 1], k[b:b + 1, :Lb].copy(), v[b:b + 1, :Lb].copy(),
                                 np.array([Lb], np.int32))
        np.testing.assert_array_equal(out_p.reshape(B, -1, d)[b], ob)


def test_empty_sequence_gives_zeros():
    q, k, v, sl = _rand_problem(6)
    sl[0] = 0
    B, L, Hkv, d = k.shape
    prob = _prob(B, q.shape[1], Hkv, d, 0.4, L)
    out, _ = oracle.attention(prob, q, k, v, sl)
    assert np.all(out.reshape(B, -1, d)[0] == 0)
    res = oracle.split_method(prob, q, k, v, sl, 4, (L + 3) // 4)
    assert np.all(res["out"].reshape(B, -1, d)[0] == 0)


def test_paged_layout_matches_contiguous():
    """The same logical cache stored through a permuted block table gives identical bits."""
    wl = W.Workload("t", 3, 4, 2, 16, W.BF16, split_len=32, seq_len_range=(5, 70), paged=True,
                    block_size=16, seed=99)
    inp = W.generate(wl)
    B, bs = wl.batch, wl.block_size
    Lmax = int(inp.seq_lens.max())
    kc = np.zeros((B, Lmax, wl.num_kv_heads, wl.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(B):
        for t in range(int(inp.seq_lens[b])):
            blk = inp.block_table[b, t // bs]
            kc[b, t] = inp.k[blk, t % bs]
            vc[b, t] = inp.v[blk, t % bs]
    common = dict(batch=B, num_q_heads=4, num_kv_heads=2, head_dim=16, dtype=oracle.BF16,
                  scale=wl.scale, phi=0.0, lo=-30.0, hi=10.0)
    pc = oracle.make_problem(max_seq_len=Lmax, **common)
    pp = oracle.make_problem(paged=True, block_size=bs, max_blocks_per_seq=inp.max_blocks_per_seq,
                             **common)
    oc, _ = oracle.attention(pc, inp.q, kc, vc, inp.seq_lens)
    op, _ = oracle.attention(pp, inp.q, inp.k, inp.v, inp.seq_lens, block_table=inp.block_table)
    np.testing.assert_array_equal(oc, op)


# ------------------------------------------------------------------------------------------
# the unified-max identity and the split algebra
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(3))
def test_phi_shift_identity(seed):
    """exp(x - max) / sum exp(x - max) == exp(x - phi) / sum exp(x - phi) for any phi where the
    exponentials stay finite (the two formulas of the theory page, s3)."""
    q, k, v, sl = _rand_problem(seed, L=50)
    B, L, Hkv, d = k.shape
    prob = _prob(B, q.shape[1], Hkv, d, 0.35, L)
    ref, _ = oracle.attention(prob, q, k, v, sl)
    for phi in (0.0, -5.0, 20.0, 3.25):
        got = oracle.attention_shifted(prob, q, k, v, sl, shift=phi)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    got = oracle.attention_shifted(prob, q, k, v, sl)       # phi from the problem (0)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("S", [1, 3, 7, 16, 50, 200])
@pytest.mark.parametrize("mode", [oracle.MODE_NORMAL, oracle.MODE_FORCE_FAST,
                                  oracle.MODE_FORCE_ONLINE])
def test_split_steps_equal_definition(S, mode):
    """phi-frame partials per split, optional online recompute, max-rescaled sum == exact
    softmax attention, for any split length (ragged last split) and any fallback pattern."""
    q, k, v, sl = _rand_problem(21, B=3, L=61)
    B, L, Hkv, d = k.shape
    # a window narrow enough that some splits fall back in normal mode
    prob = _prob(B, q.shape[1], Hkv, d, 0.8, L, lo=-1.5, hi=1.5)
    ref, _ = oracle.attention(prob, q, k, v, sl)
    res = oracle.split_method(prob, q, k, v, sl, S, (L + S - 1) // S, mode=mode,
                              want_partials=True)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-14)
    if mode == oracle.MODE_NORMAL:
        fl = res["flags"]
        assert (fl & oracle.FLAG_OUT).any() and not (fl & oracle.FLAG_OUT).all()
        # recomputed splits carry their own max, the others phi
        m = res["part_m"]
        assert np.all(m[(fl & oracle.FLAG_OUT) == 0] == 0.0)


def test_hot_key_needs_the_fallback():
    """A score of ~136 overflows float32 exp: the phi frame alone is not representable in
    float32, while the recomputed split gives the exact answer, dominated by the hot key's V."""
    wl = W.STRESS.replace(batch=2, seq_len=256, split_len=64, stress_frac=0.1)
    inp = W.generate(wl)
    assert inp.hot
    prob = oracle.make_problem(batch=2, num_q_heads=32, num_kv_heads=8, head_dim=128,
                               dtype=oracle.BF16, scale=wl.scale, phi=0, lo=-30, hi=10,
                               max_seq_len=256)
    res = oracle.split_method(prob, inp.q, inp.k, inp.v, inp.seq_lens, 64, 4,
                              want_partials=True)
    ref, _ = oracle.attention(prob, inp.q, inp.k, inp.v, inp.seq_lens)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-14)
    per_group = {}
    for (b, g, j, t) in inp.hot:
        per_group.setdefault((b, g), []).append(t)
    singles = 0
    for (b, g, j, t) in inp.hot:
        h0 = g * wl.group
        f = res["flags"][b * 32 + h0, j]
        assert f & oracle.FLAG_OUT and f & oracle.FLAG_ABOVE
        m = res["part_m"][b * 32 + h0, j]
        assert m > 100.0                                       # its own max frame
        assert m > np.log(np.finfo(np.float32).max)            # exp(m) overflows float32
        if len(per_group[(b, g)]) == 1:                        # one hot key dominates the row
            singles += 1
            vt = W.bf16_bits_to_f32(inp.v[b, t, g]).astype(np.float64)
            np.testing.assert_allclose(ref[b * 32 + h0], vt, rtol=1e-12, atol=1e-12)
    assert singles > 0


# ------------------------------------------------------------------------------------------
# window decisions
# ------------------------------------------------------------------------------------------

def test_window_decisions_closed_form():
    """d = 1, q = 1, scale = 1: the scores are the keys. Splits of 4 tokens:
    split 0 all inside; split 1 holds 10.5 (above); split 2 holds -30.5 (below);
    split 3 holds exactly 10 and -30 (closed window: inside); split 4 holds NaN."""
    keys = [0, 1, -2, 3,   0, 10.5, 0, 0,   0, 0, -30.5, 0,   10, -30, 0, 0,   0, np.nan, 0, 0]
    L = len(keys)
    q = np.ones((1, 1, 1), np.float32)
    k = np.array(keys, np.float32).reshape(1, L, 1, 1)
    prob = _prob(1, 1, 1, 1, 1.0, L)
    flags, margin = oracle.window_flags(prob, q, k, np.array([L], np.int32), 4, 5)
    F = oracle
    assert list(flags[0, 0]) == [0, F.FLAG_OUT | F.FLAG_ABOVE, F.FLAG_OUT | F.FLAG_BELOW, 0,
                                 F.FLAG_OUT | F.FLAG_NAN]
    # phi moves the window: with phi = 2 the key 10.5 is inside (x = 8.5), 12.5 would not be
    prob2 = _prob(1, 1, 1, 1, 1.0, 8, phi=2.0)
    k2 = np.array([10.5, 12.0, 0, 0, 12.5, 0, 0, 0], np.float32).reshape(1, 8, 1, 1)
    f2, _ = oracle.window_flags(prob2, q, k2, np.array([8], np.int32), 4, 2)
    assert list(f2[0, 0]) == [0, F.FLAG_OUT | F.FLAG_ABOVE]
    # the margin is the distance of the closest score to an edge (x = 10 sits on it)
    assert margin[0, 0] == 0.0


def test_split_method_flags_match_window_flags():
    q, k, v, sl = _rand_problem(31, B=2, L=40)
    B, L, Hkv, d = k.shape
    prob = _prob(B, q.shape[1], Hkv, d, 0.9, L, lo=-2.0, hi=2.0)
    S = 8
    f1, _ = oracle.window_flags(prob, q, k, sl, S, 5)
    res = oracle.split_method(prob, q, k, v, sl, S, 5)
    np.testing.assert_array_equal(f1.reshape(-1, 5), res["flags"])


# ------------------------------------------------------------------------------------------
# the split scheduler
# ------------------------------------------------------------------------------------------

def test_plan_closed_form():
    sl = np.array([0, 1, 511, 512, 513, 4096], np.int32)
    nsplit, off, n_units = oracle.plan(sl, 8, 4096, 512)
    assert list(nsplit) == [0, 1, 1, 1, 2, 8]
    assert list(off) == [0, 0, 1, 2, 3, 5, 13]
    assert n_units == 13 * 8
    # every token of every sequence is covered exactly once by [jS, min((j+1)S, L))
    for b, L in enumerate(sl):
        covered = np.zeros(L, int)
        for j in range(nsplit[b]):
            covered[j * 512:min((j + 1) * 512, L)] += 1
        assert (covered == 1).all()


def test_auto_split_len_examples():
    """Hand-worked: 8 x 4096 tokens, 8 kv heads -> 262144 pairs over 4 * 148 = 592 units ->
    443 -> next multiple of 64 = 448, inside [256, 4096]."""
    sl = np.full(8, 4096, np.int32)
    assert oracle.split_len(sl, 8, 4096, 0, 148, 4, 64, 256) == 448
    assert oracle.split_len(sl, 8, 4096, 512, 148, 4, 64, 256) == 512      # fixed is kept
    # tiny totals clamp to the minimum; a huge single sequence clamps to its rounded length
    assert oracle.split_len(np.array([10], np.int32), 1, 4096, 0, 148, 4, 64, 256) == 256
    assert oracle.split_len(np.array([0, 0], np.int32), 8, 4096, 0, 148, 4, 64, 256) == 256
    assert oracle.split_len(np.array([100000], np.int32), 8, 100000, 0, 1, 1, 64, 256) == 100032


def test_stress_injection_is_flagged_and_normal_inputs_are_not():
    wl = W.STRESS.replace(seq_len=1024, split_len=256)
    inp = W.generate(wl)
    assert len(inp.hot) == round(0.02 * 8 * 8 * 4)
    prob = oracle.make_problem(batch=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                               dtype=oracle.BF16, scale=wl.scale, phi=0, lo=-30, hi=10,
                               max_seq_len=1024)
    flags, _ = oracle.window_flags(prob, inp.q, inp.k, inp.seq_lens, 256, 4)
    for (b, g, j, t) in inp.hot:
        assert flags[b, g * wl.group, j] & oracle.FLAG_ABOVE
    hot_units = {(b, g, j) for (b, g, j, t) in inp.hot}
    for b in range(8):
        for h in range(32):
            for j in range(4):
                if (b, h // wl.group, j) not in hot_units:
                    assert flags[b, h, j] == 0


# ------------------------------------------------------------------------------------------
# per-head phi and phi observed in advance (oracle.c, R7 and R8)
# ------------------------------------------------------------------------------------------

def test_per_head_phi_is_each_heads_own_scalar_phi():
    """Per-head phi: head h decides exactly as the scalar-phi replay with phi = phi_h, and the
    method's output is still the exact softmax (phi only moves where splits fall back)."""
    q, k, v, sl = _rand_problem(11, B=2, Hq=4, Hkv=2, d=8, L=40)
    q *= 3.0                                      # scores of a few units: some cross the window
    S, ms = 8, 5
    phis = np.array([-2.0, 0.0, 1.5, 4.0], np.float32)
    prob = _prob(2, 4, 2, 8, 1.0, 40, lo=-6.0, hi=3.0)
    f_heads, _ = oracle.window_flags(prob, q, k, sl, S, ms, phi_heads=phis)
    assert f_heads.any() and not f_heads.all()
    for h, ph in enumerate(phis):
        prob_h = _prob(2, 4, 2, 8, 1.0, 40, phi=float(ph), lo=-6.0, hi=3.0)
        f_h, _ = oracle.window_flags(prob_h, q, k, sl, S, ms)
        np.testing.assert_array_equal(f_heads[:, h], f_h[:, h])
    exact, _ = oracle.attention(prob, q, k, v, sl)
    res = oracle.split_method(prob, q, k, v, sl, S, ms, phi_heads=phis)
    np.testing.assert_allclose(res["out"], exact, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(res["flags"].reshape(f_heads.shape), f_heads)


def test_score_ranges_closed_form():
    """Keys along q give known scores: q = 8 e_0, k_t = c_t e_0, scale 1/8, so s_t = c_t
    exactly (fp32). Each split's range is the min and max of its c_t."""
    L, d, S = 11, 64, 4
    c = np.array([3.0, -1.0, 2.5, 0.0, 7.0, 7.0, -4.0, 1.0, 0.5, -0.5, 9.0], np.float32)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 8.0
    k = np.zeros((1, L, 1, d), np.float32)
    k[0, :, 0, 0] = c
    prob = _prob(1, 1, 1, d, 0.125, L)
    smin, smax = oracle.score_ranges(prob, q, k, np.array([L], np.int32), S, 4)
    np.testing.assert_array_equal(smin[0, 0, :3], [-1.0, -4.0, -0.5])
    np.testing.assert_array_equal(smax[0, 0, :3], [3.0, 7.0, 9.0])
    assert np.isnan(smin[0, 0, 3]) and np.isnan(smax[0, 0, 3])


def test_score_ranges_agree_with_window_decisions():
    """A row-split is inside the window for phi exactly when phi lies in
    [max s - hi, min s - lo]: the ranges and the token-by-token decisions must agree for any
    phi."""
    q, k, v, sl = _rand_problem(12, B=3, Hq=4, Hkv=2, d=16, L=50)
    q *= 2.0
    S, ms, lo, hi = 8, 7, -3.0, 2.0
    prob = _prob(3, 4, 2, 16, 0.25, 50, lo=lo, hi=hi)
    smin, smax = oracle.score_ranges(prob, q, k, sl, S, ms)
    nb = -(-sl // S)
    for phi in (-1.0, 0.0, 0.7, 2.0):
        f, _ = oracle.window_flags(_prob(3, 4, 2, 16, 0.25, 50, phi=phi, lo=lo, hi=hi), q, k, sl,
                                   S, ms)
        for b in range(3):
            for j in range(nb[b]):
                keep = (np.float64(smax[b, :, j]) - hi <= np.float32(phi)) & \
                       (np.float32(phi) <= np.float64(smin[b, :, j]) - lo)
                np.testing.assert_array_equal((f[b, :, j] & oracle.FLAG_OUT) == 0, keep)


def _ranges_from_intervals(intervals, lo, hi):
    """One head, one sequence: row-split ranges whose keep-interval [max - hi, min - lo] is the
    given [a, b] (a > b gives a split that no phi can keep)."""
    smin = np.array([[[b_ + lo for _, b_ in intervals]]], np.float64)
    smax = np.array([[[a_ + hi for a_, _ in intervals]]], np.float64)
    return smin, smax, np.array([len(intervals)], np.int32)


@pytest.mark.parametrize("intervals,phi,kept", [
    ([(0.0, 2.0), (1.0, 3.0), (5.0, 6.0)], 1.5, 2),        # best count 2 on [1, 2]
    ([(0.0, 1.0), (2.0, 4.0)], 3.0, 1),                   # count 1 twice: the wider run wins
    ([(0.0, 1.0), (1.0, 2.0)], 1.0, 2),                   # best count only at the shared point
    ([(0.0, 1.0), (3.0, 4.0)], 0.5, 1),                   # equal widths: the first run
    ([(2.0, 1.0), (4.0, 3.0)], -7.0, 0),                  # no split can be kept: fallback
    ([(0.0, 10.0), (2.0, 3.0), (2.5, 8.0)], 2.75, 3),     # nested intervals
])
def test_pick_phi_examples(intervals, phi, kept):
    lo, hi = -30.0, 10.0
    smin, smax, ns = _ranges_from_intervals(intervals, lo, hi)
    got, k = oracle.pick_phi(smin, smax, ns, lo, hi, fallback=-7.0)
    assert got[0] == pytest.approx(phi, abs=1e-12)
    assert k[0] == kept


@pytest.mark.parametrize("seed", range(5))
def test_pick_phi_is_the_best_count_by_brute_force(seed):
    """Against a dense scan of candidate phi values: no phi keeps more splits than the pick, and
    the picked phi keeps that many."""
    rng = np.random.default_rng(seed)
    lo, hi = -5.0, 2.0
    n = 12
    mid = rng.uniform(-10, 10, n)
    width = rng.uniform(-1, 8, n)
    intervals = [(m - w / 2, m + w / 2) for m, w in zip(mid, width)]
    smin, smax, ns = _ranges_from_intervals(intervals, lo, hi)
    phi, kept = oracle.pick_phi(smin, smax, ns, lo, hi, fallback=0.0)
    a = np.array([i[0] for i in intervals])
    b = np.array([i[1] for i in intervals])
    grid = np.concatenate([np.linspace(-20, 20, 40001), a, b])
    counts = ((a[None, :] <= grid[:, None]) & (grid[:, None] <= b[None, :])).sum(axis=1)
    assert kept[0] == counts.max()
    assert ((a <= phi[0]) & (phi[0] <= b)).sum() == counts.max()


def test_picked_phi_keeps_exactly_the_counted_splits():
    """Calibrating on sample inputs and replaying the decisions with the picked per-head phi
    leaves exactly `kept` row-splits of each head inside the window."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d, L, S = 4, 4, 2, 16, 96, 16
    q = (rng.standard_normal((B, Hq, d)) * np.array([1, 3, 5, 8])[None, :, None]).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    sl = rng.integers(20, L + 1, size=B).astype(np.int32)
    lo, hi = -4.0, 3.0
    prob = _prob(B, Hq, Hkv, d, 0.25, L, lo=lo, hi=hi)
    ms = -(-L // S)
    smin, smax = oracle.score_ranges(prob, q, k, sl, S, ms)
    nb = (-(-sl // S)).astype(np.int32)
    phi, kept = oracle.pick_phi(smin, smax, nb, lo, hi, fallback=0.0)
    f, _ = oracle.window_flags(prob, q, k, sl, S, ms, phi_heads=phi.astype(np.float32))
    for h in range(Hq):
        inside = sum(int((f[b, h, j] & oracle.FLAG_OUT) == 0) for b in range(B) for j in range(nb[b]))
        assert inside == kept[h]


# ------------------------------------------------------------------------------------------
# several query tokens per sequence, causal within the last Tq positions (oracle.c, R9)
# ------------------------------------------------------------------------------------------

def test_query_token_rows_are_decodes_of_shorter_caches():
    """Query token i of a Tq-token chunk is exactly a single-token decode against the first
    L_b - Tq + 1 + i keys: two differently shaped computations must agree."""
    rng = np.random.default_rng(21)
    B, Tq, Hq, Hkv, d, L = 3, 4, 4, 2, 8, 30
    q = rng.standard_normal((B, Tq, Hq, d)).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    sl = np.array([30, 9, 4], np.int32)
    prob = _prob(B, Hq, Hkv, d, 0.5, L, q_tokens=Tq)
    multi, _ = oracle.attention(prob, q.reshape(B * Tq, Hq, d), k, v, sl)
    multi = multi.reshape(B, Tq, Hq, d)
    for i in range(Tq):
        lim = (sl - Tq + 1 + i).astype(np.int32)
        single, _ = oracle.attention(_prob(B, Hq, Hkv, d, 0.5, L), np.ascontiguousarray(q[:, i]), k,
                                     v, lim)
        np.testing.assert_allclose(multi[:, i], single.reshape(B, Hq, d), rtol=0, atol=1e-14)


def test_two_query_tokens_closed_form():
    """L = 2, Tq = 2: the first query token sees key 0 only (out = v_0); the second sees both, a
    logistic mix with weight sigma(s_1 - s_0) on v_1."""
    d = 4
    q = np.array([[[1.0, 0, 0, 0]], [[0.5, 1.0, 0, 0]]], np.float32)      # [Tq][1][d]
    k = np.array([[[[2.0, 0, 0, 0]], [[0, 3.0, 0, 0]]]], np.float32)       # [1][2][1][d]
    v = np.array([[[[1.0, 2.0, 3.0, 4.0]], [[-1.0, 0.5, 0.0, 2.0]]]], np.float32)
    prob = _prob(1, 1, 1, d, 1.0, 2, q_tokens=2)
    out, _ = oracle.attention(prob, q, k, v, np.array([2], np.int32))
    np.testing.assert_allclose(out[0], v[0, 0, 0], rtol=0, atol=0)
    s0, s1 = 0.5 * 2.0, 1.0 * 3.0
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    v64 = v.astype(np.float64)
    np.testing.assert_allclose(out[1], (1 - w1) * v64[0, 0, 0] + w1 * v64[0, 1, 0], rtol=1e-14)


def test_query_tokens_split_method_and_decisions():
    """The method's steps with Tq query tokens equal the definition, and their decisions equal
    the window replay, including splits that hold none of an early row's keys. A sequence
    shorter than Tq leaves its first rows with no key: zero rows."""
    rng = np.random.default_rng(22)
    B, Tq, Hq, Hkv, d, L, S = 3, 3, 4, 2, 8, 33, 8
    q = (rng.standard_normal((B * Tq, Hq, d)) * 2.5).astype(np.float32)
    k = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((B, L, Hkv, d)).astype(np.float32)
    sl = np.array([33, 17, 2], np.int32)                 # 17 = 2 S + 1: an empty last split
    prob = _prob(B, Hq, Hkv, d, 0.5, L, lo=-4.0, hi=3.0, q_tokens=Tq)
    ms = -(-L // S)
    exact, _ = oracle.attention(prob, q, k, v, sl)
    res = oracle.split_method(prob, q, k, v, sl, S, ms)
    np.testing.assert_allclose(res["out"], exact, rtol=1e-12, atol=1e-12)
    f, _ = oracle.window_flags(prob, q, k, sl, S, ms)
    np.testing.assert_array_equal(res["flags"].reshape(f.shape), f)
    assert f.any()
    # sequence 2 has 2 keys for 3 query tokens: its first query row sees none
    np.testing.assert_array_equal(exact.reshape(B, Tq, Hq, d)[2, 0], 0.0)
    assert np.abs(exact.reshape(B, Tq, Hq, d)[2, 1]).sum() > 0


@pytest.mark.parametrize("tile", [1, 3, 16, 64])
def test_inplace_finish_is_the_online_softmax(tile):
    """oracle.c R11: a row that continues in place with the running max from its first tile holding
    a score outside the window ends with the softmax of the plain definition (scipy's softmax
    here, a library routine), whatever the tile size; a row whose scores all stay inside keeps the
    phi frame (m = phi, l = sum exp(s - phi)); and the frame it ends in is the running max over
    phi (when some sum was held before the switch) and the scores from the switching tile on."""
    from scipy.special import softmax
    rng = np.random.default_rng(100 + tile)
    phi, lo, hi = 0.0, -30.0, 10.0
    switched = 0
    for trial in range(240):
        n, d = int(rng.integers(1, 200)), 4
        s = rng.standard_normal(n) * 3.0
        kind = trial % 4
        if kind == 1:                                   # one score far above phi + hi
            s[int(rng.integers(0, n))] += 40.0
        elif kind == 2:                                 # every score far below phi + lo
            s -= 45.0
        elif kind == 3:                                 # a few scores far below phi + lo
            s[rng.integers(0, n, size=3)] -= 60.0
        v = rng.standard_normal((n, d))
        o, l, m, sw = oracle.inplace_partial(s, v, tile, phi, lo, hi)
        np.testing.assert_allclose(o / l, softmax(s) @ v, rtol=1e-10, atol=1e-12)
        inside = (s - phi >= lo) & (s - phi <= hi)
        assert sw == (not inside.all())
        if not sw:
            assert m == phi
            np.testing.assert_allclose(l, math.fsum(np.exp(s - phi)), rtol=1e-13)
        else:
            switched += 1
            first = int(np.argmin(inside)) // tile * tile        # the switching tile's first token
            held = first > 0
            expect_m = max(([phi] if held else []) + list(s[first:]))
            assert m == expect_m
            np.testing.assert_allclose(l, math.fsum(np.exp(s - m)), rtol=1e-12)
    assert switched >= 120
