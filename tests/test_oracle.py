"""Pins for the CPU oracle, checked against facts the pages and mathematics fix.

None of these re-type the oracle's formula: each checks a closed form, an
invariant, a special case or an independent high-precision evaluation, chosen
so that a plausible slip in the oracle (a dropped max subtraction, a wrong
sign, an off-by-one in the attended range, a transposed operand, a wrong
GQA head mapping, a wrong scale, a broken chunk merge) fails one of them.

Definitions followed: realizar 0.8.5, src/cuda/executor/head_dim.rs,
``flash_decoding_attention_into`` (PAR-118) -- doc comment, Step 1 (scatter),
"Update cache lengths" (rows 0..pos), Step 3 (chunk count).
"""
import decimal
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "softmax_closed_forms.json")


def _rand(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


# ---------------------------------------------------------------- golden cases
@pytest.mark.parametrize("name", ["weights_1_2_3", "seq_len_one", "identical_keys"])
def test_golden_closed_forms(name):
    case = json.load(open(GOLDEN))["cases"][name]
    q = np.array(case["q"], np.float32)
    K = np.array(case["K"], np.float32)
    V = np.array(case["V"], np.float32)
    out64 = oracle.attend_row(q, K, V, f64=True)
    out32 = oracle.attend_row(q, K, V)
    if case.get("expected_is_input_float32"):
        assert np.array_equal(out32.view(np.int32), V[0].view(np.int32))
        return
    exp = np.array([float(Fraction(e)) for e in case["expected"]])
    err = np.abs(out64 - exp)
    assert np.all(err <= case["atol"] + case["rtol"] * np.abs(exp)), (out64, exp)


# ------------------------------------------------------------- closed forms
@pytest.mark.parametrize("D", [4, 64, 128])
def test_seq_len_one_returns_v_row_exactly(D):
    rng = np.random.default_rng(D)
    q, K, V = _rand(rng, D), _rand(rng, 1, D, scale=5), _rand(rng, 1, D)
    out = oracle.attend_row(q, K, V)
    assert np.array_equal(out.view(np.int32), V[0].view(np.int32))


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(2)
    D, L = 64, 37
    q = _rand(rng, D)
    K = np.repeat(_rand(rng, 1, D), L, axis=0)
    V = _rand(rng, L, D)
    out = oracle.attend_row(q, K, V, f64=True)
    mean = np.array([math.fsum(V[:, d].astype(np.float64)) / L for d in range(D)])
    assert np.max(np.abs(out - mean)) < 1e-14


def test_two_rows_logistic_closed_form():
    # D=4 -> scale 1/2 exactly; q = (a,0,0,0) -> s_j = a*K[j][0]/2 exactly.
    a = 3.0
    K = np.array([[0.75, 9, -9, 9], [-1.25, -7, 7, 1]], np.float32)
    V = np.array([[1.0, -2.0, 0.5, 4.0], [-3.0, 6.0, 0.25, 4.0]], np.float32)
    q = np.array([a, 0, 0, 0], np.float32)
    s0, s1 = a * 0.75 / 2, a * -1.25 / 2
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    exp = w0 * V[0].astype(np.float64) + w1 * V[1].astype(np.float64)
    out = oracle.attend_row(q, K, V, f64=True)
    assert np.max(np.abs(out - exp)) < 1e-14


@pytest.mark.parametrize("jstar", [0, 5, 11])
def test_dominant_row_selects_its_value_row(jstar):
    """One score far above the rest: out = V[j*] (catches index/sign/transpose slips)."""
    rng = np.random.default_rng(jstar)
    D, L = 8, 12
    q = np.zeros(D, np.float32)
    q[3] = 1.0
    K = _rand(rng, L, D)
    K[:, 3] = np.clip(K[:, 3], -1, 1)
    K[jstar, 3] = 200.0  # s = 200/sqrt(8) ~ 70.7 above the rest: weights e^-69 ~ 1e-30
    V = _rand(rng, L, D)
    out = oracle.attend_row(q, K, V, f64=True)
    assert np.max(np.abs(out - V[jstar])) < 1e-25


def test_scale_is_one_over_sqrt_head_dim():
    """Scores t*sqrt(D)/sqrt(D) = t: weights known exactly for D=16 (sqrt exact)."""
    D = 16
    q = np.zeros(D, np.float32)
    q[0] = 1.0
    K = np.zeros((2, D), np.float32)
    K[0, 0] = 4.0 * 1.5  # s0 = 6/4 = 1.5
    V = np.array([np.full(D, 1.0), np.full(D, 0.0)], np.float32)
    out = oracle.attend_row(q, K, V, f64=True)
    w0 = math.exp(1.5) / (math.exp(1.5) + 1.0)
    assert np.max(np.abs(out - w0)) < 1e-15


# ------------------------------------------------- high-precision brute force
def _decimal_attention(q, K, V):
    """Independent 50-digit evaluation: no max subtraction, Decimal exp/sqrt."""
    ctx = decimal.Context(prec=50)
    Dm = decimal.Decimal
    L, D = K.shape
    inv = ctx.divide(Dm(1), ctx.sqrt(Dm(D)))
    w = []
    for j in range(L):
        dot = Dm(0)
        for d in range(D):
            dot = ctx.add(dot, ctx.multiply(Dm(float(q[d])), Dm(float(K[j, d]))))
        w.append(ctx.exp(ctx.multiply(dot, inv)))
    Z = sum(w, Dm(0))
    return np.array([float(ctx.divide(sum((w[j] * Dm(float(V[j, d])) for j in range(L)), Dm(0)), Z))
                     for d in range(D)])


@pytest.mark.parametrize("seed,L,D", [(0, 1, 4), (1, 5, 8), (2, 16, 8), (3, 9, 6)])
def test_brute_force_decimal(seed, L, D):
    rng = np.random.default_rng(100 + seed)
    q, K, V = _rand(rng, D, scale=2), _rand(rng, L, D, scale=2), _rand(rng, L, D)
    out = oracle.attend_row(q, K, V, f64=True)
    ref = _decimal_attention(q, K, V)
    assert np.max(np.abs(out - ref)) <= 1e-13 * max(1.0, np.max(np.abs(ref)))


# ------------------------------------------------------- chunk (split-K) pins
@pytest.mark.parametrize("C", [1, 3, 64, 100, 257, 300])
def test_split_k_merge_equals_definition(C):
    rng = np.random.default_rng(C)
    L, D = 257, 16
    q, K, V = _rand(rng, D), _rand(rng, L, D, scale=3), _rand(rng, L, D)
    direct = oracle.attend_row(q, K, V, f64=True)
    split = oracle.attend_row_split(q, K, V, C)
    assert np.max(np.abs(direct - split)) < 1e-12


def test_split_k_with_outlier_chunk():
    """A chunk whose max dominates the others by ~60: the rescaling must carry it."""
    rng = np.random.default_rng(9)
    L, D = 200, 8
    q = np.zeros(D, np.float32)
    q[0] = 1.0
    K = _rand(rng, L, D)
    K[150, 0] = 170.0
    V = _rand(rng, L, D)
    for C in (7, 64, 128):
        assert np.max(np.abs(oracle.attend_row_split(q, K, V, C) - V[150])) < 1e-20


# ------------------------------------------------------------------ invariants
def test_permutation_invariance():
    rng = np.random.default_rng(5)
    L, D = 50, 32
    q, K, V = _rand(rng, D), _rand(rng, L, D), _rand(rng, L, D)
    perm = rng.permutation(L)
    a = oracle.attend_row(q, K, V, f64=True)
    b = oracle.attend_row(q, K[perm], V[perm], f64=True)
    assert np.max(np.abs(a - b)) < 1e-14
    # permuting V alone (breaking the K/V row pairing) must change the result
    c = oracle.attend_row(q, K, V[perm], f64=True)
    assert np.max(np.abs(a - c)) > 1e-3


def test_linearity_in_v():
    rng = np.random.default_rng(6)
    L, D = 40, 16
    q, K = _rand(rng, D), _rand(rng, L, D)
    V1, V2 = _rand(rng, L, D), _rand(rng, L, D)
    # coefficients that keep 2*V1 - 0.5*V2 exact in float32 are not guaranteed,
    # so compare in double on the (float32) combined input
    Vc = (np.float32(2.0) * V1).astype(np.float32)
    a = oracle.attend_row(q, K, V1, f64=True)
    b = oracle.attend_row(q, K, Vc, f64=True)
    assert np.max(np.abs(2.0 * a - b)) < 1e-14
    s = (V1 + V2).astype(np.float32)
    exact = V1.astype(np.float64) + V2.astype(np.float64) - s.astype(np.float64)
    o12 = oracle.attend_row(q, K, s, f64=True)
    o1 = oracle.attend_row(q, K, V1, f64=True)
    o2 = oracle.attend_row(q, K, V2, f64=True)
    bound = np.max(np.abs(exact)) + 1e-13
    assert np.max(np.abs(o12 - (o1 + o2))) <= bound


def test_output_in_convex_hull_of_v():
    rng = np.random.default_rng(7)
    L, D = 64, 32
    q, K, V = _rand(rng, D, scale=3), _rand(rng, L, D, scale=3), _rand(rng, L, D)
    out = oracle.attend_row(q, K, V, f64=True)
    assert np.all(out >= V.min(axis=0) - 1e-15)
    assert np.all(out <= V.max(axis=0) + 1e-15)


def test_shift_invariance_without_overflow():
    """Adding t to every score leaves the softmax unchanged; with t = 800,
    exp(s) overflows double, so only a max-subtracted evaluation survives."""
    D, L = 4, 6
    rng = np.random.default_rng(8)
    q = np.array([1.0, 0, 0, 0], np.float32)  # s_j = K[j][0] / 2
    K = (np.round(rng.uniform(-4, 4, (L, D)) * 8) / 8).astype(np.float32)
    V = _rand(rng, L, D)
    Ks = K.copy()
    Ks[:, 0] += np.float32(1600.0)  # exact in float32: every score + 800
    a = oracle.attend_row(q, K, V, f64=True)
    b = oracle.attend_row(q, Ks, V, f64=True)
    assert np.all(np.isfinite(b))
    assert np.max(np.abs(a - b)) < 1e-15


# ------------------------------------------------------------------- GQA map
def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(11)
    H, Hkv, D, L = 8, 2, 16, 30
    G = H // Hkv
    q = _rand(rng, H, D)
    K, V = _rand(rng, Hkv, L, D), _rand(rng, Hkv, L, D)
    gqa = oracle.attend_seq(q, K, V, L)
    mha = oracle.attend_seq(q, np.repeat(K, G, axis=0), np.repeat(V, G, axis=0), L)
    assert np.array_equal(gqa, mha)


def test_gqa_query_head_reads_contiguous_group():
    """V of kv head g is the constant g: query head h must output h // G."""
    rng = np.random.default_rng(12)
    H, Hkv, D, L = 12, 3, 8, 10
    q = _rand(rng, H, D)
    K = _rand(rng, Hkv, L, D)
    V = np.stack([np.full((L, D), float(g), np.float32) for g in range(Hkv)])
    out = oracle.attend_seq(q, K, V, L)
    for h in range(H):
        assert np.all(out[h] == h // (H // Hkv))


# ------------------------------------------------------- layout, range, mask
def test_decode_attends_rows_zero_through_position_only():
    rng = np.random.default_rng(13)
    M, H, Hkv, D, Lmax = 3, 4, 2, 8, 20
    pos = np.array([0, 7, 19], np.int32)
    q = _rand(rng, M, H, D)
    Kc, Vc = _rand(rng, M, Hkv, Lmax, D), _rand(rng, M, Hkv, Lmax, D)
    clean = oracle.decode(q, Kc, Vc, pos)
    Kp, Vp = Kc.copy(), Vc.copy()
    for i, p in enumerate(pos):
        Kp[i, :, p + 1:, :] = np.nan
        Vp[i, :, p + 1:, :] = np.nan
    poisoned = oracle.decode(q, Kp, Vp, pos)
    assert np.all(np.isfinite(poisoned))
    assert np.array_equal(clean, poisoned)
    # position 0: the V row itself; the last row is included (dominant-row probe)
    assert np.array_equal(clean[0, 0], Vc[0, 0, 0])
    qd, Kd = q.copy(), Kc.copy()
    qd[1] = 0.0
    qd[1, :, 0] = 1.0
    Kd[1, :, :, 0] = np.clip(Kd[1, :, :, 0], -1, 1)
    Kd[1, :, 7, 0] = 100.0  # row 7 = position of sequence 1: s = 35 vs <= 0.36
    out = oracle.decode(qd, Kd, Vc, pos)
    for h in range(H):
        assert np.max(np.abs(out[1, h] - Vc[1, h // 2, 7])) < 1e-6


def test_decode_layout_matches_per_sequence_attention():
    rng = np.random.default_rng(14)
    M, H, Hkv, D, Lmax = 4, 6, 3, 16, 33
    pos = rng.integers(0, Lmax, M).astype(np.int32)
    q = _rand(rng, M, H, D)
    Kc, Vc = _rand(rng, M, Hkv, Lmax, D), _rand(rng, M, Hkv, Lmax, D)
    full = oracle.decode(q, Kc, Vc, pos)
    for i in range(M):
        L = int(pos[i]) + 1
        per = oracle.attend_seq(q[i], Kc[i, :, :L, :].copy(), Vc[i, :, :L, :].copy(), L)
        assert np.array_equal(full[i], per)


def test_decode_out_of_range_position_is_nan_and_counted():
    rng = np.random.default_rng(15)
    M, H, Hkv, D, Lmax = 3, 2, 1, 4, 8
    pos = np.array([3, 8, -1], np.int32)
    q = _rand(rng, M, H, D)
    Kc, Vc = _rand(rng, M, Hkv, Lmax, D), _rand(rng, M, Hkv, Lmax, D)
    out = oracle.decode(q, Kc, Vc, pos)
    assert np.all(np.isfinite(out[0]))
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(out[2]))


# ----------------------------------------------------------------- scatter
def test_scatter_replaces_exactly_the_position_rows():
    rng = np.random.default_rng(16)
    M, Hkv, D, Lmax = 5, 3, 8, 12
    pos = np.array([0, 11, 4, 4, 7], np.int32)
    Kc0, Vc0 = _rand(rng, M, Hkv, Lmax, D), _rand(rng, M, Hkv, Lmax, D)
    kr, vr = _rand(rng, M, Hkv, D), _rand(rng, M, Hkv, D)
    Kc, Vc = Kc0.copy(), Vc0.copy()
    assert oracle.kv_scatter(kr, vr, pos, Kc, Vc) == 0
    # expected cache built with numpy advanced indexing (independent route)
    Ke, Ve = Kc0.copy(), Vc0.copy()
    Ke[np.arange(M), :, pos, :] = kr
    Ve[np.arange(M), :, pos, :] = vr
    assert np.array_equal(Kc.view(np.int32), Ke.view(np.int32))
    assert np.array_equal(Vc.view(np.int32), Ve.view(np.int32))
    changed = np.argwhere(np.any(Kc.view(np.int32) != Kc0.view(np.int32), axis=3))
    assert len(changed) <= M * Hkv


def test_scatter_skips_out_of_range_positions():
    rng = np.random.default_rng(17)
    M, Hkv, D, Lmax = 3, 2, 4, 6
    pos = np.array([6, -2, 5], np.int32)
    Kc0, Vc0 = _rand(rng, M, Hkv, Lmax, D), _rand(rng, M, Hkv, Lmax, D)
    kr, vr = _rand(rng, M, Hkv, D), _rand(rng, M, Hkv, D)
    Kc, Vc = Kc0.copy(), Vc0.copy()
    assert oracle.kv_scatter(kr, vr, pos, Kc, Vc) == 2
    assert np.array_equal(Kc[:2], Kc0[:2]) and np.array_equal(Vc[:2], Vc0[:2])
    assert np.array_equal(Kc[2, :, 5], kr[2]) and np.array_equal(Vc[2, :, 5], vr[2])


# ---------------------------------------------------------------- pool slots and finished sequences
def _slot_case(M=5, S=8, Hkv=2, G=2, D=16, Lmax=12, seed=41):
    rng = np.random.default_rng(seed)
    H = Hkv * G
    q = rng.standard_normal((M, H, D)).astype(np.float32)
    k_rows = rng.standard_normal((M, Hkv, D)).astype(np.float32)
    v_rows = rng.standard_normal((M, Hkv, D)).astype(np.float32)
    k_pool = rng.standard_normal((S, Hkv, Lmax, D)).astype(np.float32)
    v_pool = rng.standard_normal((S, Hkv, Lmax, D)).astype(np.float32)
    pos = rng.integers(0, Lmax, M).astype(np.int32)
    slots = rng.permutation(S)[:M].astype(np.int32)
    return q, k_rows, v_rows, pos, slots, k_pool, v_pool


def test_slots_identity_reduces_to_scatter_then_decode():
    """slot i for sequence i and nothing finished is the plain step (pinned above)."""
    q, kr, vr, pos, _, kp, vp = _slot_case(S=5)
    kc, vc = kp.copy(), vp.copy()
    assert oracle.kv_scatter(kr, vr, pos, kc, vc) == 0
    want = oracle.decode(q, kc, vc, pos)
    out = np.zeros_like(q)
    assert oracle.decode_step_slots(q, kr, vr, pos, None, None, kp, vp, out) == []
    assert np.array_equal(out, want)
    assert np.array_equal(kp, kc) and np.array_equal(vp, vc)


def test_slots_follow_the_sequence_not_its_index():
    """Relabelling the pool (pool'[perm[s]] = pool[s], slot'_i = perm[slot_i])
    changes neither the outputs nor what each sequence's slot holds."""
    q, kr, vr, pos, slots, kp, vp = _slot_case()
    out1 = np.zeros_like(q)
    kp1, vp1 = kp.copy(), vp.copy()
    oracle.decode_step_slots(q, kr, vr, pos, slots, None, kp1, vp1, out1)
    perm = np.random.default_rng(3).permutation(kp.shape[0])
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    out2 = np.zeros_like(q)
    oracle.decode_step_slots(q, kr, vr, pos, perm[slots].astype(np.int32), None, kp2, vp2, out2)
    assert np.array_equal(out1, out2)
    assert np.array_equal(kp2[perm], kp1) and np.array_equal(vp2[perm], vp1)
    # and each sequence attends its own slot's rows: a slot-i-for-i answer differs
    out3 = np.zeros_like(q)
    oracle.decode_step_slots(q, kr, vr, pos, None, None, kp.copy(), vp.copy(), out3)
    assert not np.array_equal(out1, out3)


def test_slot_scatter_writes_only_the_position_rows_of_each_slot():
    q, kr, vr, pos, slots, kp, vp = _slot_case()
    want_k, want_v = kp.copy(), vp.copy()
    want_k[slots, :, pos, :] = kr
    want_v[slots, :, pos, :] = vr
    oracle.decode_step_slots(q, kr, vr, pos, slots, None, kp, vp, np.zeros_like(q))
    assert np.array_equal(kp, want_k) and np.array_equal(vp, want_v)


def test_finished_sequences_keep_their_output_and_still_scatter():
    q, kr, vr, pos, slots, kp, vp = _slot_case()
    done = np.array([0, 1, 0, 1, 0], np.uint8)
    before = np.random.default_rng(9).standard_normal(q.shape).astype(np.float32)
    out = before.copy()
    kp0, vp0 = kp.copy(), vp.copy()
    oracle.decode_step_slots(q, kr, vr, pos, slots, done, kp, vp, out)
    for i in range(len(done)):
        if done[i]:
            assert np.array_equal(out[i], before[i])
        else:
            assert not np.array_equal(out[i], before[i])
        assert np.array_equal(kp[slots[i], :, pos[i]], kr[i])  # scattered either way
    # the live sequences equal a run without the finished ones
    live = np.flatnonzero(done == 0)
    out_live = np.zeros((len(live),) + q.shape[1:], np.float32)
    oracle.decode_step_slots(q[live], kr[live], vr[live], pos[live], slots[live], None,
                             kp0, vp0, out_live)
    assert np.array_equal(out[live], out_live)


def test_bad_slot_or_position_is_skipped_and_nan():
    q, kr, vr, pos, slots, kp, vp = _slot_case()
    slots = slots.copy()
    pos = pos.copy()
    slots[1] = kp.shape[0]      # one past the pool
    slots[2] = -1
    pos[3] = kp.shape[2]        # one past Lmax
    done = np.array([0, 0, 1, 0, 0], np.uint8)
    kp0, vp0 = kp.copy(), vp.copy()
    out = np.zeros_like(q)
    bad = oracle.decode_step_slots(q, kr, vr, pos, slots, done, kp, vp, out)
    assert bad == [1, 2, 3]
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(out[3]))
    assert np.array_equal(out[2], np.zeros_like(out[2]))  # finished: untouched
    for i in (0, 4):
        assert np.all(np.isfinite(out[i]))
    touched = {(int(slots[i]), int(pos[i])) for i in (0, 4)}
    for s in range(kp.shape[0]):
        for r in range(kp.shape[2]):
            same = np.array_equal(kp[s, :, r], kp0[s, :, r]) and \
                np.array_equal(vp[s, :, r], vp0[s, :, r])
            assert same == ((s, r) not in touched)


# ---------------------------------------------------------------- batched argmax
def test_argmax_first_maximum_on_ties():
    x = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [-1.0, -2.0, -1.0, -3.0]],
                 np.float32)
    assert oracle.argmax_rows(x).tolist() == [1, 0, 0]


def test_argmax_ignores_nan_and_handles_infinities():
    nan, inf = np.nan, np.inf
    x = np.array([[nan, 1.0, nan, 0.5],
                  [nan, nan, nan, nan],
                  [-inf, -inf, -inf, -inf],
                  [0.0, inf, 7.0, inf],
                  [nan, -inf, -1e30, nan]], np.float32)
    assert oracle.argmax_rows(x).tolist() == [1, 0, 0, 1, 2]


def test_argmax_matches_a_sort_on_random_rows():
    """Against an independent rule: stable sort by (-value, index)."""
    rng = np.random.default_rng(17)
    x = rng.standard_normal((6, 3001)).astype(np.float32)
    x[2, 100] = x[2, 2000] = 50.0          # a tie far apart: the first wins
    x[4, :] = np.round(x[4, :])            # many ties
    got = oracle.argmax_rows(x)
    for i in range(x.shape[0]):
        order = sorted(range(x.shape[1]), key=lambda j: (-float(x[i, j]), j))
        assert got[i] == order[0]
    assert got[2] == 100


# ---------------------------------------------------------------- prefill attention
def test_prefill_causal_first_row_is_first_value_row():
    rng = np.random.default_rng(2)
    q, k, v = (rng.standard_normal((2, 16, 16)).astype(np.float32) for _ in range(3))
    out = oracle.prefill_attention(q, k, v, causal=True, fp16_inputs=False)
    assert np.array_equal(out[:, 0, :], v[:, 0, :].astype(np.float64))


def test_prefill_equals_per_row_decode_attention():
    """Row i of causal prefill is the decode attention of query i over keys
    0..i (the pinned decode oracle); non-causal rows attend all keys."""
    rng = np.random.default_rng(3)
    H, S, D = 2, 32, 64
    q, k, v = (rng.standard_normal((H, S, D)).astype(np.float32) for _ in range(3))
    c = oracle.prefill_attention(q, k, v, causal=True, fp16_inputs=False)
    n = oracle.prefill_attention(q, k, v, causal=False, fp16_inputs=False)
    for h in range(H):
        for i in (0, 1, 17, S - 1):
            want = oracle.attend_row(q[h, i], k[h, :i + 1], v[h, :i + 1], f64=True)
            assert np.allclose(c[h, i], want, rtol=1e-12, atol=1e-13)
            want = oracle.attend_row(q[h, i], k[h], v[h], f64=True)
            assert np.allclose(n[h, i], want, rtol=1e-12, atol=1e-13)
    assert np.allclose(c[:, S - 1], n[:, S - 1], rtol=1e-12, atol=1e-13)


def test_prefill_identical_keys_give_running_mean():
    rng = np.random.default_rng(4)
    H, S, D = 1, 16, 16
    q = rng.standard_normal((H, S, D)).astype(np.float32)
    k = np.tile(rng.standard_normal((1, 1, D)).astype(np.float32), (H, S, 1))
    v = rng.standard_normal((H, S, D)).astype(np.float32)
    out = oracle.prefill_attention(q, k, v, causal=True, fp16_inputs=False)
    for i in range(S):
        want = [math.fsum(float(v[0, j, d]) for j in range(i + 1)) / (i + 1) for d in range(D)]
        assert np.allclose(out[0, i], want, rtol=1e-13, atol=1e-14)


def test_prefill_fp16_inputs_are_rounded_first():
    """The FP16 mode equals the exact mode applied to half-rounded inputs,
    and differs from the unrounded result."""
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((2, 32, 64)).astype(np.float32) for _ in range(3))
    r = [a.astype(np.float16).astype(np.float32) for a in (q, k, v)]
    a = oracle.prefill_attention(q, k, v, causal=True, fp16_inputs=True)
    b = oracle.prefill_attention(*r, causal=True, fp16_inputs=False)
    assert np.array_equal(a, b)
    c = oracle.prefill_attention(q, k, v, causal=True, fp16_inputs=False)
    assert not np.array_equal(a, c) and np.abs(a - c).max() < 1e-2
