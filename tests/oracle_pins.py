"""Pins that tie the float64 oracle to facts fixed outside itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a closed form, a brute-force evaluation in 50-digit arithmetic, a library
routine (numpy matmul + scipy.special), or the associativity of the
log-sum-exp merge (Tree Attention explainer, aibr.jp/archives/143699,
sections 1-3: the sequence-axis reduction is an exact tree).  The pins are
plain functions so that the mutation test can run every one of them against
a deliberately broken copy of the oracle and check that each planted
mistake is caught.
"""
from __future__ import annotations

import itertools
import math

import mpmath
import numpy as np
import scipy.special

import oracle


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f32(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


# ------------------------------------------------------------ closed forms

def pin_identical_keys_give_mean_of_v():
    """All keys equal: every weight is 1/L, so out = mean(V[:L]), lse = s + ln L."""
    rng = _rng(11)
    B, Hq, Hkv, S, D = 1, 2, 1, 37, 8
    q = _f32(rng, B, Hq, D)
    k0 = _f32(rng, D)
    k = np.ascontiguousarray(np.broadcast_to(k0, (B, Hkv, S, D)))
    v = _f32(rng, B, Hkv, S, D)
    scale = 0.3
    for L in (1, 5, 36, 37):
        out, lse = oracle.decode(q, k, v, scale, seqlens=[L])
        mean = v[0, 0, :L].astype(np.float64).mean(0)
        for h in range(Hq):
            s0 = scale * float(q[0, h].astype(np.float64) @ k0.astype(np.float64))
            assert np.max(np.abs(out[h] - mean)) < 1e-12
            assert abs(lse[h] - (s0 + math.log(L))) < 1e-12


def pin_zero_query_is_uniform():
    """q = 0: all scores 0, out = mean(V[:L]), lse = ln L."""
    rng = _rng(12)
    B, Hq, Hkv, S, D = 2, 2, 2, 50, 4
    q = np.zeros((B, Hq, D), np.float32)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    seqlens = [50, 17]
    out, lse = oracle.decode(q, k, v, 0.5, seqlens=seqlens)
    for b in range(B):
        for h in range(Hq):
            r = b * Hq + h
            mean = v[b, h, :seqlens[b]].astype(np.float64).mean(0)
            assert np.max(np.abs(out[r] - mean)) < 1e-12
            assert abs(lse[r] - math.log(seqlens[b])) < 1e-12


def pin_single_dominant_logit():
    """One key aligned with q and far above the rest: out = v_j*, lse = s_j*."""
    rng = _rng(13)
    S, D = 40, 16
    q = _f32(rng, 1, 1, D)
    k = _f32(rng, 1, 1, S, D, scale=0.05)
    jstar = 23
    k[0, 0, jstar] = 4.0 * q[0, 0]
    v = _f32(rng, 1, 1, S, D)
    scale = 1.0
    s = scale * (k[0, 0].astype(np.float64) @ q[0, 0].astype(np.float64))
    gap = s[jstar] - np.max(np.delete(s, jstar))
    assert gap > 40  # weights of the other keys are below e^-40
    out, lse = oracle.decode(q, k, v, scale)
    assert np.max(np.abs(out[0] - v[0, 0, jstar])) < 1e-12
    assert abs(lse[0] - s[jstar]) < 1e-12


def pin_single_key():
    """S = 1: out = v_0 exactly and lse = s_0."""
    rng = _rng(14)
    D = 8
    q = _f32(rng, 1, 1, D)
    k = _f32(rng, 1, 1, 1, D)
    v = _f32(rng, 1, 1, 1, D)
    out, lse = oracle.decode(q, k, v, 0.7)
    s0 = 0.7 * float(q[0, 0].astype(np.float64) @ k[0, 0, 0].astype(np.float64))
    assert np.array_equal(out[0], v[0, 0, 0].astype(np.float64))
    assert abs(lse[0] - s0) < 1e-13


def pin_shift_invariance():
    """An extra dimension where every key is 1 shifts all logits by scale*t:
    out is unchanged and lse moves by exactly that shift."""
    rng = _rng(15)
    B, Hq, Hkv, S, D = 1, 3, 3, 29, 5
    q = _f32(rng, B, Hq, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    t, scale = 2.5, 0.25
    q2 = np.concatenate([q, np.full((B, Hq, 1), t, np.float32)], axis=-1)
    k2 = np.concatenate([k, np.ones((B, Hkv, S, 1), np.float32)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, Hkv, S, 1), np.float32)], axis=-1)
    out, lse = oracle.decode(q, k, v, scale)
    out2, lse2 = oracle.decode(q2, k2, v2, scale)
    assert np.max(np.abs(out2[:, :D] - out)) < 1e-12
    assert np.max(np.abs(lse2 - (lse + scale * t))) < 1e-12


def pin_zero_keys_count():
    """K = 0: every score is 0, so lse = ln(count of attended keys) and out = mean."""
    rng = _rng(16)
    B, Hq, Hkv, S, D = 3, 2, 1, 300, 4
    q = _f32(rng, B, Hq, D)
    k = np.zeros((B, Hkv, S, D), np.float32)
    v = _f32(rng, B, Hkv, S, D)
    seqlens = [1, 255, 300]
    out, lse = oracle.decode(q, k, v, 1.0, seqlens=seqlens)
    for b in range(B):
        for h in range(Hq):
            assert abs(lse[b * Hq + h] - math.log(seqlens[b])) < 1e-12
            assert np.max(np.abs(out[b * Hq + h] - v[b, 0, :seqlens[b]].astype(np.float64).mean(0))) < 1e-12


def pin_large_logits_stay_finite():
    """Logits near 1000 (exp overflows a double) after a far smaller first key, with
    a gap d between the two large ones: lse = s1 + ln(1 + e^-d) and
    out = (v1 + e^-d v2) / (1 + e^-d) (the first key's weight e^-1003 is below
    double precision)."""
    q = np.ones((1, 1, 1), np.float32)
    k = np.array([-3.0, 1000.0, 998.5], np.float32).reshape(1, 1, 3, 1)
    v = np.array([5.0, 2.0, -1.0], np.float32).reshape(1, 1, 3, 1)
    out, lse = oracle.decode(q, k, v, 1.0)
    d = float(k[0, 0, 1, 0]) - float(k[0, 0, 2, 0])
    w = math.exp(-d)
    assert abs(lse[0] - (1000.0 + math.log1p(w))) < 1e-12
    assert abs(out[0, 0] - (2.0 - w) / (1.0 + w)) < 1e-12
    m, l, o = oracle.decode_partials(q, k, v, 1.0, 0, 0, [0, 1, 3])
    out2, lse2 = oracle.combine(m[None], l[None], o[None])
    assert abs(lse2[0] - lse[0]) < 1e-12 and abs(out2[0, 0] - out[0, 0]) < 1e-12


def pin_empty_sequence():
    """An empty attended set gives out = 0 and lse = -inf (the reading taken)."""
    rng = _rng(17)
    q = _f32(rng, 2, 1, 4)
    k = _f32(rng, 2, 1, 6, 4)
    v = _f32(rng, 2, 1, 6, 4)
    out, lse = oracle.decode(q, k, v, 1.0, seqlens=[0, 6])
    assert np.array_equal(out[0], np.zeros(4)) and lse[0] == -np.inf
    assert np.isfinite(lse[1])


def pin_combine_closed_form():
    """Two partials: (m=0, l=1, o=1) and (m=ln 3, l=1, o=2) merge to weights 1:3,
    so out = (1 + 3*2) / (1 + 3) = 7/4 and lse = ln 4; an empty partial is ignored."""
    m = np.array([[0.0, math.log(3.0), -np.inf]])
    l = np.array([[1.0, 1.0, 0.0]])
    o = np.array([[[1.0], [2.0], [0.0]]])
    out, lse = oracle.combine(m, l, o)
    assert abs(out[0, 0] - 1.75) < 1e-15
    assert abs(lse[0] - math.log(4.0)) < 1e-15
    out, lse = oracle.combine(np.full((1, 2), -np.inf), np.zeros((1, 2)), np.zeros((1, 2, 3)))
    assert lse[0] == -np.inf and np.array_equal(out[0], np.zeros(3))


# ------------------------------------------------------------ brute force

def _mp_attend(q, K, V, scale):
    """Naive softmax in 50-digit arithmetic: no max subtraction, no tricks."""
    with mpmath.workdps(50):
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in zip(q, kr))
             for kr in K]
        e = [mpmath.exp(x) for x in s]
        z = mpmath.fsum(e)
        out = [float(mpmath.fsum(e[j] * mpmath.mpf(float(V[j][d])) for j in range(len(K))) / z)
               for d in range(len(V[0]))]
        return out, float(mpmath.log(z))


def pin_brute_force_decode():
    rng = _rng(18)
    for S in range(1, 9):
        for D in (1, 2, 4):
            for G in (1, 2):
                Hkv = 2
                Hq = Hkv * G
                q = _f32(rng, 1, Hq, D)
                k = _f32(rng, 1, Hkv, S, D, scale=1.5)
                v = _f32(rng, 1, Hkv, S, D)
                L = max(1, S - (S // 3))
                out, lse = oracle.decode(q, k, v, 0.9, seqlens=[L])
                for h in range(Hq):
                    ref, ref_lse = _mp_attend(q[0, h], k[0, h // G, :L], v[0, h // G, :L], 0.9)
                    assert np.max(np.abs(out[h] - np.array(ref))) < 1e-13, (S, D, G, h)
                    assert abs(lse[h] - ref_lse) < 1e-13


def pin_brute_force_prefill():
    rng = _rng(19)
    for S in (1, 2, 5, 8):
        H, Hkv, D = 4, 2, 3
        q = _f32(rng, 1, H, S, D)
        k = _f32(rng, 1, Hkv, S, D)
        v = _f32(rng, 1, Hkv, S, D)
        out, lse = oracle.prefill_causal(q, k, v, 0.6)
        for h in range(H):
            for i in range(S):
                r = h * S + i
                ref, ref_lse = _mp_attend(q[0, h, i], k[0, h // 2, :i + 1], v[0, h // 2, :i + 1], 0.6)
                assert np.max(np.abs(out[r] - np.array(ref))) < 1e-13, (S, h, i)
                assert abs(lse[r] - ref_lse) < 1e-13


# ------------------------------------------------------------ library routines

def pin_library_routines():
    """numpy float64 matmul for the scores, scipy.special.logsumexp / softmax for the rest."""
    rng = _rng(20)
    B, Hq, Hkv, S, D = 2, 6, 2, 300, 32
    G = Hq // Hkv
    q = _f32(rng, B, Hq, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    seqlens = [300, 123]
    scale = 1 / math.sqrt(D)
    out, lse = oracle.decode(q, k, v, scale, seqlens=seqlens)
    for b in range(B):
        L = seqlens[b]
        for h in range(Hq):
            Kd = k[b, h // G, :L].astype(np.float64)
            Vd = v[b, h // G, :L].astype(np.float64)
            s = scale * (Kd @ q[b, h].astype(np.float64))
            r = b * Hq + h
            assert abs(lse[r] - scipy.special.logsumexp(s)) < 1e-12
            assert np.max(np.abs(out[r] - scipy.special.softmax(s) @ Vd)) < 1e-12


def pin_library_routines_prefill():
    rng = _rng(21)
    B, H, Hkv, S, D = 1, 4, 1, 70, 16
    q = _f32(rng, B, H, S, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    scale = 0.25
    out, lse = oracle.prefill_causal(q, k, v, scale)
    Kd = k[0, 0].astype(np.float64)
    Vd = v[0, 0].astype(np.float64)
    for h in range(H):
        s_all = scale * (q[0, h].astype(np.float64) @ Kd.T)
        for i in range(S):
            s = s_all[i, :i + 1]
            r = h * S + i
            assert abs(lse[r] - scipy.special.logsumexp(s)) < 1e-12
            assert np.max(np.abs(out[r] - scipy.special.softmax(s) @ Vd[:i + 1])) < 1e-12


# ------------------------------------------------------------ tree law

def _compositions(S):
    """All ways to cut [0, S) into consecutive non-empty chunks, as bound lists."""
    for cuts in itertools.product((0, 1), repeat=S - 1):
        b = [0] + [i + 1 for i, c in enumerate(cuts) if c] + [S]
        yield b


def pin_tree_law_every_composition():
    """Merging per-chunk partials equals the single pass, for every way of cutting the
    sequence into chunks (S <= 12) and for a permuted order of the partials."""
    rng = _rng(22)
    D = 3
    for S in (1, 2, 3, 7, 12):
        q = _f32(rng, 1, 1, D, scale=2.0)
        k = _f32(rng, 1, 1, S, D, scale=2.0)
        v = _f32(rng, 1, 1, S, D)
        ref_out, ref_lse = oracle.decode(q, k, v, 1.0)
        for bounds in _compositions(S):
            m, l, o = oracle.decode_partials(q, k, v, 1.0, 0, 0, bounds)
            perm = rng.permutation(len(m))
            out, lse = oracle.combine(m[perm][None], l[perm][None], o[perm][None])
            assert np.max(np.abs(out[0] - ref_out[0])) <= 1e-12 * max(1.0, np.max(np.abs(ref_out)))
            assert abs(lse[0] - ref_lse[0]) <= 1e-12 * max(1.0, abs(ref_lse[0]))


def pin_tree_law_random_splits():
    """Random splits with empty chunks and chunks wholly past the sequence length,
    merged in random order, and merged in two levels (a tree), equal the single pass."""
    rng = _rng(23)
    B, Hq, Hkv, S, D = 2, 4, 2, 777, 8
    q = _f32(rng, B, Hq, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    seqlens = [777, 400]
    ref_out, ref_lse = oracle.decode(q, k, v, 0.35, seqlens=seqlens)
    for trial in range(6):
        n = int(rng.integers(2, 40))
        inner = np.sort(rng.integers(0, S + 1, size=n - 1))
        bounds = np.concatenate([[0], inner, [S]])
        for b in range(B):
            for h in range(Hq):
                m, l, o = oracle.decode_partials(q, k, v, 0.35, b, h, bounds, seqlens=seqlens)
                perm = rng.permutation(len(m))
                out, lse = oracle.combine(m[perm][None], l[perm][None], o[perm][None])
                r = b * Hq + h
                assert np.max(np.abs(out[0] - ref_out[r])) < 1e-12
                assert abs(lse[0] - ref_lse[r]) < 1e-12
                # two-level tree: merge groups of 5, then merge the group results
                gm, gl, go = [], [], []
                for g0 in range(0, len(m), 5):
                    o1, lse1 = oracle.combine(m[None, g0:g0 + 5], l[None, g0:g0 + 5], o[None, g0:g0 + 5])
                    if lse1[0] == -np.inf:
                        gm.append(-np.inf)
                        gl.append(0.0)
                        go.append(np.zeros(D))
                    else:  # (m, l, o) = (lse, 1, out) is a valid partial for the group
                        gm.append(lse1[0])
                        gl.append(1.0)
                        go.append(o1[0])
                out2, lse2 = oracle.combine(np.array(gm)[None], np.array(gl)[None], np.array(go)[None])
                assert np.max(np.abs(out2[0] - ref_out[r])) < 1e-12
                assert abs(lse2[0] - ref_lse[r]) < 1e-12


# ------------------------------------------------------------ structure

def pin_gqa_equals_repeated_mha():
    """GQA with G = Hq/Hkv equals Hq independent heads on K/V repeated per group
    (query head h reads KV head floor(h/G))."""
    rng = _rng(24)
    B, Hq, Hkv, S, D = 2, 8, 2, 64, 8
    G = Hq // Hkv
    q = _f32(rng, B, Hq, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    k_rep = np.ascontiguousarray(np.repeat(k, G, axis=1))
    v_rep = np.ascontiguousarray(np.repeat(v, G, axis=1))
    out, lse = oracle.decode(q, k, v, 0.4, seqlens=[64, 31])
    out_r, lse_r = oracle.decode(q, k_rep, v_rep, 0.4, seqlens=[64, 31])
    assert np.array_equal(out, out_r) and np.array_equal(lse, lse_r)
    qp = _f32(rng, B, Hq, S, D)
    out, lse = oracle.prefill_causal(qp, k, v, 0.4)
    out_r, lse_r = oracle.prefill_causal(qp, k_rep, v_rep, 0.4)
    assert np.array_equal(out, out_r) and np.array_equal(lse, lse_r)


def pin_prefill_row_is_decode_of_prefix():
    """Causal prefill row i equals decode of that query over the first i+1 keys."""
    rng = _rng(25)
    B, H, Hkv, S, D = 1, 4, 2, 23, 8
    q = _f32(rng, B, H, S, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    out, lse = oracle.prefill_causal(q, k, v, 0.3)
    for i in range(S):
        qi = np.ascontiguousarray(q[:, :, i, :])
        o_d, l_d = oracle.decode(qi, k, v, 0.3, seqlens=[i + 1])
        for h in range(H):
            assert np.max(np.abs(out[h * S + i] - o_d[h])) < 1e-13
            assert abs(lse[h * S + i] - l_d[h]) < 1e-13


def pin_masked_keys_never_read():
    """Keys at or past the sequence length are NaN; the result stays finite and equals
    the result on the truncated cache."""
    rng = _rng(26)
    B, Hq, Hkv, S, D = 3, 2, 1, 40, 4
    q = _f32(rng, B, Hq, D)
    k = _f32(rng, B, Hkv, S, D)
    v = _f32(rng, B, Hkv, S, D)
    seqlens = [40, 13, 1]
    kn, vn = k.copy(), v.copy()
    for b, L in enumerate(seqlens):
        kn[b, :, L:] = np.nan
        vn[b, :, L:] = np.nan
    out, lse = oracle.decode(q, kn, vn, 0.5, seqlens=seqlens)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    for b, L in enumerate(seqlens):
        o_t, l_t = oracle.decode(q[b:b + 1], np.ascontiguousarray(k[b:b + 1, :, :L]),
                                 np.ascontiguousarray(v[b:b + 1, :, :L]), 0.5)
        assert np.array_equal(out[b * Hq:(b + 1) * Hq], o_t) and np.array_equal(lse[b * Hq:(b + 1) * Hq], l_t)


def pin_row_subset_matches_all_rows():
    """Computing a listed subset of rows gives the same numbers as computing all rows."""
    rng = _rng(27)
    q = _f32(rng, 2, 4, 1, 8).reshape(2, 4, 8)
    k = _f32(rng, 2, 2, 50, 8)
    v = _f32(rng, 2, 2, 50, 8)
    out, lse = oracle.decode(q, k, v, 0.3)
    rows = [7, 0, 3]
    o2, l2 = oracle.decode(q, k, v, 0.3, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


# ------------------------------------------------------------ paged KV cache

def _paged_case(rng, B, Hkv, G, page, lens, D=4, extra=2):
    """A shuffled page pool built with explicit loops (independent of the
    oracle's numpy gather): returns q, pools, table, and the key rows of each
    sequence listed as (page, row) pairs."""
    P = max((L + page - 1) // page for L in lens)
    used = [(L + page - 1) // page for L in lens]
    n_pages = sum(used) + extra
    perm = rng.permutation(n_pages)
    kp = (rng.standard_normal((n_pages, Hkv, page, D)) * 1.3).astype(np.float32)
    vp = rng.standard_normal((n_pages, Hkv, page, D)).astype(np.float32)
    table = np.zeros((B, P), dtype=np.int32)
    where = []
    nxt = 0
    for b in range(B):
        rows = []
        for pg in range(P):
            if pg < used[b]:
                table[b, pg] = perm[nxt]
                nxt += 1
            else:
                table[b, pg] = perm[-1]  # a page of no sequence: never read
        for j in range(lens[b]):
            rows.append((int(table[b, j // page]), j % page))
        where.append(rows)
    q = rng.standard_normal((B, Hkv * G, D)).astype(np.float32)
    return q, kp, vp, table, where


def pin_paged_brute_force():
    """Paged decode against 50-digit attention over the keys listed page by
    page with plain loops."""
    rng = _rng(41)
    for page in (1, 3, 4):
        lens = [5, 1, 7]
        q, kp, vp, table, where = _paged_case(rng, 3, 2, 2, page, lens)
        out, lse = oracle.decode_paged(q, kp, vp, table, lens, 0.7)
        for b in range(3):
            for h in range(4):
                kv = h // 2
                ks = np.array([kp[pg, kv, r] for pg, r in where[b]])
                vs = np.array([vp[pg, kv, r] for pg, r in where[b]])
                ref, ref_lse = _mp_attend(q[b, h], ks, vs, 0.7)
                assert np.max(np.abs(out[b * 4 + h] - np.array(ref))) < 1e-13, (page, b, h)
                assert abs(lse[b * 4 + h] - ref_lse) < 1e-13


def pin_paged_page_permutation():
    """Relabelling the physical pages (and the table with them) changes
    nothing; pages of no sequence may hold anything."""
    rng = _rng(42)
    lens = [23, 9, 16]
    q, kp, vp, table, _ = _paged_case(rng, 3, 2, 2, 4, lens)
    a = oracle.decode_paged(q, kp, vp, table, lens, 0.5)
    perm = rng.permutation(kp.shape[0])
    inv = np.argsort(perm)
    kp2, vp2 = kp[perm], vp[perm]
    table2 = inv[table].astype(np.int32)
    b_ = oracle.decode_paged(q, kp2, vp2, table2, lens, 0.5)
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


# ------------------------------------------------------------ pi-Attention key set

def pin_pi_brute_force():
    """pi-Attention decode against 50-digit attention over the keys chosen one by
    one from the definition: j in the window [i - w, i], or i - j a positive
    multiple of the period."""
    rng = _rng(51)
    B, Hkv, G, S, D = 2, 2, 2, 23, 4
    q = _f32(rng, B, Hkv * G, D)
    k = _f32(rng, B, Hkv, S, D, scale=1.4)
    v = _f32(rng, B, Hkv, S, D)
    for window, period in ((0, 1), (2, 3), (4, 5), (0, 7), (30, 2), (3, 50)):
        lens = [23, 9]
        out, lse = oracle.decode_pi(q, k, v, 0.6, window, period, seqlens=lens)
        for b in range(B):
            i = lens[b] - 1
            chosen = [j for j in range(lens[b]) if i - window <= j <= i or (i - j) % period == 0]
            for h in range(Hkv * G):
                ref, ref_lse = _mp_attend(q[b, h], k[b, h // G, chosen], v[b, h // G, chosen], 0.6)
                assert np.max(np.abs(out[b * Hkv * G + h] - np.array(ref))) < 1e-13, (window, period, b, h)
                assert abs(lse[b * Hkv * G + h] - ref_lse) < 1e-13


def pin_pi_special_cases():
    """Period 1, or a window reaching key 0, attends every key (plain decode);
    a period longer than the sequence leaves the window only."""
    rng = _rng(52)
    q = _f32(rng, 1, 4, 8)
    k = _f32(rng, 1, 2, 40, 8)
    v = _f32(rng, 1, 2, 40, 8)
    dense = oracle.decode(q, k, v, 0.4)
    for window, period in ((0, 1), (5, 1), (39, 9), (100, 3)):
        got = oracle.decode_pi(q, k, v, 0.4, window, period)
        assert np.array_equal(got[0], dense[0]) and np.array_equal(got[1], dense[1]), (window, period)
    tail = oracle.decode(q, np.ascontiguousarray(k[:, :, 33:]), np.ascontiguousarray(v[:, :, 33:]), 0.4)
    got = oracle.decode_pi(q, k, v, 0.4, 6, 41)
    assert np.array_equal(got[0], tail[0]) and np.array_equal(got[1], tail[1])


# ------------------------------------------------------------ packed variable-length prefill

def pin_varlen_prefill_brute_force():
    """Packed causal prefill against 50-digit attention of each token over the
    earlier tokens of its own sequence, looped token by token."""
    rng = _rng(61)
    cu = [0, 3, 3, 8, 9]
    T, H, Hkv, D = cu[-1], 4, 2, 4
    q = _f32(rng, T, H, D)
    k = _f32(rng, T, Hkv, D, scale=1.3)
    v = _f32(rng, T, Hkv, D)
    out, lse = oracle.prefill_causal_varlen(q, k, v, cu, 0.8)
    for s in range(len(cu) - 1):
        for t in range(cu[s], cu[s + 1]):
            for h in range(H):
                ref, ref_lse = _mp_attend(q[t, h], k[cu[s]:t + 1, h // 2], v[cu[s]:t + 1, h // 2], 0.8)
                assert np.max(np.abs(out[t, h] - np.array(ref))) < 1e-13, (s, t, h)
                assert abs(lse[h, t] - ref_lse) < 1e-13


def pin_varlen_prefill_sequences_independent():
    """A sequence's output depends on its own tokens only."""
    rng = _rng(62)
    cu = [0, 6, 13]
    q = _f32(rng, 13, 2, 4)
    k = _f32(rng, 13, 1, 4)
    v = _f32(rng, 13, 1, 4)
    a = oracle.prefill_causal_varlen(q, k, v, cu, 0.5)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[6:] += 3.0
    k2[6:] *= -2.0
    v2[6:] += 1.0
    b = oracle.prefill_causal_varlen(q2, k2, v2, cu, 0.5)
    assert np.array_equal(a[0][:6], b[0][:6]) and np.array_equal(a[1][:, :6], b[1][:, :6])
    assert not np.array_equal(a[0][6:], b[0][6:])


# ------------------------------------------------------------ FP8 (E4M3) KV cache

def pin_e4m3_values_match_the_library():
    """All 256 E4M3 bit patterns decode as torch's float8_e4m3fn does."""
    import torch
    bits = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_float(bits)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])


def pin_fp8_brute_force():
    """FP8 decode against 50-digit attention over keys and values dequantised
    element by element (sign * 2^(e-7) * (1 + m/8), or 2^-6 * m/8) times the
    (sequence, KV head) scale."""
    rng = _rng(71)
    B, Hkv, G, S, D = 2, 2, 2, 9, 4
    k8 = rng.integers(0, 256, size=(B, Hkv, S, D)).astype(np.uint8)
    v8 = rng.integers(0, 256, size=(B, Hkv, S, D)).astype(np.uint8)
    k8[(k8 & 0x7f) == 0x7f] = 0x38  # no NaN patterns
    v8[(v8 & 0x7f) == 0x7f] = 0x40
    k8 = np.where((k8 >> 3) & 15 >= 13, k8 & 0x87, k8).astype(np.uint8)  # keep logits moderate
    ks = rng.uniform(0.01, 0.05, B * Hkv)
    vs = rng.uniform(0.5, 2.0, B * Hkv)
    q = _f32(rng, B, Hkv * G, D)

    def val(bt):
        bt = int(bt)
        sgn = -1 if bt >> 7 else 1
        e, m = (bt >> 3) & 15, bt & 7
        return sgn * (mpmath.mpf(m) / 8 * mpmath.mpf(2) ** -6 if e == 0 else (1 + mpmath.mpf(m) / 8) * mpmath.mpf(2) ** (e - 7))

    out, lse = oracle.decode_fp8(q, k8, v8, ks, vs, 0.7)
    for b in range(B):
        for h in range(Hkv * G):
            u = b * Hkv + h // G
            kk = np.array([[float(val(x) * ks[u]) for x in row] for row in k8[b, h // G]])
            vv = np.array([[float(val(x) * vs[u]) for x in row] for row in v8[b, h // G]])
            ref, ref_lse = _mp_attend(q[b, h], kk, vv, 0.7)
            assert np.max(np.abs(out[b * Hkv * G + h] - np.array(ref))) < 1e-12 * max(1.0, float(np.max(np.abs(vv))))
            assert abs(lse[b * Hkv * G + h] - ref_lse) < 1e-12


def pin_fp8_scales_are_linear():
    """A key scale multiplies the logits, a value scale the output."""
    rng = _rng(72)
    k8 = rng.integers(0, 0x60, size=(1, 1, 12, 8)).astype(np.uint8)
    v8 = rng.integers(0, 0x70, size=(1, 1, 12, 8)).astype(np.uint8)
    q = _f32(rng, 1, 2, 8)
    a = oracle.decode_fp8(q, k8, v8, [0.02], [1.0], 0.5)
    b_ = oracle.decode_fp8(q, k8, v8, [0.01], [3.0], 1.0)
    assert np.max(np.abs(3.0 * a[0] - b_[0])) < 1e-12 and np.max(np.abs(a[1] - b_[1])) < 1e-12


# ------------------------------------------------------------ NVFP4 KV cache

def pin_e2m1_values_match_the_format_table():
    """The 16 E2M1 codes: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0-7
    (the FP4 E2M1 element table of the microscaling formats), the same with
    the sign bit (code + 8) negative."""
    table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mine = oracle.e2m1_to_float(np.arange(16))
    assert np.array_equal(mine[:8], table) and np.array_equal(mine[8:], -table)
    assert np.array_equal(oracle.e2m1_to_float(np.arange(16) + 16 * 5), mine)  # only the low 4 bits count


def pin_nvfp4_block_scale_covers_16_elements():
    """A block scale multiplies exactly its 16 consecutive elements, and the
    low nibble of a byte is the even element: codes 0x42 (elements 1.0, 2.0)
    everywhere, block scales 1.0 (0x38) except block 5 (2.0, 0x40)."""
    codes = np.full((1, 1, 3, 64), 0x42, dtype=np.uint8)
    bs = np.full((1, 1, 3, 8), 0x38, dtype=np.uint8)
    bs[0, 0, 1, 5] = 0x40
    vals = oracle.nvfp4_dequantize(codes, bs, np.full((1, 1, 1, 1), 0.5))
    expect = np.tile(np.array([0.5, 1.0]), 64).reshape(1, 1, 1, 128).repeat(3, axis=2)
    expect[0, 0, 1, 80:96] *= 2.0
    assert np.array_equal(vals, expect)


def pin_nvfp4_brute_force():
    """NVFP4 decode against 50-digit attention over keys and values dequantised
    element by element: element d of a key is the E2M1 value of nibble d % 2 of
    byte d // 2 (sign * 2^(e-1) * (1 + m/2), or m/2 when e = 0), times the E4M3
    scale of block d // 16, times the (sequence, KV head) factor."""
    rng = _rng(73)
    B, Hkv, G, S, D = 2, 2, 2, 7, 32
    k4 = rng.integers(0, 256, size=(B, Hkv, S, D // 2)).astype(np.uint8)
    v4 = rng.integers(0, 256, size=(B, Hkv, S, D // 2)).astype(np.uint8)
    kbs = rng.integers(0x20, 0x40, size=(B, Hkv, S, D // 16)).astype(np.uint8)   # scales 2^-3 .. 2^0
    vbs = rng.integers(0x30, 0x50, size=(B, Hkv, S, D // 16)).astype(np.uint8)
    kf = rng.uniform(0.05, 0.2, B * Hkv)
    vf = rng.uniform(0.5, 2.0, B * Hkv)
    q = _f32(rng, B, Hkv * G, D)

    def e2m1(n):
        sgn = -1 if n & 8 else 1
        e, m = (n >> 1) & 3, n & 1
        return sgn * (mpmath.mpf(m) / 2 if e == 0 else (1 + mpmath.mpf(m) / 2) * mpmath.mpf(2) ** (e - 1))

    def e4m3(bt):
        e, m = (int(bt) >> 3) & 15, int(bt) & 7
        return mpmath.mpf(m) / 8 * mpmath.mpf(2) ** -6 if e == 0 else (1 + mpmath.mpf(m) / 8) * mpmath.mpf(2) ** (e - 7)

    def row(codes, scales, fac):
        out = []
        for d in range(D):
            byte = int(codes[d // 2])
            nib = byte & 15 if d % 2 == 0 else byte >> 4
            out.append(float(e2m1(nib) * e4m3(scales[d // 16]) * mpmath.mpf(float(fac))))
        return out

    out, lse = oracle.decode_nvfp4(q, k4, kbs, v4, vbs, kf, vf, 0.9)
    for b in range(B):
        for h in range(Hkv * G):
            u = b * Hkv + h // G
            kk = np.array([row(k4[b, h // G, j], kbs[b, h // G, j], kf[u]) for j in range(S)])
            vv = np.array([row(v4[b, h // G, j], vbs[b, h // G, j], vf[u]) for j in range(S)])
            ref, ref_lse = _mp_attend(q[b, h], kk, vv, 0.9)
            assert np.max(np.abs(out[b * Hkv * G + h] - np.array(ref))) < 1e-12 * max(1.0, float(np.max(np.abs(vv))))
            assert abs(lse[b * Hkv * G + h] - ref_lse) < 1e-12


ALL_PINS = [f for name, f in sorted(globals().items()) if name.startswith("pin_") and callable(f)]
