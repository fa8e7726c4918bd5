"""Pins of the CPU oracle against facts fixed by the mathematics or the pages.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a brute force over all
subsets, or a value printed on the TidalDecode review page.  None of them
re-types the oracle's own formula: each checks it through a different route.

``tests/test_oracle_pins.py`` runs them against the oracle, and
``tests/test_oracle_mutants.py`` shows that every planted mistake in the
oracle (``ORACLE_MUTANT``) trips at least one of them.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

import oracle as O

D = 128


def _bits(x):
    return O.bf16_bits(np.asarray(x, dtype=np.float32))


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    lim = atol + rtol * (np.max(np.abs(b)) if b.size else 0.0)
    assert err <= lim, f"{what}: max err {err:.3e} > {lim:.3e}"


def pin_bf16_widening(orc):
    """Known bf16 bit patterns widen to their exact values."""
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x3E00: 0.125, 0x0000: 0.0, 0x8000: -0.0,
             0x4049: 3.140625, 0x7F7F: 3.3895313892515355e38, 0x0001: 9.183549615799121e-41}
    for bits, val in cases.items():
        assert orc.bf16_to_double(bits) == val, hex(bits)


def pin_single_token(orc):
    """With one cached token softmax is [1], so the output is that token's V row."""
    rs = np.random.RandomState(1)
    q, K, V = (_bits(rs.randn(*s)) for s in [(D,), (1, D), (1, D)])
    out = orc.attend(q, K, V, O.scale_for(D))
    _close(out, O.bits_to_f64(V[0]), rtol=0, atol=0, what="N=1")


def pin_equal_keys_mean(orc):
    """Identical keys give uniform weights, so the output is the mean of V."""
    rs = np.random.RandomState(2)
    n = 37
    krow = rs.randn(D)
    K = _bits(np.tile(krow, (n, 1)))
    V = _bits(rs.randn(n, D))
    q = _bits(rs.randn(D))
    out = orc.attend(q, K, V, O.scale_for(D))
    _close(out, O.bits_to_f64(V).mean(axis=0), rtol=1e-12, atol=1e-14, what="equal keys")


def pin_two_token_logistic(orc):
    """Two tokens: softmax of two logits is the logistic of their difference.

    q = 2 e0 + e5, k0 = e0, k1 = -e5, so q.k0 = 2, q.k1 = -1 and the logit
    gap is 3 / sqrt(128).  v0 = 4 e3, v1 = -2 e7."""
    q = np.zeros(D); q[0] = 2.0; q[5] = 1.0
    K = np.zeros((2, D)); K[0, 0] = 1.0; K[1, 5] = -1.0
    V = np.zeros((2, D)); V[0, 3] = 4.0; V[1, 7] = -2.0
    scale = O.scale_for(D)
    w0 = 1.0 / (1.0 + math.exp(-3.0 * scale))
    expect = np.zeros(D); expect[3] = 4.0 * w0; expect[7] = -2.0 * (1.0 - w0)
    out = orc.attend(_bits(q), _bits(K), _bits(V), scale)
    _close(out, expect, rtol=1e-13, atol=1e-15, what="two-token logistic")


def pin_softmax_properties(orc):
    """softmax: non-negative, sums to 1, order-preserving, shift-invariant."""
    rs = np.random.RandomState(3)
    a = rs.randn(500) * 4.0
    p = orc.softmax(a)
    assert np.all(p >= 0)
    assert abs(p.sum() - 1.0) < 1e-12, p.sum()
    order = np.argsort(a)
    assert np.all(np.diff(p[order]) >= 0), "softmax must preserve order"
    _close(orc.softmax(a + 123.25), p, rtol=1e-12, atol=1e-15, what="shift")
    # ratio of two weights is exp of the logit gap
    assert abs(p[0] / p[1] - math.exp(a[0] - a[1])) <= 1e-12 * math.exp(a[0] - a[1])


def pin_one_hot_dominance(orc):
    """A key whose logit exceeds every other by ~45 takes all the weight."""
    rs = np.random.RandomState(4)
    n = 64
    K = rs.randint(-1, 2, size=(n, D)).astype(np.float64)
    K[:, 0] = 0.0
    K[17, 0] = 64.0
    q = np.zeros(D); q[0] = 8.0
    V = rs.randn(n, D)
    out = orc.attend(_bits(q), _bits(K), _bits(V), O.scale_for(D))
    _close(out, O.bits_to_f64(_bits(V))[17], rtol=1e-15, atol=1e-15, what="dominant key")


def pin_permutation_invariance(orc):
    """Reordering the cached tokens (keys and values together) changes nothing."""
    rs = np.random.RandomState(5)
    n = 50
    q, K, V = _bits(rs.randn(D)), _bits(rs.randn(n, D)), _bits(rs.randn(n, D))
    perm = rs.permutation(n)
    a = orc.attend(q, K, V, O.scale_for(D))
    b = orc.attend(q, K[perm], V[perm], O.scale_for(D))
    _close(a, b, rtol=1e-12, atol=1e-14, what="permutation")


def pin_linearity_in_v(orc):
    """The output is linear in V (integer V, so V1 + V2 and 2 V are exact in bf16)."""
    rs = np.random.RandomState(6)
    n = 40
    q, K = _bits(rs.randn(D)), _bits(rs.randn(n, D))
    V1 = rs.randint(-3, 4, size=(n, D)).astype(np.float64)
    V2 = rs.randint(-3, 4, size=(n, D)).astype(np.float64)
    s = O.scale_for(D)
    o1 = orc.attend(q, K, _bits(V1), s)
    o2 = orc.attend(q, K, _bits(V2), s)
    o12 = orc.attend(q, K, _bits(V1 + V2), s)
    o2x = orc.attend(q, K, _bits(2.0 * V1), s)
    _close(o12, o1 + o2, rtol=1e-12, atol=1e-13, what="additivity")
    _close(o2x, 2.0 * o1, rtol=1e-12, atol=1e-13, what="homogeneity")


def pin_key_shift_invariance(orc):
    """Adding one vector w to every key shifts every logit by scale*q.w."""
    rs = np.random.RandomState(7)
    n = 30
    q = rs.randint(-2, 3, size=D).astype(np.float64)
    K = rs.randint(-2, 3, size=(n, D)).astype(np.float64)
    w = rs.randint(-2, 3, size=D).astype(np.float64)
    V = _bits(rs.randn(n, D))
    s = O.scale_for(D)
    _close(orc.attend(_bits(q), _bits(K + w), V, s), orc.attend(_bits(q), _bits(K), V, s),
           rtol=1e-12, atol=1e-14, what="key shift")


def pin_integer_logit(orc):
    """For small-integer vectors the dot product is an exact integer."""
    rs = np.random.RandomState(8)
    for _ in range(5):
        q = rs.randint(-3, 4, size=D)
        k = rs.randint(-3, 4, size=D)
        exact = int(np.dot(q.astype(np.int64), k.astype(np.int64)))
        s = O.scale_for(D)
        assert orc.logit(_bits(q), _bits(k), s) == s * exact
        assert orc.logit(_bits(q), _bits(k), 1.0) == float(exact)


def pin_group_score_closed_form(orc):
    """Summed logits of a query group equal one logit of the summed query."""
    rs = np.random.RandomState(9)
    G, n = 4, 60
    qg = rs.randint(-2, 3, size=(G, D)).astype(np.float64)     # sum stays exact in bf16
    K = rs.randint(-2, 3, size=(n, D)).astype(np.float64)
    s = O.scale_for(D)
    got = orc.group_scores(_bits(qg), _bits(K), n, s)
    qsum = _bits(qg.sum(axis=0))
    want = np.array([orc.logit(qsum, _bits(K[t]), s) for t in range(n)])
    _close(got, want, rtol=1e-14, atol=1e-14, what="group closed form")


def _brute_topk(s, k):
    """Best subset by exhaustive search: maximal score sum, then the
    lexicographically smallest ascending position list (ties to lower positions)."""
    n = len(s)
    keep = min(k, n)
    best = None
    for comb in itertools.combinations(range(n), keep):
        key = (-sum(s[i] for i in comb), comb)
        if best is None or key < best:
            best = key
    out = list(best[1]) if best else []
    return out + [-1] * (k - keep)


def pin_topk_bruteforce(orc):
    """Top-k against exhaustive subset search on tiny inputs with many ties."""
    rs = np.random.RandomState(10)
    for trial in range(60):
        n = rs.randint(1, 10)
        k = rs.randint(1, 11)
        s = rs.randint(-2, 3, size=n).astype(np.float64)
        got = list(orc.topk(s, k))
        want = _brute_topk([int(x) for x in s], k)
        assert got == want, f"trial {trial}: s={s.tolist()} k={k} got {got} want {want}"


def pin_topk_invariants(orc):
    """Larger cases: size, order, dominance, tie rule, padding, signed zero."""
    rs = np.random.RandomState(11)
    n, k = 1000, 100
    s = np.round(rs.randn(n) * 3.0, 1)             # many exact ties
    idx = orc.topk(s, k)
    assert len(idx) == k and np.all(idx >= 0) and np.all(np.diff(idx) > 0)
    chosen = np.zeros(n, bool); chosen[idx] = True
    lo = s[chosen].min()
    assert np.all(s[~chosen] <= lo)
    ties_out = np.where((~chosen) & (s == lo))[0]
    ties_in = np.where(chosen & (s == lo))[0]
    if ties_out.size and ties_in.size:
        assert ties_in.max() < ties_out.min(), "ties must go to the lower position"
    # k >= n: every position, ascending, then -1
    assert list(orc.topk(np.array([3.0, 1.0, 2.0]), 5)) == [0, 1, 2, -1, -1]
    # all equal: the first k positions
    assert list(orc.topk(np.zeros(10), 4)) == [0, 1, 2, 3]
    # -0.0 and +0.0 tie, so the lower position wins
    assert list(orc.topk(np.array([-1.0, 0.0, -0.0, 5.0]), 2)) == [1, 3]
    assert list(orc.topk(np.array([-1.0, -0.0, 0.0, 5.0]), 2)) == [1, 3]
    # negative scores only
    assert list(orc.topk(np.array([-5.0, -1.0, -3.0, -1.0]), 2)) == [1, 3]


def pin_topk_planted(orc):
    """Scores far above the noise are exactly the selected set."""
    rs = np.random.RandomState(12)
    n, k = 5000, 64
    s = rs.randn(n)
    planted = np.sort(rs.choice(n, size=k, replace=False))
    s[planted] += 100.0
    assert np.array_equal(orc.topk(s, k), planted)


def _group_inputs(rs, L, G, n):
    q = [_bits(rs.randn(G, D)) for _ in range(L)]
    K = [_bits(rs.randn(n, D)) for _ in range(L)]
    V = [_bits(rs.randn(n, D)) for _ in range(L)]
    return q, K, V


def pin_sparse_with_all_tokens_is_full(orc):
    """With k = N the persisted set is every position, so sparse equals full."""
    rs = np.random.RandomState(13)
    G, n = 2, 48
    q, K, V = _group_inputs(rs, 1, G, n)
    modes = [O.MODE_FULL_SELECT, O.MODE_SPARSE]
    out, per, _, rc = orc.decode_group(modes, q * 2, K * 2, V * 2, n, n, O.scale_for(D))
    assert rc == O.OK
    assert list(per[0]) == list(range(n))
    _close(out[1], out[0], rtol=1e-12, atol=1e-14, what="k=N sparse vs full")


def pin_sparse_k1_is_argmax_row(orc):
    """With k = 1 the sparse output is the V row of the highest-scoring key."""
    rs = np.random.RandomState(14)
    n = 70
    q, K, V = _group_inputs(rs, 2, 1, n)
    s = O.scale_for(D)
    qf, Kf = O.bits_to_f64(q[0][0]), O.bits_to_f64(K[0])
    best = int(np.argmax(Kf @ qf))
    out, per, _, rc = orc.decode_group([O.MODE_FULL_SELECT, O.MODE_SPARSE], q, K, V, n, 1, s)
    assert rc == O.OK and per[0][0] == best
    _close(out[1][0], O.bits_to_f64(V[1])[best], rtol=0, atol=0, what="k=1")


def pin_schedule_persistence(orc):
    """Sparse layers use the set of the most recent selection layer (Figure 2)."""
    rs = np.random.RandomState(15)
    n, k, G = 200, 8, 1
    A = np.sort(rs.choice(np.arange(1, 100), size=k, replace=False))
    Bset = np.sort(rs.choice(np.arange(100, 200), size=k, replace=False))
    modes = [O.MODE_FULL, O.MODE_FULL_SELECT, O.MODE_SPARSE, O.MODE_FULL_SELECT,
             O.MODE_SPARSE, O.MODE_SPARSE]
    L = len(modes)
    qv = np.zeros(D); qv[0] = 8.0
    q = [_bits(qv.reshape(1, D)) for _ in range(L)]
    K, V = [], []
    for layer in range(L):
        Kl = rs.randint(-1, 2, size=(n, D)).astype(np.float64); Kl[:, 0] = 0.0
        if layer == 1:
            Kl[A, 0] = 16.0
        if layer == 3:
            Kl[Bset, 0] = 16.0
        Vl = np.zeros((n, D))
        Vl[A, 0] = 1.0
        Vl[Bset, 1] = 1.0
        K.append(_bits(Kl)); V.append(_bits(Vl))
    out, per, final, rc = orc.decode_group(modes, q, K, V, n, k, O.scale_for(D))
    assert rc == O.OK
    assert np.array_equal(per[1], A) and np.array_equal(per[2], A)
    assert np.array_equal(per[3], Bset)
    assert np.array_equal(per[4], Bset) and np.array_equal(per[5], Bset)
    assert np.array_equal(final, Bset)
    assert abs(out[2][0][0] - 1.0) < 1e-14 and out[2][0][1] == 0.0
    assert abs(out[4][0][1] - 1.0) < 1e-14 and out[4][0][0] == 0.0


def pin_sparse_before_selection_fails(orc):
    rs = np.random.RandomState(16)
    q, K, V = _group_inputs(rs, 2, 1, 10)
    _, _, _, rc = orc.decode_group([O.MODE_FULL, O.MODE_SPARSE], q, K, V, 10, 4, O.scale_for(D))
    assert rc == O.ERR_NO_SELECTION


def pin_padding_is_skipped(orc):
    """-1 entries of a persisted set are not positions: the sparse output is
    attention over the live entries only."""
    rs = np.random.RandomState(17)
    n = 64
    q, K, V = _group_inputs(rs, 1, 1, n)
    live = np.array([5, 9, 33, 40], dtype=np.int32)
    idx = np.concatenate([live, np.full(4, -1, np.int32)])
    out, _, _, rc = orc.decode_group([O.MODE_SPARSE], q, K, V, n, 8, O.scale_for(D), idx_in=idx)
    assert rc == O.OK
    want = orc.attend(q[0][0], K[0][live], V[0][live], O.scale_for(D))
    _close(out[0][0], want, rtol=1e-13, atol=1e-15, what="padding")


def pin_empty_context(orc):
    """No cached token: the output is zero and the selected set is all padding."""
    rs = np.random.RandomState(18)
    q, K, V = _group_inputs(rs, 2, 2, 4)
    out, per, _, rc = orc.decode_group([O.MODE_FULL_SELECT, O.MODE_SPARSE], q, K, V, 0, 3,
                                       O.scale_for(D))
    assert rc == O.OK
    assert np.all(out == 0.0) and list(per[0]) == [-1, -1, -1]


def pin_gqa_head_mapping(orc):
    """Query head h reads KV head h // G (consecutive heads share a KV head)."""
    B, Hq, Hkv, n = 1, 8, 2, 16
    G = Hq // Hkv
    rs = np.random.RandomState(19)
    q = _bits(rs.randn(B, Hq, D))
    K = _bits(rs.randn(B, Hkv, n, D))
    Vv = np.zeros((B, Hkv, n, D)); Vv[0, 0] = 1.0; Vv[0, 1] = -1.0
    outs, _, rc = orc.decode_step([O.MODE_FULL], [q], [K], [_bits(Vv)], [n], 0, O.scale_for(D))
    assert rc == O.OK
    for h in range(Hq):
        want = 1.0 if h // G == 0 else -1.0
        assert np.allclose(outs[0][0, h], want, rtol=0, atol=1e-14), h


def pin_batched_step_equals_groups(orc):
    """The batched step equals running each (batch, KV head) group alone."""
    rs = np.random.RandomState(20)
    B, Hq, Hkv, Nmax, k = 2, 4, 2, 40, 6
    G = Hq // Hkv
    lens = [40, 23]
    modes = [O.MODE_FULL, O.MODE_FULL_SELECT, O.MODE_SPARSE]
    L = len(modes)
    q = [_bits(rs.randn(B, Hq, D)) for _ in range(L)]
    K = [_bits(rs.randn(B, Hkv, Nmax, D)) for _ in range(L)]
    V = [_bits(rs.randn(B, Hkv, Nmax, D)) for _ in range(L)]
    s = O.scale_for(D)
    outs, idx, rc = orc.decode_step(modes, q, K, V, lens, k, s)
    assert rc == O.OK
    for b in range(B):
        for g in range(Hkv):
            o, _, fin, rc = orc.decode_group(modes, [x[b, g * G:(g + 1) * G] for x in q],
                                             [x[b, g] for x in K], [x[b, g] for x in V],
                                             lens[b], k, s)
            assert rc == O.OK
            assert np.array_equal(fin, idx[b, g])
            for layer in range(L):
                _close(outs[layer][b, g * G:(g + 1) * G], o[layer], rtol=0, atol=0,
                       what=f"b{b} g{g} l{layer}")
    assert np.all(idx[1] < lens[1])


def pin_index_overlap(orc):
    """Set intersection sizes: identity, disjoint sets, symmetry, padding,
    and random sets against Python's own set intersection."""
    a = np.array([3, 9, 12, 40, -1, -1], np.int32)
    assert orc.index_overlap(a, a) == 4                        # padding is no position
    assert orc.index_overlap(a, np.array([0, 1, 2, 4, 5, 6], np.int32)) == 0
    assert orc.index_overlap(np.full(5, -1, np.int32), np.full(5, -1, np.int32)) == 0
    assert orc.index_overlap(a, np.array([40, 3, -1, -1, -1, -1], np.int32)) == 2  # any order
    rs = np.random.RandomState(11)
    for k in (1, 7, 64, 300):
        for _ in range(5):
            n = rs.randint(k, 4 * k + 1)
            x = np.sort(rs.choice(n, k, replace=False)).astype(np.int32)
            y = np.sort(rs.choice(n, k, replace=False)).astype(np.int32)
            y[rs.randint(0, k + 1):] = -1                       # a shorter set
            want = len(set(x.tolist()) & set(int(v) for v in y if v >= 0))
            assert orc.index_overlap(x, y) == want
            assert orc.index_overlap(y, x) == want


def pin_overlap_of_planted_selections(orc):
    """Two selection layers whose scores plant sets sharing m positions select
    sets that overlap in exactly m positions (the Figure 4(a) measure)."""
    rs = np.random.RandomState(12)
    n, k, m = 500, 40, 25
    heavy1 = rs.choice(n, k, replace=False)
    keep = heavy1[:m]
    rest = np.setdiff1d(np.arange(n), heavy1)
    heavy2 = np.concatenate([keep, rs.choice(rest, k - m, replace=False)])
    s1 = rs.rand(n)
    s2 = rs.rand(n)
    s1[heavy1] += 10.0
    s2[heavy2] += 10.0
    assert orc.index_overlap(orc.topk(s1, k), orc.topk(s2, k)) == m


def pin_coverage_closed_forms(orc):
    """Coverage budgets with closed forms: uniform scores need ceil((1 - tau) n)
    tokens; scores -i ln 2 give masses 2^-i / (2 - 2^(1-n)), so the budget is
    the smallest k with (1 - 2^-k) >= (1 - tau)(1 - 2^-n), in any position
    order; k_max caps it."""
    assert orc.coverage_count(np.zeros(10), 0.25, 100) == 8          # 7.5 -> 8
    assert orc.coverage_count(np.zeros(10), 0.25, 5) == 5            # capped
    assert orc.coverage_count(np.full(1000, 3.5), 0.1, 1000) == 900
    n = 20
    geo = -np.arange(n) * math.log(2.0)
    for tau in (0.5, 0.1, 0.01, 0.001):
        want = next(k for k in range(1, n + 1)
                    if 1.0 - 2.0 ** -k >= (1.0 - tau) * (1.0 - 2.0 ** -n))
        assert orc.coverage_count(geo, tau, n) == want
        perm = np.random.RandomState(int(tau * 1e4)).permutation(n)
        assert orc.coverage_count(geo[perm], tau, n) == want
    # one dominant score: p0 = e^10 / (e^10 + 4), the others e^0 / (e^10 + 4)
    z = math.exp(10.0) + 4.0
    s = np.array([10.0, 0.0, 0.0, 0.0, 0.0])
    assert orc.coverage_count(s, 0.01, 5) == 1
    tau = 1e-4
    want = next(k for k in range(1, 6) if (math.exp(10.0) + (k - 1)) / z >= 1.0 - tau)
    assert orc.coverage_count(s, tau, 5) == want == 3
    assert orc.coverage_count(np.zeros(0), 0.1, 4) == 0


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
