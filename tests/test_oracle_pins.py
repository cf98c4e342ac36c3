"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test names the passage it rests on.  Kinds of pin used here: values printed on
the pages (golden fixtures), closed forms, special cases that reduce to a library
routine (numpy matmul / cumsum / softmax), invariants the pages state, and brute force
on tiny integer inputs, where every partial sum is an exact integer in double.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def ints(rng, shape, r=3):
    return rng.integers(-r, r + 1, size=shape).astype(np.float64)


# ---------------------------------------------------------------------------
# cost model and state size: "attention と線形の間", sections 1 and 3 (printed tables)
# ---------------------------------------------------------------------------
def test_cost_model_matches_printed_table(golden):
    for C, state, score, total, area in golden("chunked_cost_model_L1024_d64.txt"):
        cm = oracle.cost_model(1024, 64, int(C))
        assert (cm["state"], cm["score"], cm["total"], cm["intra_memory"]) == (
            int(state), int(score), int(total), int(area))


def test_cost_model_growth_table(golden):
    for L, full, c64 in golden("chunked_growth_d64.txt"):
        L = int(L)
        assert oracle.cost_model(L, 64, L)["total"] == int(full)
        assert oracle.cost_model(L, 64, 64)["total"] == int(c64)
        assert oracle.cost_model(L, 64, L)["is_full_attention"]
    # the page's claims: fixed part never moves; score part x1024 exactly from C=1 to
    # C=1024; the two ends differ by more than 16x; doubling L multiplies C=L by ~4 and
    # C=64 by exactly 2.
    fixed = {oracle.cost_model(1024, 64, c)["state"] for c in (1, 32, 64, 128, 256, 1024)}
    assert fixed == {8388608}
    assert oracle.cost_model(1024, 64, 1024)["score"] == 1024 * oracle.cost_model(1024, 64, 1)[
        "score"]
    assert oracle.cost_model(1024, 64, 1024)["total"] > 16 * oracle.cost_model(1024, 64, 1)[
        "total"]
    assert oracle.cost_model(2048, 64, 64)["total"] == 2 * oracle.cost_model(1024, 64, 64)["total"]
    r = oracle.cost_model(2048, 64, 2048)["total"] / oracle.cost_model(1024, 64, 1024)["total"]
    assert 3.5 < r < 4.0
    assert oracle.cost_model(1024, 64, 1)["is_linear"]


def test_state_vs_kv_table_and_crossover(golden):
    for L, st, kv in golden("chunked_state_vs_kv_d64.txt"):
        assert oracle.state_vs_kv(int(L), 64) == (int(st), int(kv))
    # state size independent of L; state larger than the KV cache while short, smaller
    # once long (crossover at L = d/2 for d_k = d_v = d)
    assert len({oracle.state_vs_kv(L, 64)[0] for L in (1, 7, 128, 10 ** 6)}) == 1
    assert oracle.state_vs_kv(16, 64)[0] > oracle.state_vs_kv(16, 64)[1]
    assert oracle.state_vs_kv(64, 64)[0] < oracle.state_vs_kv(64, 64)[1]


def test_recurrence_state_shape_independent_of_L():
    rng = np.random.default_rng(1)
    for L in (1, 5, 300):
        _, S, z = oracle.state_recurrence(ints(rng, (L, 6)), ints(rng, (L, 6)), ints(rng, (L, 5)),
                                          return_state=True)
        assert S.shape == (6, 5) and z.shape == (6,)


# ---------------------------------------------------------------------------
# orders of evaluation: "attention と線形の間", sections 1 and 2
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,d,dv", [(1, 2, 2), (4, 2, 2), (13, 3, 5), (64, 16, 16)])
def test_causal_definition_is_tril_matmul(L, d, dv):
    """CausalScoresFirst = tril(q k^T) v: exact against numpy's matmul on integers."""
    rng = np.random.default_rng(L * 100 + d)
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, dv))
    ref = np.tril(q @ k.T) @ v
    assert np.array_equal(oracle.scores_first(q, k, v), ref)
    # selected rows only
    rows = [L - 1, 0] if L > 1 else [0]
    assert np.array_equal(oracle.scores_first(q, k, v, rows=rows), ref[rows])
    # normalised: tril(A) v / tril(A) 1, with positive scores
    qp, kp = np.abs(q) + 1, np.abs(k) + 1
    A = np.tril(qp @ kp.T)
    np.testing.assert_allclose(oracle.scores_first(qp, kp, v, normalize=True),
                               (A @ v) / A.sum(1, keepdims=True), rtol=1e-14, atol=0)


@pytest.mark.parametrize("L,d", [(1, 2), (4, 2), (13, 3), (64, 16)])
def test_chunked_equals_definition_for_every_C(L, d):
    """The page fixes: any chunk size gives the same value (C=1 is the state recurrence,
    C=L the masked scores, a non-dividing C changes nothing).  Integers: exact."""
    rng = np.random.default_rng(7 + L)
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, d))
    ref = oracle.scores_first(q, k, v)
    assert np.array_equal(oracle.state_recurrence(q, k, v), ref)
    for C in list(range(-1, L + 3)):
        assert np.array_equal(oracle.chunked(q, k, v, C), ref), C


def test_chunked_normalised_equals_definition():
    rng = np.random.default_rng(3)
    L, d = 37, 4
    q, k, v = np.abs(ints(rng, (L, d))) + 1, np.abs(ints(rng, (L, d))) + 1, ints(rng, (L, d))
    ref = oracle.scores_first(q, k, v, normalize=True)
    for C in (1, 2, 5, 16, 37, 64):
        np.testing.assert_allclose(oracle.chunked(q, k, v, C, normalize=True), ref, rtol=1e-14)
    np.testing.assert_allclose(oracle.state_recurrence(q, k, v, normalize=True), ref, rtol=1e-14)


def test_negative_control_unmasked_intra_fails():
    """The page reports a first version whose chunk interiors were unmasked; it matched
    neither end.  The planted mistake must be visible to the parity check."""
    rng = np.random.default_rng(11)
    L, d = 16, 4
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, d))
    ref = oracle.scores_first(q, k, v)
    for C in (2, 4, 8, 16):
        bad = oracle.chunked(q, k, v, C, unmasked_intra=True)
        assert not np.array_equal(bad, ref)
    # at C=1 the mask excludes nothing, so the planted mistake is invisible there
    assert np.array_equal(oracle.chunked(q, k, v, 1, unmasked_intra=True), ref)


def test_noncausal_orders_agree_and_last_row(golden):
    """Section 1: (q k^T) v == q (k^T v).  The printed example shows the causal and
    non-causal outputs share their last row (18 20): the last query sees every key."""
    rows = {r[0]: [int(x) for x in r[1:]] for r in golden("chunked_worked_example_outputs.txt")}
    assert rows["noncausal"][-2:] == rows["causal_C1"][-2:]
    assert all(rows[f"causal_C{c}"] == rows["causal_C1"] for c in (2, 3, 4))
    rng = np.random.default_rng(5)
    for L, d in ((4, 2), (9, 3), (40, 8)):
        q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, d))
        sf = oracle.scores_first(q, k, v, causal=False)
        assert np.array_equal(sf, (q @ k.T) @ v)
        assert np.array_equal(oracle.state_first(q, k, v), sf)
        assert np.array_equal(oracle.scores_first(q, k, v)[-1], sf[-1])


# ---------------------------------------------------------------------------
# recurrent vs parallel cumsum form: Performer page, "因果的Linear Attentionの再帰実装"
# ---------------------------------------------------------------------------
def test_recurrence_equals_parallel_cumsum_form():
    rng = np.random.default_rng(2)
    L, D, dv = 32, 16, 16
    Q, K, V = rng.standard_normal((L, D)) * 0.5, rng.standard_normal((L, D)) * 0.5, \
        rng.standard_normal((L, dv)) * 0.5
    fq, fk = oracle.phi(Q, "elu1"), oracle.phi(K, "elu1")
    S_cum = np.cumsum(fk[:, :, None] * V[:, None, :], axis=0)     # [L, D, dv]
    z_cum = np.cumsum(fk, axis=0)
    par = np.einsum("ti,tij->tj", fq, S_cum) / np.einsum("ti,ti->t", fq, z_cum)[:, None]
    np.testing.assert_allclose(oracle.state_recurrence(fq, fk, V, normalize=True), par,
                               rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# normaliser closed forms
# ---------------------------------------------------------------------------
def test_normaliser_v_ones_gives_one():
    rng = np.random.default_rng(4)
    L, D = 50, 8
    fq, fk = oracle.phi(rng.standard_normal((L, D)), "elu1"), oracle.phi(
        rng.standard_normal((L, D)), "elu1")
    out = oracle.state_recurrence(fq, fk, np.ones((L, 3)), normalize=True)
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)
    out2 = oracle.scores_first(fq, fk, np.ones((L, 3)), normalize=True)
    np.testing.assert_allclose(out2, 1.0, rtol=1e-14)


def test_normaliser_constant_features_is_running_mean():
    """elu+1 of zero inputs is the constant feature 1; the normalised output is then the
    running mean of v."""
    rng = np.random.default_rng(6)
    L, dv = 40, 5
    v = rng.standard_normal((L, dv))
    zeros = np.zeros((L, 7))
    fq, fk = oracle.phi(zeros, "elu1"), oracle.phi(zeros, "elu1")
    assert np.array_equal(fq, np.ones((L, 7)))
    ref = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(oracle.state_recurrence(fq, fk, v, normalize=True), ref,
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(oracle.chunked(fq, fk, v, 8, normalize=True), ref, rtol=1e-13,
                               atol=1e-15)


def test_equal_state_gives_equal_outputs():
    """Two histories with the same (S, z) give the same outputs from then on (the
    state-collision criterion of the sparse-vs-linear essay): a permuted history has the
    same sums."""
    rng = np.random.default_rng(9)
    L, D, dv = 20, 4, 3
    fk = np.abs(ints(rng, (L, D))) + 1
    v = ints(rng, (L, dv))
    perm = rng.permutation(L)
    _, S1, z1 = oracle.state_recurrence(fk, fk, v, return_state=True)
    _, S2, z2 = oracle.state_recurrence(fk[perm], fk[perm], v[perm], return_state=True)
    assert np.array_equal(S1, S2) and np.array_equal(z1, z2)
    q2, k2, v2 = np.abs(ints(rng, (10, D))) + 1, np.abs(ints(rng, (10, D))) + 1, ints(rng, (10, dv))
    o1 = oracle.state_recurrence(q2, k2, v2, normalize=True, S0=S1, z0=z1)
    o2 = oracle.state_recurrence(q2, k2, v2, normalize=True, S0=S2, z0=z2)
    assert np.array_equal(o1, o2)


# ---------------------------------------------------------------------------
# feature maps: Performer page, ELU feature map and FAVOR+
# ---------------------------------------------------------------------------
def test_elu1_closed_form():
    x = np.array([-3.0, -1.0, -1e-300, 0.0, 1e-300, 0.5, 2.0])
    out = oracle.phi(x[None, :], "elu1")[0]
    ref = np.array([math.exp(-3.0), math.exp(-1.0), 1.0, 1.0, 1.0, 1.5, 3.0])
    np.testing.assert_allclose(out, ref, rtol=1e-15)
    assert (oracle.phi(np.linspace(-30, 30, 1001)[None, :], "elu1") > 0).all()


def test_favor_single_feature_closed_form():
    """One feature row omega = e_0, d = 16: phi(x) = exp(x_0/2 - |x|^2/8) / 1."""
    d = 16
    om = np.zeros((1, d))
    om[0, 0] = 1.0
    x = np.linspace(-1, 1, d)[None, :]
    xs = x / d ** 0.25
    ref = math.exp(xs[0, 0] - 0.5 * float((xs @ xs.T)[0, 0]))
    assert oracle.phi(x, "favor", om)[0, 0] == pytest.approx(ref, rel=1e-15)


def test_favor_is_unbiased_for_exp_kernel():
    """E[phi(q)^T phi(k)] = exp(q_hat . k_hat) for omega rows i.i.d. N(0, I) (the
    Gaussian moment generating function, Performer page, FAVOR+ derivation).  With
    m = 65536 features the estimate is within 5 standard errors."""
    d, m = 8, 65536
    rng = np.random.default_rng(12)
    q, k = rng.standard_normal((1, d)) * 0.7, rng.standard_normal((1, d)) * 0.7
    om = synth.iid_gaussian(3, m, d)
    fq, fk = oracle.phi(q, "favor", om), oracle.phi(k, "favor", om)
    terms = fq[0] * fk[0] * m                       # per-feature estimator samples
    est, se = terms.mean(), terms.std() / math.sqrt(m)
    truth = math.exp(float(((q / d ** 0.25) @ (k / d ** 0.25).T)[0, 0]))
    assert abs(est - truth) < 5 * se
    assert abs(float(fq[0] @ fk[0]) - est) < 1e-12 * truth
    assert (fq > 0).all()


def _softmax_attention(Q, K, V):
    s = Q @ K.T / np.sqrt(Q.shape[1])
    s -= s.max(1, keepdims=True)
    e = np.exp(s)
    return (e / e.sum(1, keepdims=True)) @ V


def test_favor_approximates_softmax_at_printed_scale(golden):
    """Loose sanity check against the page's printed error order (about 1e-4 at n=64,
    d=32, m=64): the mean over draws stays within a factor 30 of it."""
    p = {r[0]: r[1] for r in golden("performer_mse_vs_softmax.txt")}
    n, d, m, sc, order = int(p["n"]), int(p["d"]), int(p["m"]), float(p["scale"]), float(
        p["mse_order"])
    mses = []
    for seed in range(5):
        g = np.random.default_rng(1000 + seed)
        Q, K, V = (g.standard_normal((n, d)) * sc for _ in range(3))
        om = synth.block_orthogonal_gaussian(seed, m, d).astype(np.float64)
        out = oracle.scores_first(oracle.phi(Q, "favor", om), oracle.phi(K, "favor", om), V,
                                  causal=False, normalize=True)
        mses.append(np.mean((out - _softmax_attention(Q, K, V)) ** 2))
    assert order / 30 < np.mean(mses) < order * 30


def test_favor_error_falls_with_m():
    """The page's m sweep: the error falls as m grows (roughly 1/sqrt(m))."""
    n, d = 128, 64
    g = np.random.default_rng(77)
    Q, K, V = (g.standard_normal((n, d)) * 0.4 for _ in range(3))
    ref = _softmax_attention(Q, K, V)

    def mse(m):
        vals = []
        for seed in range(6):
            om = synth.block_orthogonal_gaussian(seed + 10 * m, m, d).astype(np.float64)
            out = oracle.scores_first(oracle.phi(Q, "favor", om), oracle.phi(K, "favor", om), V,
                                      causal=False, normalize=True)
            vals.append(np.mean((out - ref) ** 2))
        return np.mean(vals)

    assert mse(512) < mse(8) / 4


def test_block_orthogonal_omega():
    """Performer page, orthogonal random features: rows within each d x d block are
    mutually orthogonal; the row norms are chi(d) draws (mean near sqrt(d))."""
    m, d = 256, 64
    om = synth.block_orthogonal_gaussian(5, m, d).astype(np.float64)
    assert om.shape == (m, d)
    for b in range(m // d):
        blk = om[b * d:(b + 1) * d]
        G = blk @ blk.T
        off = G - np.diag(np.diag(G))
        assert np.abs(off).max() < 1e-4 * np.diag(G).max()
    norms = np.linalg.norm(om, axis=1)
    assert abs(norms.mean() - math.sqrt(d)) < 0.5


# ---------------------------------------------------------------------------
# log-linear mask: Log Linear Attention slides 15-22 and 34
# ---------------------------------------------------------------------------
def test_fenwick_buckets_t7_match_slides(golden):
    rows = golden("loglinear_fenwick_t7.txt")
    buckets = {int(r[0]): sorted(int(x) for x in r[1:]) for r in rows if r[0] != "boundaries"}
    got = {}
    for s in range(8):
        got.setdefault(oracle.fenwick_level(7, s), []).append(s)
    assert {k: sorted(v) for k, v in got.items()} == buckets
    # slide 20: boundaries 7 -> 6 -> 4 -> 0 by removing the lowest set bit
    b = [int(x) for x in next(r for r in rows if r[0] == "boundaries")[1:]]
    seq, t = [7], 7
    while t:
        t -= t & -t
        seq.append(t)
    assert seq == b


def test_fenwick_bucket_sizes_partition_the_past():
    for t in range(0, 300):
        counts = {}
        for s in range(t + 1):
            lv = oracle.fenwick_level(t, s)
            counts[lv] = counts.get(lv, 0) + 1
        assert counts.pop(0) == 1
        for lv, c in counts.items():
            assert (t >> (lv - 1)) & 1 == 1 and c == 2 ** (lv - 1)
        assert max(counts, default=0) <= synth.num_levels(t + 1) - 1


@pytest.mark.parametrize("L", [1, 2, 7, 8, 33, 64, 100])
def test_loglinear_recurrence_equals_definition(L):
    """The Fenwick decoding recurrence (slide 22, as read for the XOR level rule)
    reproduces the masked definition exactly on integers with integer weights."""
    rng = np.random.default_rng(L)
    d = 3
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, 2))
    nl = synth.num_levels(L)
    lam = rng.integers(0, 4, size=(L, nl)).astype(np.float64)
    ref = oracle.scores_first(q, k, v, lam=lam)
    assert np.array_equal(oracle.loglinear_recurrence(q, k, v, lam), ref)
    # normalised with positive features
    qp, kp = np.abs(q) + 1, np.abs(k) + 1
    lamp = lam + 1
    np.testing.assert_allclose(oracle.loglinear_recurrence(qp, kp, v, lamp, normalize=True),
                               oracle.scores_first(qp, kp, v, lam=lamp, normalize=True),
                               rtol=1e-13)


def test_loglinear_all_weights_one_is_linear_attention():
    """Slide 17: with every lambda equal to 1 the log-linear form is linear attention."""
    rng = np.random.default_rng(21)
    L, d = 70, 4
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, d))
    lam = np.ones((L, synth.num_levels(L)))
    assert np.array_equal(oracle.loglinear_recurrence(q, k, v, lam), oracle.scores_first(q, k, v))


def test_loglinear_only_level0_is_diagonal():
    rng = np.random.default_rng(22)
    L, d = 30, 4
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, 3))
    lam = np.zeros((L, synth.num_levels(L)))
    lam[:, 0] = rng.integers(1, 5, size=L)
    ref = (lam[:, 0] * np.einsum("ti,ti->t", q, k))[:, None] * v
    assert np.array_equal(oracle.loglinear_recurrence(q, k, v, lam), ref)


def test_loglinear_low_levels_only_is_block_diagonal():
    """Slide 34: level 0 plus levels inside a chunk of C = 2^c tokens form the
    block-diagonal part D; zeroing levels >= 1 + c leaves per-chunk masked attention."""
    rng = np.random.default_rng(23)
    L, d, C = 64, 4, 8
    q, k, v = ints(rng, (L, d)), ints(rng, (L, d)), ints(rng, (L, 3))
    lam = np.ones((L, synth.num_levels(L)))
    lam[:, 1 + int(math.log2(C)):] = 0.0
    out = oracle.loglinear_recurrence(q, k, v, lam)
    for c0 in range(0, L, C):
        sl = slice(c0, c0 + C)
        assert np.array_equal(out[sl], np.tril(q[sl] @ k[sl].T) @ v[sl])


def test_noncausal_normalised_equals_matrix_products():
    """Bidirectional normalised form ("Linear Attention / Performerの理論と実装", the
    non-causal normalised output): out = (phi(Q) phi(K)^T V) / (phi(Q) phi(K)^T 1), a plain
    matrix-product expression computed here with numpy; both oracle orders must match it."""
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=(2, 37, 6)), rng.normal(size=(2, 37, 6))
    v = rng.normal(size=(2, 37, 5))
    for fm in ("elu1", "identity"):
        fq = np.where(q >= 0, q + 1, np.exp(q)) if fm == "elu1" else q
        fk = np.where(k >= 0, k + 1, np.exp(k)) if fm == "elu1" else k
        A = fq @ np.swapaxes(fk, 1, 2)
        for norm in (False, True):
            want = A @ v
            if norm:
                want = want / A.sum(-1, keepdims=True)
            for method in ("recurrence", "scores_first"):
                got = oracle.forward(q, k, v, fm=fm, normalize=norm, method=method, causal=False)
                assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (fm, norm, method)


# ---------------------------------------------------------------------------
# Retention decay: "Linear Attention / Performerの理論と実装", the section on the RNN
# without forgetting (S_t = gamma S_{t-1} + phi(k_t) v_t^T, 0 < gamma < 1)
# ---------------------------------------------------------------------------
def _decay_both(q, k, v, gamma, normalize=False):
    a = oracle.forward(q, k, v, normalize=normalize, gamma=gamma, method="recurrence")
    b = oracle.forward(q, k, v, normalize=normalize, gamma=gamma, method="scores_first")
    return a, b


@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.98])
def test_decay_geometric_series_closed_form(gamma):
    """One feature, q = k = v = 1: y_t = sum_{s<=t} gamma^(t-s) = (1 - gamma^(t+1)) / (1 -
    gamma).  A wrong exponent (gamma^(t-s+1), gamma^(s-t)) or decaying after the write
    breaks it at t = 0 already."""
    L = 40
    one = np.ones((1, L, 1))
    t = np.arange(L)
    want = (1 - gamma ** (t + 1)) / (1 - gamma)
    for got in _decay_both(one, one, one, gamma):
        assert np.allclose(got[0, :, 0], want, rtol=1e-13, atol=0)


def test_decay_single_value_spike():
    """Only v_{s0} is non-zero: y_t = gamma^(t-s0) (q_t . k_{s0}) v_{s0} for t >= s0 and 0
    before, with random q, k (fixes the direction of the exponent and the index s)."""
    rng = np.random.default_rng(11)
    L, d, dv, s0, gamma = 30, 5, 3, 7, 0.83
    q, k = rng.normal(size=(1, L, d)), rng.normal(size=(1, L, d))
    v = np.zeros((1, L, dv))
    v[0, s0] = rng.normal(size=dv)
    want = np.zeros((L, dv))
    for t in range(s0, L):
        want[t] = gamma ** (t - s0) * (q[0, t] @ k[0, s0]) * v[0, s0]
    for got in _decay_both(q, k, v, gamma):
        assert np.allclose(got[0], want, rtol=1e-12, atol=1e-14)


def test_decay_gamma_one_is_plain_linear_attention():
    """gamma = 1 leaves the additive update S_t = S_{t-1} + phi(k_t) v_t^T: on small
    integers both decay routines equal numpy's tril(q k^T) v exactly."""
    rng = np.random.default_rng(12)
    q, k, v = ints(rng, (2, 23, 4)), ints(rng, (2, 23, 4)), ints(rng, (2, 23, 3))
    want = np.stack([np.tril(q[h] @ k[h].T) @ v[h] for h in range(2)])
    for got in _decay_both(q, k, v, 1.0):
        assert np.array_equal(got, want)


def test_decay_normalised_constant_values():
    """Normalised with z decaying alike, y_t is a weighted mean of the values: constant
    values come back unchanged for any gamma (positive elu+1 features keep den > 0)."""
    rng = np.random.default_rng(13)
    q, k = rng.normal(size=(1, 50, 6)), rng.normal(size=(1, 50, 6))
    v = np.full((1, 50, 4), 2.5)
    for gamma in (0.6, 0.95):
        for method in ("recurrence", "scores_first"):
            got = oracle.forward(q, k, v, fm="elu1", normalize=True, gamma=gamma, method=method)
            assert np.allclose(got, 2.5, rtol=1e-13)


def test_decay_matrix_form_with_numpy():
    """The decayed causal output as one matrix expression, numpy only: (Q K^T * G) V with
    G[t, s] = gamma^(t-s) for s <= t, 0 above the diagonal; normalised rows divide by
    the row sums of Q K^T * G."""
    rng = np.random.default_rng(14)
    L, gamma = 45, 0.9
    q, k = rng.normal(size=(2, L, 5)), rng.normal(size=(2, L, 5))
    v = rng.normal(size=(2, L, 3))
    t = np.arange(L)
    G = np.tril(gamma ** (t[:, None] - t[None, :]).clip(min=0))
    for norm in (False, True):
        fq = np.where(q >= 0, q + 1, np.exp(q))
        fk = np.where(k >= 0, k + 1, np.exp(k))
        A = (fq @ np.swapaxes(fk, 1, 2)) * G
        want = A @ v
        if norm:
            want = want / A.sum(-1, keepdims=True)
        for m in ("recurrence", "scores_first"):
            got = oracle.forward(q, k, v, fm="elu1", normalize=norm, gamma=gamma, method=m)
            assert np.allclose(got, want, rtol=1e-11, atol=1e-12), norm


def test_decay_printed_retention_after_ten_steps(golden):
    """"Kimi K3 と Qwen 3.8 の Attention 機構比較分析", section 3.3.7: a memory written at
    step 0 whose later keys are all orthogonal to it keeps gamma^t of itself; the page
    prints about 0.82 for gamma = 0.98 after 10 steps.  Here: key e_1 with value 1 at
    t = 0, keys e_2 (value 0) after, and the query e_1 reads the memory at t = 10."""
    (gamma, steps, printed), = golden("decay_retention_gamma098_t10.txt")
    gamma, steps, printed = float(gamma), int(steps), float(printed)
    L, D = steps + 1, 2
    k = np.zeros((1, L, D)); k[0, 0, 0] = 1; k[0, 1:, 1] = 1
    q = np.zeros((1, L, D)); q[0, :, 0] = 1
    v = np.zeros((1, L, 1)); v[0, 0, 0] = 1
    for got in _decay_both(q, k, v, gamma):
        kept = got[0, steps, 0]
        assert abs(kept - printed) < 0.005
        assert kept == pytest.approx(gamma ** steps, rel=1e-14)


# ---------------------------------------------------------------------------
# backward pass: the chain rule on the definition, pinned by finite differences of the
# oracle's forward recurrence (another code path) and by numpy matrix products
# ---------------------------------------------------------------------------
def _fd_grads(q, k, v, dout, fm, omega, normalize, gamma, eps=1e-6):
    """Central differences of loss = sum(out * dout) through oracle.forward (recurrence)."""
    def loss(qq, kk, vv):
        out = oracle.forward(qq[None], kk[None], vv[None], fm=fm, omega=omega,
                             normalize=normalize, gamma=gamma, method="recurrence")[0]
        return float((out * dout).sum())
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(*g.shape):
            plus = [b.copy() for b in base]
            minus = [b.copy() for b in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("fm", ["identity", "elu1", "favor"])
@pytest.mark.parametrize("normalize", [False, True])
@pytest.mark.parametrize("gamma", [None, 0.8])
def test_backward_matches_finite_differences(fm, normalize, gamma):
    rng = np.random.default_rng(31)
    L, d, dv = 7, 3, 2
    q, k = rng.normal(size=(L, d)) * 0.7, rng.normal(size=(L, d)) * 0.7
    if fm == "identity" and normalize:
        q, k = np.abs(q) + 0.2, np.abs(k) + 0.2  # keep the denominators away from zero
    v, dout = rng.normal(size=(L, dv)), rng.normal(size=(L, dv))
    omega = synth.block_orthogonal_gaussian(5, 8, d) if fm == "favor" else None
    dq, dk, dvv = oracle.backward(q[None], k[None], v[None], dout[None], fm=fm, omega=omega,
                                  normalize=normalize, gamma=gamma)
    fq, fk, fv = _fd_grads(q, k, v, dout, fm, omega, normalize, gamma)
    for got, want in ((dq[0], fq), (dk[0], fk), (dvv[0], fv)):
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7), np.abs(got - want).max()


def test_backward_identity_unnormalised_is_masked_matmuls():
    """out = tril(Q K^T) V gives dV = tril(Q K^T)^T dO, dQ = tril(dO V^T) K and
    dK = tril(dO V^T)^T Q; on small integers every partial sum is exact."""
    rng = np.random.default_rng(32)
    q, k = ints(rng, (1, 11, 4)), ints(rng, (1, 11, 4))
    v, dout = ints(rng, (1, 11, 3)), ints(rng, (1, 11, 3))
    dq, dk, dvv = oracle.backward(q, k, v, dout)
    A = np.tril(q[0] @ k[0].T)
    G = np.tril(dout[0] @ v[0].T)
    assert np.array_equal(dvv[0], A.T @ dout[0])
    assert np.array_equal(dq[0], G @ k[0])
    assert np.array_equal(dk[0], G.T @ q[0])


# backward under the log-linear mask ("論文紹介：Log Linear Attention", slide 17): the chain
# rule on the masked definition, pinned by finite differences of the Fenwick recurrence
def _fd_grads_ll(q, k, v, dout, lam, fm, omega, normalize, eps=1e-6):
    def loss(qq, kk, vv):
        out = oracle.forward(qq[None], kk[None], vv[None], fm=fm, omega=omega,
                             normalize=normalize, lam=lam[None], method="recurrence")[0]
        return float((out * dout).sum())
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(*g.shape):
            plus = [b.copy() for b in base]
            minus = [b.copy() for b in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            g[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        grads.append(g)
    return grads


@pytest.mark.parametrize("fm", ["identity", "elu1", "favor"])
@pytest.mark.parametrize("normalize", [False, True])
def test_loglinear_backward_matches_finite_differences(fm, normalize):
    rng = np.random.default_rng(37)
    L, d, dv = 11, 3, 2                     # levels 0..4, three of them inter-pair levels
    q, k = rng.normal(size=(L, d)) * 0.7, rng.normal(size=(L, d)) * 0.7
    if fm == "identity" and normalize:
        q, k = np.abs(q) + 0.2, np.abs(k) + 0.2
    v, dout = rng.normal(size=(L, dv)), rng.normal(size=(L, dv))
    lam = rng.uniform(0.1, 1.0, size=(L, 5))
    omega = synth.block_orthogonal_gaussian(5, 8, d) if fm == "favor" else None
    dq, dk, dvv = oracle.backward(q[None], k[None], v[None], dout[None], fm=fm, omega=omega,
                                  normalize=normalize, lam=lam[None])
    fq, fk, fv = _fd_grads_ll(q, k, v, dout, lam, fm, omega, normalize)
    for got, want in ((dq[0], fq), (dk[0], fk), (dvv[0], fv)):
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7), np.abs(got - want).max()


def test_loglinear_backward_all_ones_is_plain_backward():
    """lambda == 1 is plain linear attention (slide 17), so its gradients are the plain
    chain rule's."""
    rng = np.random.default_rng(38)
    L, d, dv = 40, 4, 3
    fq, fk = np.abs(rng.normal(size=(L, d))), np.abs(rng.normal(size=(L, d)))
    v, dout = rng.normal(size=(L, dv)), rng.normal(size=(L, dv))
    for normalize in (False, True):
        a = oracle.backward_features(fq, fk, v, dout, normalize, lam=np.ones((L, 7)))
        b = oracle.backward_features(fq, fk, v, dout, normalize)
        for x, y in zip(a, b):
            assert np.allclose(x, y, rtol=1e-13, atol=1e-13)


def test_loglinear_backward_level_zero_only_is_diagonal():
    """Only lambda^(0) nonzero: out_t = lambda_t^(0) (phi(q_t).phi(k_t)) v_t, whose gradients
    are dphi(q)_t = lambda_t^(0) (dout_t.v_t) phi(k_t), dphi(k)_t = lambda_t^(0) (dout_t.v_t)
    phi(q_t) and dv_t = lambda_t^(0) (phi(q_t).phi(k_t)) dout_t, exactly on integers."""
    rng = np.random.default_rng(39)
    L, d, dv = 33, 4, 3
    fq = rng.integers(-3, 4, size=(L, d)).astype(float)
    fk = rng.integers(-3, 4, size=(L, d)).astype(float)
    v = rng.integers(-3, 4, size=(L, dv)).astype(float)
    dout = rng.integers(-3, 4, size=(L, dv)).astype(float)
    lam = np.zeros((L, 7))
    lam[:, 0] = rng.integers(1, 4, size=L)
    dfq, dfk, dvo = oracle.backward_features(fq, fk, v, dout, False, lam=lam)
    g = lam[:, 0] * (dout * v).sum(1)
    a = lam[:, 0] * (fq * fk).sum(1)
    assert np.array_equal(dfq, g[:, None] * fk)
    assert np.array_equal(dfk, g[:, None] * fq)
    assert np.array_equal(dvo, a[:, None] * dout)
