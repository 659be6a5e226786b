"""Pins of the fp64 oracle against facts fixed outside the oracle itself:
published known-answer vectors, the pages' worked numbers, closed forms,
invariants, brute force on tiny inputs and distributional identities checked
by simulation.  No GPU needed."""

import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import dsd_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------- Philox

def test_philox_known_answers():
    kat = _golden("philox4x32_10_kat.json")
    for vec in kat["vectors"]:
        ctr = [int(x, 16) for x in vec["ctr"]]
        key = [int(x, 16) for x in vec["key"]]
        out = [int(x) for x in O.philox4x32_10(*ctr, *key)]
        assert out == [int(x, 16) for x in vec["out"]]


def test_uniform_endpoints_exact_in_fp32():
    u = O.uniform_from_word(np.array([0, 0xFFFFFFFF, 1 << 9, 0x80000000], dtype=np.uint64))
    assert u[0] == 2.0 ** -24
    assert u[1] == 1.0 - 2.0 ** -24
    assert u[2] == 1.5 * 2.0 ** -23
    assert u[3] == 0.5 + 2.0 ** -24
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    assert np.all((u > 0) & (u < 1))


def test_vocab_uniforms_select_word_by_index():
    seed = 0x1234_5678_9ABC_DEF0
    u = O.vocab_uniforms(seed, position=3, req=77, stream=2, V=10)
    for v in range(10):
        words = O.philox4x32_10(v // 4, 3, 77, 2, seed & 0xFFFFFFFF, seed >> 32)
        assert u[v] == O.uniform_from_word(words[v % 4])


def test_gumbel_moments():
    # Standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2/6.
    g = O.vocab_gumbel(seed=99, position=0, req=0, stream=0, V=400_000)
    assert abs(g.mean() - np.euler_gamma) < 0.01
    assert abs(g.var() - math.pi ** 2 / 6) < 0.02


# ------------------------------------------------------------------- survival

def test_survival_worked_example_from_the_page():
    ex = _golden("survival_worked_example.json")
    for case in ex["cases"]:
        conf = np.full((1, case["positions"]), case["c"])
        a = O.survival(conf)
        assert a[0, -1] == pytest.approx(case["a_last"], rel=1e-14)
        assert round(a[0, -1], 3) == case["page_rounded"]
    # the page's point: the optimistic product overstates survival by ~44%
    ratio = 0.377149515625 / 0.262144
    assert 1.43 < ratio < 1.45


def test_survival_clamps_and_is_monotone():
    conf = np.array([[1.5, 0.5, -0.2, 0.9], [0.9, 0.9, 0.9, 1.0]])
    a = O.survival(conf)
    assert a[0].tolist() == [1.0, 0.5, 0.0, 0.0]
    assert np.allclose(a[1], [0.9, 0.81, 0.729, 0.729])
    rng = np.random.default_rng(0)
    a = O.survival(rng.random((50, 7)))
    assert np.all(np.diff(a, axis=1) <= 0)
    with pytest.raises(ValueError):
        O.survival(np.array([[0.5, np.nan]]))


# ---------------------------------------------------------------- Markov bias

def test_markov_bias_one_hot_selects_a_column_of_w():
    # V != r so a transposed table cannot pass silently.
    V, r = 11, 3
    rng = np.random.default_rng(1)
    W = rng.standard_normal((V, r))
    E = np.zeros((V, r))
    E[5, 2] = 1.0
    assert np.array_equal(O.markov_bias(E, W, 5), W[:, 2])
    E[5, 0] = 2.0
    assert np.allclose(O.markov_bias(E, W, 5), W[:, 2] + 2 * W[:, 0])


def test_markov_bias_by_hand_rows():
    g = _golden("markov_propose_by_hand.json")
    E, W = np.array(g["E"], float), np.array(g["W"], float)
    expected = {0: [2, 0, -1, 1], 1: [0, 3, 1, -2], 2: [2, 3, 0, -1], 3: [0, 0, 0, 0]}
    for prev, b in expected.items():
        assert O.markov_bias(E, W, prev).tolist() == b


def test_markov_bias_silu_variant():
    E = np.array([[0.0, 1.0, -30.0]])
    W = np.eye(3)
    b = O.markov_bias(E, W, 0, act="silu")
    assert b[0] == 0.0
    assert b[1] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)  # silu(1)
    assert abs(b[2]) < 1e-11


# -------------------------------------------------------------------- propose

@pytest.mark.parametrize("variant,baf", [("bias_at_first", True), ("no_bias_at_first", False)])
def test_propose_by_hand(variant, baf):
    g = _golden("markov_propose_by_hand.json")
    out = O.propose(np.array(g["U"], float), np.array(g["E"], float), np.array(g["W"], float),
                    np.full((1, 3), 0.9), np.array(g["prev_tok"]), bias_at_first=baf)
    exp = g[variant]
    assert out["tokens"][0].tolist() == exp["tokens"]
    assert out["logit_at_tok"][0].tolist() == exp["logit_at_tok"]
    for j, row in enumerate(exp["logits"]):
        lse = math.log(sum(math.exp(x) for x in row))
        assert out["lse_q"][0, j] == pytest.approx(lse, rel=1e-14)


def test_propose_zero_tables_is_positionwise_argmax():
    rng = np.random.default_rng(2)
    R, G, V, r = 3, 5, 50, 4
    U = rng.standard_normal((R, G, V)) * 2
    out = O.propose(U, np.zeros((V, r)), rng.standard_normal((V, r)), rng.random((R, G)),
                    rng.integers(0, V, R))
    assert np.array_equal(out["tokens"], U.argmax(axis=2))
    assert np.allclose(out["lse_q"], special.logsumexp(U, axis=2), rtol=1e-14)
    assert np.allclose(out["logit_at_tok"], U.max(axis=2))


def test_propose_single_position_matches_dense_transition_matrix():
    # gamma = 1: x = argmax(U_0 + T[prev]) with the V x V transition matrix
    # T = E W^T built explicitly (the low-rank factorisation of the pages).
    rng = np.random.default_rng(3)
    V, r = 40, 6
    E, W = rng.standard_normal((V, r)), rng.standard_normal((V, r))
    T = np.zeros((V, V))
    for i in range(V):
        for v in range(V):
            T[i, v] = sum(E[i, k] * W[v, k] for k in range(r))
    U = rng.standard_normal((8, 1, V))
    prev = rng.integers(0, V, 8)
    out = O.propose(U, E, W, np.ones((8, 1)), prev)
    for rr in range(8):
        assert out["tokens"][rr, 0] == int(np.argmax(U[rr, 0] + T[prev[rr]]))


def test_propose_greedy_brute_force_chain():
    # gamma = 3 chain, tiny V: at every step the chosen token beats every
    # other token under the bias of the previously chosen one.
    rng = np.random.default_rng(4)
    V, r, G = 9, 3, 3
    E, W = rng.standard_normal((V, r)), rng.standard_normal((V, r))
    U = rng.standard_normal((5, G, V))
    prev = rng.integers(0, V, 5)
    out = O.propose(U, E, W, np.ones((5, G)), prev)
    for rr in range(5):
        p = int(prev[rr])
        for j in range(G):
            scores = [U[rr, j, v] + float(np.dot(E[p], W[v])) for v in range(V)]
            assert out["tokens"][rr, j] == max(range(V), key=lambda v: (scores[v], -v))
            p = int(out["tokens"][rr, j])


def test_propose_ties_take_the_lowest_index():
    U = np.zeros((1, 2, 6))
    U[0, 0, [2, 4]] = 1.0
    U[0, 1, [5, 1]] = 3.0
    out = O.propose(U, np.zeros((6, 2)), np.zeros((6, 2)), np.ones((1, 2)), np.array([0]))
    assert out["tokens"][0].tolist() == [2, 1]
    assert out["margin"][0].tolist() == [0.0, 0.0]


def test_propose_sampling_follows_softmax_of_scaled_logits():
    # Gumbel-max sampling: over many seeds, x ~ softmax(l / T).
    V, T = 5, 0.7
    U = np.array([[[0.3, -1.0, 1.2, 0.0, 0.8]]])
    E, W = np.zeros((V, 2)), np.zeros((V, 2))
    n = 8000
    counts = np.zeros(V)
    for s in range(n):
        out = O.propose(U, E, W, np.ones((1, 1)), np.array([0]), temperature=T, seed=1000 + s)
        counts[out["tokens"][0, 0]] += 1
    p = special.softmax(U[0, 0] / T)
    chi2 = stats.chisquare(counts, p * n)
    assert chi2.pvalue > 1e-3
    out = O.propose(U, E, W, np.ones((1, 1)), np.array([0]), temperature=T, seed=5)
    x = out["tokens"][0, 0]
    assert out["lse_q"][0, 0] == pytest.approx(special.logsumexp(U[0, 0] / T), rel=1e-14)
    assert out["logit_at_tok"][0, 0] == pytest.approx(U[0, 0, x] / T, rel=1e-14)


def test_propose_sampling_depends_on_request_id_not_slot():
    rng = np.random.default_rng(6)
    V = 30
    U = rng.standard_normal((2, 3, V))
    E, W = rng.standard_normal((V, 2)), rng.standard_normal((V, 2))
    prev = np.array([3, 9])
    a = O.propose(U, E, W, np.ones((2, 3)), prev, req_id=np.array([10, 20]), temperature=1.0, seed=7)
    b = O.propose(U[::-1], E, W, np.ones((2, 3)), prev[::-1], req_id=np.array([20, 10]),
                  temperature=1.0, seed=7)
    assert np.array_equal(a["tokens"], b["tokens"][::-1])


# ------------------------------------------------------------------- schedule

def test_schedule_by_hand():
    g = _golden("schedule_by_hand.json")
    a = O.survival(np.array(g["conf"]))
    assert np.allclose(a, g["survival"], rtol=1e-15)
    for case in g["cases"]:
        out = O.schedule(np.array(g["survival"]), np.array(case["sps"], float))
        assert out["keep_len"].tolist() == case["keep_len"]
        assert out["theta"] == pytest.approx(case["theta"], rel=1e-14)
        assert out["B"] == case["B"]


def _theta(a, sps, ls):
    R = a.shape[0]
    B = sum(1 + l for l in ls)
    if B > len(sps):
        return -np.inf
    tau = sum(1 + a[r, :ls[r]].sum() for r in range(R))
    return tau * sps[B - 1]


@pytest.mark.parametrize("seed", range(12))
def test_schedule_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 5))
    G = int(rng.integers(1, 4))
    a = O.survival(rng.random((R, G)) ** 0.5)
    n = R * (G + 1) - int(rng.integers(0, 2))       # sometimes one slot short
    n = max(n, R)
    knee = rng.uniform(0, n)
    sps = 1.0 / (1.0 + rng.uniform(0.01, 0.5) * np.maximum(0.0, np.arange(1, n + 1) - knee))
    best = max(_theta(a, sps, ls) for ls in itertools.product(range(G + 1), repeat=R))
    out = O.schedule(a, sps)
    assert out["theta"] == pytest.approx(best, rel=1e-12)
    assert _theta(a, sps, out["keep_len"]) == pytest.approx(best, rel=1e-12)


def test_schedule_constant_sps_keeps_everything():
    rng = np.random.default_rng(7)
    a = O.survival(0.05 + 0.95 * rng.random((6, 7)))
    out = O.schedule(a, np.full(6 * 8, 1e3))
    assert out["keep_len"].tolist() == [7] * 6


def test_schedule_flat_then_inverse_table_keeps_nothing():
    # SPS = 1e3 up to B = R, then proportional to 1/B: Theta is proportional
    # to tau/B, which starts at 1 and drops with every slot of survival < 1.
    rng = np.random.default_rng(8)
    R = 12
    a = O.survival(rng.beta(5, 2, size=(R, 7)))
    B = np.arange(1, 129, dtype=float)
    sps = np.where(B <= R, 1e3, 1e3 * R / B)
    out = O.schedule(a, sps)
    assert out["keep_len"].tolist() == [0] * R
    assert out["theta"] == pytest.approx(R * 1e3)


def test_schedule_result_is_a_prefix_per_request_even_with_ties():
    a = np.array([[1.0, 1.0, 0.5], [1.0, 0.5, 0.5]])
    sps = np.array([100, 100, 100, 100, 99, 98, 70, 10], float)
    out = O.schedule(a, sps)
    items = out["sorted_items"]
    assert [(r, j) for _, r, j in items[:5]] == [(0, 0), (0, 1), (1, 0), (0, 2), (1, 1)]
    # Theta by cut k = 0..6: 200, 300, 400, 495, 539, 420, 65  ->  k* = 4
    assert out["keep_len"].tolist() == [3, 1]
    assert out["theta"] == pytest.approx(539.0)


# --------------------------------------------------------------------- verify

def test_verify_greedy_by_hand():
    P = np.zeros((1, 4, 4))
    P[0, 0] = [5, 1, 0, 0]     # argmax 0
    P[0, 1] = [0, 0, 1, 4]     # argmax 3
    P[0, 2] = [0, 6, 2, 0]     # argmax 1
    P[0, 3] = [0, 0, 0, 9]     # argmax 3
    tokens = np.array([[0, 3, 2]])
    U = np.zeros((1, 3, 4))
    E = W = np.zeros((4, 2))
    for kl, acc, nxt in [(3, 2, 1), (2, 2, 1), (1, 1, 3), (0, 0, 0)]:
        out = O.verify(P, U, E, W, np.array([0]), tokens, np.array([kl]))
        assert (out["accept_len"][0], out["next_token"][0]) == (acc, nxt)
    tokens2 = np.array([[0, 3, 1]])
    out = O.verify(P, U, E, W, np.array([0]), tokens2, np.array([3]))
    assert (out["accept_len"][0], out["next_token"][0]) == (3, 3)   # bonus row 3


def test_verify_identical_distributions_accept_everything():
    rng = np.random.default_rng(9)
    V, G = 20, 4
    U = rng.standard_normal((2, G, V))
    E, W = rng.standard_normal((V, 3)) * 0.5, rng.standard_normal((V, 3)) * 0.5
    prev = np.array([1, 2])
    prop = O.propose(U, E, W, np.ones((2, G)), prev, temperature=0.9, seed=3)
    P = np.zeros((2, G + 1, V))
    for r in range(2):
        for t in range(G):
            P[r, t] = O._draft_logits(U, E, W, prev, prop["tokens"], r, t, True, "none")
        P[r, G] = rng.standard_normal(V)
    out = O.verify(P, U, E, W, prev, prop["tokens"], np.array([G, 2]), temperature=0.9, seed=3)
    assert out["accept_len"].tolist() == [G, 2]


def _committed(out, tokens, r=0):
    k = int(out["accept_len"][r])
    return list(tokens[r, :k]) + [int(out["next_token"][r])]


def test_verify_rejection_sampling_reproduces_the_target_distribution():
    # The pages' losslessness claim: the first committed token is distributed
    # as p_0, and given that position 0 was accepted the second one is
    # distributed as p_1, whatever q is.  Checked by simulation over seeds.
    V, T = 4, 0.8
    U = np.array([[[1.5, 0.0, -0.5, 0.3], [0.0, 1.0, 0.2, -1.0]]])
    E = np.array([[0.5, 0.0], [0.0, 0.7], [0.3, 0.3], [-0.4, 0.2]])
    W = np.array([[1.0, -0.5], [0.2, 0.8], [-0.6, 0.1], [0.4, 0.4]])
    P = np.array([[[0.0, 1.0, 0.5, -0.5], [1.2, -0.3, 0.0, 0.6], [0.0, 0.0, 2.0, 0.0]]])
    prev = np.array([2])
    p0 = special.softmax(P[0, 0] / T)
    p1 = special.softmax(P[0, 1] / T)
    n = 6000
    first = np.zeros(V)
    second = np.zeros(V)
    for s in range(n):
        prop = O.propose(U, E, W, np.ones((1, 2)), prev, temperature=T, seed=50_000 + s)
        out = O.verify(P, U, E, W, prev, prop["tokens"], np.array([2]), temperature=T,
                       seed=50_000 + s)
        seq = _committed(out, prop["tokens"])
        first[seq[0]] += 1
        if len(seq) >= 2:
            second[seq[1]] += 1
    assert stats.chisquare(first, p0 * n).pvalue > 1e-3
    m = second.sum()
    assert m > 1000
    assert stats.chisquare(second, p1 * m).pvalue > 1e-3
    # q differs from p, so the test is not vacuous
    q0 = special.softmax((U[0, 0] + W @ E[2]) / T)
    assert 0.5 * np.abs(q0 - p0).sum() > 0.1


def _random_pair(rng, V, p_zero=False, q_equal=False):
    p = rng.dirichlet(np.full(V, 0.7))
    if p_zero:
        p[rng.integers(V)] = 0.0
        p /= p.sum()
    q = p.copy() if q_equal else rng.dirichlet(np.full(V, 0.7))
    return p, q


def _commit_distribution(p, q):
    """Distribution of the token committed at one position when the draft
    proposes x ~ q and the oracle's accept test and correction draw decide,
    summed exactly over every draft outcome x."""
    out = np.zeros_like(p)
    for x in range(p.size):
        if q[x] == 0.0:
            continue                      # the draft never proposes x
        a = O.accept_probability(p[x], q[x])
        w, _ = O.correction_weights(p, q)
        out[x] += q[x] * a
        out += q[x] * (1.0 - a) * (w / w.sum())
    return out


@pytest.mark.parametrize("V", [2, 3, 4, 5])
def test_rejection_step_is_exactly_lossless(V):
    # [WALK] 4.4 / [READ] 3.1 (acceptance as overlap, lossless verification):
    # sum_x q(x) [min(1, p/q) delta_{x=v} + (1 - min(1, p/q)) res(v)] = p(v)
    # for every v, by exact enumeration over the draft outcome x
    rng = np.random.default_rng(100 + V)
    cases = [_random_pair(rng, V) for _ in range(40)]
    cases += [_random_pair(rng, V, p_zero=True) for _ in range(10)]
    cases += [_random_pair(rng, V, q_equal=True) for _ in range(3)]
    q_one_hot = np.zeros(V)
    q_one_hot[V - 1] = 1.0
    cases.append((rng.dirichlet(np.ones(V)), q_one_hot))    # a point-mass draft
    for p, q in cases:
        assert np.max(np.abs(_commit_distribution(p, q) - p)) <= 1e-12
    # the probability of accepting is the overlap sum_v min(p, q)
    for p, q in cases:
        acc = sum(q[x] * O.accept_probability(p[x], q[x]) for x in range(V) if q[x] > 0)
        assert abs(acc - np.minimum(p, q).sum()) <= 1e-12


def test_rejection_two_positions_joint_is_exact():
    # Two drafted positions where both the draft q1 and the target p1 of the
    # second position depend on the first token (the Markov head does this to
    # q).  The first two committed tokens (a, b) must have the target's joint
    # law p0(a) p1(b | a).  A rejection at position 0 ends the cycle; the
    # second token then comes from the target itself, p1(. | a).
    rng = np.random.default_rng(7)
    for V in (2, 3, 4):
        for _ in range(10):
            p0, q0 = _random_pair(rng, V)
            p1 = rng.dirichlet(np.full(V, 0.7), size=V)   # p1[a] = p1(. | a)
            q1 = rng.dirichlet(np.full(V, 0.7), size=V)
            J = np.zeros((V, V))
            for x0 in range(V):
                a0 = O.accept_probability(p0[x0], q0[x0])
                w0, _ = O.correction_weights(p0, q0)
                c0 = w0 / w0.sum()
                # accepted at 0: position 1 is verified against p1(. | x0)
                J[x0] += q0[x0] * a0 * _commit_distribution(p1[x0], q1[x0])
                # rejected at 0: a ~ c0 and b ~ p1(. | a)
                J += q0[x0] * (1.0 - a0) * c0[:, None] * p1
            assert np.max(np.abs(J - p0[:, None] * p1)) <= 1e-12


def test_correction_weights_by_hand_and_empty_residual():
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.5, 0.3])
    w, fb = O.correction_weights(p, q)
    assert not fb and np.allclose(w, [0.3, 0.0, 0.0], atol=1e-15)
    w, fb = O.correction_weights(p, p.copy())
    assert fb and np.array_equal(w, p)                 # empty residual: draw from p
    tiny = p.copy()
    tiny[0] += 1e-14
    tiny[1] -= 1e-14
    w, fb = O.correction_weights(tiny, p)               # residual 1e-14 <= 1e-12: fall back
    assert fb and np.array_equal(w, tiny)
    assert O.accept_probability(0.3, 0.5) == 0.6
    assert O.accept_probability(0.5, 0.2) == 1.0


def test_verify_uses_the_accept_threshold_and_the_empty_residual_fallback(monkeypatch):
    # T = 1, no Markov bias (E = W = 0), so q = softmax(U[0, 0]) and
    # p = softmax(P[0, 0]).  The draft token 3 is very unlikely under q
    # (q(3) ~ 3e-9) and P lowers its logit by about 1e-6: accept probability
    # about 1 - 1e-6, residual mass about 3e-15.
    V = 4
    U = np.array([[[0.0, 5.0, 2.0, -15.0]]])
    P = np.zeros((1, 2, V))
    P[0, 0] = U[0, 0]
    P[0, 0, 3] += math.log(1.0 - 1e-6)
    P[0, 1] = [0.0, 1.0, 0.0, 0.0]
    E = np.zeros((V, 2))
    W = np.zeros((V, 2))
    tokens = np.array([[3]])
    q = special.softmax(U[0, 0])
    p = special.softmax(P[0, 0])
    thr = min(1.0, p[3] / q[3])
    assert 1.0 - 2e-6 < thr < 1.0
    # the correction noise: +100 on token 3, so a draw from p picks 3 while
    # a draw from the residual (which is 0 at token 3) cannot
    monkeypatch.setattr(O, "vocab_gumbel",
                        lambda seed, pos, req, stream, V_: np.array([0.0, 0.0, 0.0, 100.0]))

    def run(u):
        monkeypatch.setattr(O, "accept_uniform", lambda seed, t, req: u)
        out = O.verify(P, U, E, W, np.array([0]), tokens, np.array([1]), temperature=1.0)
        return int(out["accept_len"][0]), int(out["next_token"][0])

    # u just below the threshold: accepted, then the bonus row (argmax + noise)
    assert run(thr - 1e-9) == (1, 3)
    # u just above: rejected; the residual sum (~3e-15) is below 1e-12 sum(p),
    # so the correction is drawn from p and the +100 noise selects token 3
    assert run(1.0 - 2.0 ** -24) == (0, 3)
    # a larger gap between p and q at token 3: a real residual, which is zero
    # at token 3, so the correction is the residual's best entry instead
    P[0, 0, 3] = -16.0
    q2 = special.softmax(P[0, 0])
    res = np.maximum(0.0, q2 - q)
    assert res.sum() > 1e-12 and res[3] == 0.0
    assert run(1.0 - 2.0 ** -24) == (0, int(np.argmax(np.where(res > 0, np.log(res), -np.inf))))


def test_top2_margin_by_hand():
    assert O.top2_margin([1.0, 3.5, 2.25, -1.0]) == 1.25
    assert O.top2_margin([2.0, 2.0, 1.0]) == 0.0
    assert O.top2_margin([7.0]) == float("inf")
    # the exemption rule's input from a greedy proposal: with no Markov bias
    # each position's margin is the gap between its two largest base logits
    U = np.zeros((1, 2, 5))
    U[0, 0] = [0.0, 5.0, 4.9995, 1.0, -2.0]       # margin 5e-4: below 1e-3, exempt
    U[0, 1] = [4.998, 0.0, 5.0, 3.0, 1.0]         # margin 2e-3: checked
    out = O.propose(U, np.zeros((5, 2)), np.zeros((5, 2)), np.ones((1, 2)), np.array([0]))
    assert out["tokens"][0].tolist() == [1, 2]
    assert abs(out["margin"][0, 0] - 5e-4) < 1e-12
    assert abs(out["margin"][0, 1] - 2e-3) < 1e-12


# -------------------------------------------------------------------- overlap

def test_overlap_identity_and_bounds():
    rng = np.random.default_rng(10)
    P = rng.standard_normal((6, 7, 300)) * 2
    Q = P + rng.standard_normal((6, 7, 300)) * rng.uniform(0.1, 3, size=(6, 1, 1))
    out = O.overlap(P, Q, np.full(6, 7))
    assert np.allclose(out["a"], 1.0 - 0.5 * out["l1"], atol=1e-12)
    assert np.all((out["a"] > 0) & (out["a"] < 1))


def test_overlap_equal_and_disjoint():
    rng = np.random.default_rng(11)
    V = 64
    P = rng.standard_normal((2, 7, V))
    out = O.overlap(P, P.copy(), np.array([7, 7]))
    assert np.allclose(out["a"], 1.0, atol=1e-14)
    assert np.allclose(out["tau"], 8.0)
    Pd = np.full((1, 7, V), -1e4)
    Qd = np.full((1, 7, V), -1e4)
    Pd[0, :, : V // 2] = 0.0
    Qd[0, :, V // 2:] = 0.0
    out = O.overlap(Pd, Qd, np.array([7]))
    assert np.allclose(out["a"], 0.0, atol=1e-300)
    assert np.allclose(out["l1"], 2.0)
    assert out["tau"][0] == 1.0


def _two_point_logits(alphas):
    # p = (1, 0), q = (alpha, 1 - alpha)  =>  sum min(p, q) = alpha.
    G = len(alphas)
    P = np.zeros((1, G, 2))
    Q = np.zeros((1, G, 2))
    P[0, :, 1] = -1e9
    for i, al in enumerate(alphas):
        Q[0, i] = [math.log(al), math.log1p(-al)] if 0 < al < 1 else (
            [0.0, -1e9] if al == 1 else [-1e9, 0.0])
    return P, Q


@pytest.mark.parametrize("alpha", [1.0, 0.0, 0.5, 0.8, 0.37])
def test_tau_closed_forms(alpha):
    P, Q = _two_point_logits([alpha] * 7)
    out = O.overlap(P, Q, np.array([7]))
    assert np.allclose(out["a"], alpha, atol=1e-12)
    closed = 1.0 + sum(alpha ** k for k in range(1, 8))
    assert out["tau"][0] == pytest.approx(closed, rel=1e-12, abs=1e-12)
    if alpha == 1.0:
        assert out["tau"][0] == pytest.approx(8.0)
    if alpha == 0.0:
        assert out["tau"][0] == 1.0


def test_tau_first_position_zero_is_one():
    P, Q = _two_point_logits([0.0, 0.9, 0.9, 0.9, 0.9, 0.9, 0.9])
    assert O.overlap(P, Q, np.array([7]))["tau"][0] == pytest.approx(1.0)


def test_overlap_valid_len_aggregation_by_hand():
    al = [[0.9, 0.8, 0.7, 0.6, 0.5, 0.4, 0.3], [0.5, 0.5, 0.5, 0.2, 0.2, 0.2, 0.2],
          [0.1] * 7]
    P = np.concatenate([_two_point_logits(x)[0] for x in al])
    Q = np.concatenate([_two_point_logits(x)[1] for x in al])
    vl = np.array([7, 3, 0])
    out = O.overlap(P, Q, vl)
    assert np.allclose(out["a"][1], [0.5, 0.5, 0.5, 0, 0, 0, 0], atol=1e-12)
    assert np.allclose(out["a"][2], 0.0)
    tau0 = 1 + 0.9 + 0.72 + 0.504 + 0.3024 + 0.1512 + 0.06048 + 0.018144
    tau1 = 1 + 0.5 + 0.25 + 0.125
    assert out["tau"][:2] == pytest.approx([tau0, tau1], rel=1e-12)
    assert out["tau"][2] == 1.0
    assert out["mean_tau"] == pytest.approx((tau0 + tau1) / 2, rel=1e-12)
    assert out["accept_rate"] == pytest.approx([0.7, 0.65, 0.6, 0.6, 0.5, 0.4, 0.3], rel=1e-12)


# ---------------------------------------------------------------------------
# Teacher-forced loss forward ([READ] 4.1)
# ---------------------------------------------------------------------------

def test_loss_position_weights_match_the_page():
    g = _golden("loss_position_weights.json")
    w = O.position_weights(g["gamma"], g["decay"])
    assert abs(w.sum() - 1.0) < 1e-15
    assert abs(w[6] / w[0] - g["w6_page_rounded"]) < 5e-4
    raw = w / w[0]
    for j, v in enumerate(g["w_first_four_page_rounded"]):
        assert abs(raw[j] - v) < 5e-3


def test_bce_with_logits_special_values():
    assert abs(O.bce_with_logits(0.0, 0.5) - np.log(2.0)) < 1e-15
    assert abs(O.bce_with_logits(0.0, 1.0) - np.log(2.0)) < 1e-15
    # y = 1: -log sigma(z); y = 0: -log(1 - sigma(z)); symmetric in (z, y) -> (-z, 1 - y)
    for z in (-30.0, -2.5, 0.3, 4.0, 30.0):
        sig = 1.0 / (1.0 + np.exp(-z))
        assert abs(O.bce_with_logits(z, 1.0) + np.log(sig)) < 1e-12 * max(1.0, abs(z))
        assert abs(O.bce_with_logits(z, 0.25) - O.bce_with_logits(-z, 0.75)) < 1e-12
    # minimum over y is at y = sigma(z) (the entropy of sigma(z))
    z = 1.3
    sig = 1.0 / (1.0 + np.exp(-z))
    ent = -(sig * np.log(sig) + (1 - sig) * np.log(1 - sig))
    assert abs(O.bce_with_logits(z, sig) - ent) < 1e-12


def _loss_inputs(B=3, G=4, V=24, r=6, seed=5, scale=1.0):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2.0, (B, G, V))
    E = rng.normal(0, scale, (V, r))
    W = rng.normal(0, scale, (V, r))
    prev = rng.integers(0, V, (B, G))
    P = U + rng.normal(0, 0.7, (B, G, V))
    tgt = rng.integers(0, V, (B, G))
    z = rng.normal(0, 1.5, (B, G))
    return U, E, W, prev, P, tgt, z


def test_loss_equal_distributions():
    # P equals the draft logits up to a per-row constant: p = q, so
    # l1 = 0, a = 1, and the confidence loss is -log sigma(z)
    U, E, W, prev, _, tgt, z = _loss_inputs()
    B, G, V = U.shape
    P = np.empty_like(U)
    for b in range(B):
        for j in range(G):
            P[b, j] = U[b, j] + O.markov_bias(E, W, int(prev[b, j])) + 3.0 * b - j
    out = O.loss_forward(U, E, W, prev, P, tgt, z)
    assert np.max(out["l1"]) < 1e-12
    assert np.all(np.abs(out["accept"] - 1.0) < 1e-12)
    assert abs(out["conf_loss"] - np.mean(np.logaddexp(0.0, -z))) < 1e-12
    assert abs(out["l1_loss"]) < 1e-12


def test_loss_uniform_draft_cross_entropy_is_log_v():
    U, E, W, prev, P, tgt, z = _loss_inputs()
    U0 = np.zeros_like(U)
    E0 = np.zeros_like(E)
    out = O.loss_forward(U0, E0, W, prev, P, tgt, z)
    assert np.all(np.abs(out["ce"] - np.log(U.shape[2])) < 1e-12)


def test_loss_disjoint_supports_have_zero_accept():
    B, G, V = 2, 3, 8
    U = np.full((B, G, V), -200.0)
    P = np.full((B, G, V), -200.0)
    U[..., 0] = 0.0
    P[..., 5] = 0.0
    E = np.zeros((V, 4))
    W = np.zeros((V, 4))
    out = O.loss_forward(U, E, W, np.zeros((B, G), int), P, np.zeros((B, G), int),
                         np.zeros((B, G)))
    assert np.all(np.abs(out["l1"] - 2.0) < 1e-12)
    assert np.all(out["accept"] == 0.0)


def test_loss_total_is_the_weighted_combination():
    U, E, W, prev, P, tgt, z = _loss_inputs(seed=9)
    base = O.loss_forward(U, E, W, prev, P, tgt, z)
    only_ce = O.loss_forward(U, E, W, prev, P, tgt, z, ce_alpha=1.0, l1_alpha=0.0, conf_alpha=0.0)
    only_l1 = O.loss_forward(U, E, W, prev, P, tgt, z, ce_alpha=0.0, l1_alpha=1.0, conf_alpha=0.0)
    only_cf = O.loss_forward(U, E, W, prev, P, tgt, z, ce_alpha=0.0, l1_alpha=0.0, conf_alpha=1.0)
    assert abs(only_ce["loss"] - base["ce_loss"]) < 1e-15
    assert abs(only_l1["loss"] - base["l1_loss"]) < 1e-15
    assert abs(only_cf["loss"] - base["conf_loss"]) < 1e-15
    assert abs(base["loss"] - (0.1 * base["ce_loss"] + 0.9 * base["l1_loss"] + base["conf_loss"])) < 1e-12


def test_loss_matches_torch_functional_on_cpu():
    # An independent implementation of the same definitions with PyTorch's CPU
    # softmax / cross_entropy / binary_cross_entropy_with_logits in float64.
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    U, E, W, prev, P, tgt, z = _loss_inputs(B=4, G=5, V=40, r=8, seed=13, scale=0.6)
    for baf in (True, False):
        out = O.loss_forward(U, E, W, prev, P, tgt, z, bias_at_first=baf)
        Ut = torch.tensor(U, dtype=torch.float64)
        emb = torch.tensor(E, dtype=torch.float64)[torch.tensor(prev)]           # [B, G, r]
        bias = emb @ torch.tensor(W, dtype=torch.float64).T                      # [B, G, V]
        if not baf:
            bias[:, 0] = 0.0
        dl = Ut + bias
        p = F.softmax(torch.tensor(P, dtype=torch.float64), dim=-1)
        q = F.softmax(dl, dim=-1)
        l1 = (p - q).abs().sum(-1)
        acc = (1.0 - 0.5 * l1).clamp(0.0, 1.0)
        ce = F.cross_entropy(dl.transpose(1, 2), torch.tensor(tgt), reduction="none")
        G = U.shape[1]
        w = torch.exp(-torch.arange(G, dtype=torch.float64) / 4.0)
        w = w / w.sum()
        wce = (ce.mean(0) * w).sum()
        wl1 = (l1.mean(0) * w).sum()
        cl = F.binary_cross_entropy_with_logits(torch.tensor(z, dtype=torch.float64), acc)
        assert np.max(np.abs(out["l1"] - l1.numpy())) < 1e-12
        assert np.max(np.abs(out["ce"] - ce.numpy())) < 1e-10
        assert abs(out["ce_loss"] - float(wce)) < 1e-10
        assert abs(out["l1_loss"] - float(wl1)) < 1e-12
        assert abs(out["conf_loss"] - float(cl)) < 1e-12
        assert abs(out["loss"] - float(0.1 * wce + 0.9 * wl1 + cl)) < 1e-10


# ---------------------------------------------------------------------------
# Confidence side ([TRAIN] confidence head; [WALK] 4.3; [READ] 3.1, 5)
# ---------------------------------------------------------------------------

def test_threshold_keep_by_hand():
    c = np.array([[0.9, 0.8, 0.4, 0.9],
                  [0.3, 0.9, 0.9, 0.9],
                  [0.7, 0.7, 0.7, 0.7],
                  [0.7, np.nan, 0.9, 0.9]])
    assert list(O.threshold_keep(c, 0.5)) == [2, 0, 4, 1]
    assert list(O.threshold_keep(c[:3], 0.0)) == [4, 4, 4]      # 0 keeps everything
    assert list(O.threshold_keep(c[:3], 1.01)) == [0, 0, 0]
    assert list(O.threshold_keep(c, 0.7)) == [2, 0, 4, 1]        # >= keeps a tie


def test_confidence_head_by_hand():
    # H = 2, rank 2, V = 3.  w_c = (1, -1 | 2, 0.5), b_c = -0.5
    E = np.array([[1.0, 0.0], [0.0, 2.0], [-1.0, 1.0]])
    h = np.array([[[0.5, 0.25], [1.0, 1.0], [0.0, 3.0]]])      # R = 1, gamma = 3
    w = np.array([1.0, -1.0, 2.0, 0.5])
    out = O.confidence_head(h, E, w, -0.5, prev_tok=[2], tokens=np.array([[1, 0, 2]]))
    # j = 0 uses E[prev_tok] = E[2]; j = 1 uses E[tokens[0]] = E[1]; j = 2 uses E[0]
    s = [0.25 + (-2.0 + 0.5) - 0.5, 0.0 + (0.0 + 1.0) - 0.5, -3.0 + 2.0 - 0.5]
    assert np.allclose(out["logit"][0], s, atol=1e-15)
    c = [1.0 / (1.0 + np.exp(-v)) for v in s]
    assert np.allclose(out["conf"][0], c, rtol=1e-14)
    assert np.allclose(out["survival"][0], np.cumprod(c), rtol=1e-14)
    assert O.sigmoid(0.0) == 0.5 and O.sigmoid(800.0) == 1.0 and O.sigmoid(-800.0) == 0.0


def _page_cumprod_batch(G=6):
    # 5^G requests whose accepted prefix length L satisfies P(L >= k) = 0.8^k exactly
    L = []
    for k in range(G + 1):
        ge = 5 ** (G - k) * 4 ** k
        gt = 5 ** (G - k - 1) * 4 ** (k + 1) if k < G else 0
        L += [k] * (ge - gt)
    return np.array(L)


def test_calibration_reproduces_the_page_example():
    g = _golden("calibration_cumprod_example.json")
    G = g["gamma"]
    L = _page_cumprod_batch(G)
    c = np.full((len(L), G), g["predicted_step"])
    out = O.calibration(c, L, n_bins=10)
    assert abs(out["pos_pred"][G - 1] - g["predicted_survival_pos6_page_rounded"]) < 5e-4
    assert abs(out["pos_real"][G - 1] - g["true_survival_pos6_page_rounded"]) < 5e-4
    ratio = out["pos_pred"][G - 1] / out["pos_real"][G - 1]
    assert round(100 * (ratio - 1)) == g["overestimate_page_percent"]
    # the empirical step acceptance is exactly the true step probability
    assert np.allclose(out["pos_real"], g["true_step"] ** np.arange(1, G + 1), rtol=1e-12)
    # abs error over tested positions: 0.8 * |0.85 - 1| + 0.2 * |0.85 - 0| = 0.29
    assert abs(out["abs_error"] - 0.29) < 1e-12
    # each position's survival falls in its own bin, so ECE = the mean bias
    assert abs(out["ece"] - out["cumprod_bias"]) < 1e-12
    bias = np.mean(0.85 ** np.arange(1, G + 1) - 0.8 ** np.arange(1, G + 1))
    assert abs(out["cumprod_bias"] - bias) < 1e-12


def test_calibration_perfect_and_edges():
    # gamma = 1, c = 0.5, half of the requests accepted: perfectly calibrated
    out = O.calibration(np.full((4, 1), 0.5), [1, 1, 0, 0], n_bins=4)
    assert out["ece"] == 0.0 and out["cumprod_bias"] == 0.0 and out["abs_error"] == 0.5
    assert list(out["count"]) == [0, 0, 4, 0] and out["n_tested"] == 4
    # survival 1 goes to the last bin, 0 to the first; untested positions
    # (after the first rejection) do not count toward the step error
    out = O.calibration(np.array([[1.0, 0.0, 1.0]]), [1], n_bins=5)
    assert list(out["count"]) == [2, 0, 0, 0, 1]
    assert out["n_tested"] == 2 and out["abs_error"] == 0.0
    assert abs(out["ece"] - 0.0) < 1e-15


# ---------------------------------------------------------------------------
# Gated Markov head ([READ] 2.3 GatedMarkovHead: g = sigmoid(W_g [h; m]),
# b = W_up (g * m))
# ---------------------------------------------------------------------------

def test_gated_head_by_hand():
    # rank 2, H = 1, V = 3; previous token 1 with E[1] = (1, -2), h = (3)
    E = np.array([[0.0, 0.0], [1.0, -2.0], [5.0, 5.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 1.0]])         # [V, rank]
    W_g = np.array([[1.0, 0.0, 0.0],                           # z_0 = h = 3
                    [0.0, 0.0, 1.0]])                          # z_1 = m_1 = -2
    gm = O.gated_rep(E, W_g, np.array([3.0]), 1)
    s3, sm2 = 1.0 / (1.0 + np.exp(-3.0)), 1.0 / (1.0 + np.exp(2.0))
    assert np.allclose(gm, [s3 * 1.0, sm2 * -2.0], rtol=1e-14)
    b = O.head_bias(E, W, 1, gate=dict(h=np.array([[[3.0]]]), W_g=W_g), r=0, j=0)
    assert np.allclose(b, [s3, -2.0 * sm2, 2.0 * s3 - 2.0 * sm2], rtol=1e-14)


def test_gated_head_limits():
    rng = np.random.default_rng(3)
    V, r, H = 40, 8, 5
    E = rng.normal(0, 1, (V, r))
    W = rng.normal(0, 1, (V, r))
    h = rng.normal(0, 1, (1, 1, H))
    zero = dict(h=h, W_g=np.zeros((r, H + r)))
    # a zero gate matrix opens every gate half way: half the vanilla bias
    assert np.allclose(O.head_bias(E, W, 7, gate=zero), 0.5 * O.markov_bias(E, W, 7), rtol=1e-13)
    # a constant hidden unit with a large weight saturates the gates
    hc = np.ones((1, 1, H))
    Wg = np.zeros((r, H + r))
    Wg[:, 0] = 60.0
    assert np.allclose(O.head_bias(E, W, 7, gate=dict(h=hc, W_g=Wg)),
                       O.markov_bias(E, W, 7), rtol=1e-12, atol=1e-12)
    Wg[:, 0] = -60.0
    assert np.max(np.abs(O.head_bias(E, W, 7, gate=dict(h=hc, W_g=Wg)))) < 1e-20


def test_gated_propose_single_step_by_hand():
    # gamma = 1: x = argmax(U_0 + W (g * m)) with m = E[prev]
    E = np.array([[0.0, 0.0], [1.0, -2.0], [5.0, 5.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 1.0]])
    W_g = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 1.0]])
    h = np.array([[[3.0]]])
    U = np.array([[[0.5, 0.0, 0.0]]])
    out = O.propose(U, E, W, np.array([[0.9]]), [1], gate=dict(h=h, W_g=W_g))
    s3, sm2 = 1.0 / (1.0 + np.exp(-3.0)), 1.0 / (1.0 + np.exp(2.0))
    ell = [0.5 + s3, -2.0 * sm2, 2.0 * s3 - 2.0 * sm2]   # 1.4526, -0.2384, 1.6670
    assert int(out["tokens"][0, 0]) == int(np.argmax(ell)) == 2
    assert abs(out["logit_at_tok"][0, 0] - ell[2]) < 1e-14


# ---------------------------------------------------------------------------
# RNN head ([NOTES] 2.3, RNN 头; [READ] 2.3 RNNHead): u = [s; m; h],
# g = sigmoid(W_g u), c = tanh(W_c u), s' = g s + (1 - g) c,
# o = tanh(W_o [s'; m; h]), b = W o, s = 0 at the start of the block
# ---------------------------------------------------------------------------

def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_rnn_step_by_hand():
    # rank 1, H = 1: the gate reads the Markov row, the candidate the hidden
    # state, the output the new state
    E = np.array([[0.5], [-1.0]])
    W_rnn = np.array([[[0.0, 2.0, 0.0]],      # W_g: z = 2 m
                      [[0.0, 0.0, 1.0]],      # W_c: c = tanh(h)
                      [[1.0, 0.0, 0.0]]])     # W_o: o = tanh(s')
    s1, o1 = O.rnn_step(E, W_rnn, np.array([1.0]), np.zeros(1), 0)
    g1 = _sig(1.0)                           # z = 2 * 0.5
    assert abs(s1[0] - (1.0 - g1) * math.tanh(1.0)) < 1e-15
    assert abs(o1[0] - math.tanh((1.0 - g1) * math.tanh(1.0))) < 1e-15
    # second step: previous token 1 (m = -1), h = 0, so c = 0 and the state
    # only decays by its gate sigmoid(-2)
    s2, o2 = O.rnn_step(E, W_rnn, np.array([0.0]), s1, 1)
    assert abs(s2[0] - _sig(-2.0) * s1[0]) < 1e-15
    assert abs(o2[0] - math.tanh(_sig(-2.0) * s1[0])) < 1e-15
    # the same two steps through rnn_reps (state from zero, tokens chained)
    reps = O.rnn_reps(E, W_rnn, np.array([[[1.0], [0.0]]]), [0], np.array([[1, 0]]))
    assert np.allclose(reps[0, :, 0], [o1[0], o2[0]], rtol=0, atol=1e-15)


def test_rnn_head_without_candidate_is_the_markov_head_on_tanh_rows():
    # W_c = 0 keeps the state at zero; W_o = [0, I, 0] outputs tanh(m), so the
    # head's bias is W tanh(E[prev]): the plain Markov head on the table tanh(E)
    rng = np.random.default_rng(21)
    R, G, V, r, H = 3, 4, 60, 5, 7
    E = rng.normal(0, 1, (V, r))
    W = rng.normal(0, 1, (V, r))
    U = rng.normal(0, 2, (R, G, V))
    W_rnn = np.zeros((3, r, 2 * r + H))
    W_rnn[0] = rng.normal(0, 1, (r, 2 * r + H))     # any gate
    W_rnn[2][:, r:2 * r] = np.eye(r)
    h = rng.normal(0, 1, (R, G, H))
    conf = np.full((R, G), 0.8)
    prev = rng.integers(0, V, R)
    for T in (0.0, 1.0):
        a = O.propose(U, E, W, conf, prev, None, T, 5, rnn=dict(h=h, W_rnn=W_rnn))
        b = O.propose(U, np.tanh(E), W, conf, prev, None, T, 5)
        assert np.array_equal(a["tokens"], b["tokens"])
        assert np.allclose(a["lse_q"], b["lse_q"], rtol=0, atol=1e-12)
        assert np.allclose(a["logit_at_tok"], b["logit_at_tok"], rtol=0, atol=1e-12)


def test_rnn_state_is_a_geometric_filter_of_the_history():
    # W_g = 0 (every gate 1/2), c = tanh(m), o = tanh(s):
    #   s_j = sum_{i <= j} 2^-(j - i + 1) tanh(m_i)
    rng = np.random.default_rng(22)
    V, r, H, G = 30, 3, 2, 6
    E = rng.normal(0, 1, (V, r))
    W_rnn = np.zeros((3, r, 2 * r + H))
    W_rnn[1][:, r:2 * r] = np.eye(r)
    W_rnn[2][:, :r] = np.eye(r)
    tokens = rng.integers(0, V, (1, G))
    prev = [int(rng.integers(0, V))]
    reps = O.rnn_reps(E, W_rnn, rng.normal(0, 1, (1, G, H)), prev, tokens)
    chain = [prev[0]] + list(tokens[0, :-1])
    for j in range(G):
        s = sum(0.5 ** (j - i + 1) * np.tanh(E[chain[i]]) for i in range(j + 1))
        assert np.allclose(reps[0, j], np.tanh(s), rtol=0, atol=1e-14)
    # without a bias at the first position, position 0 has no output and the
    # recursion starts at position 1 from a zero state
    reps0 = O.rnn_reps(E, W_rnn, np.zeros((1, G, H)), prev, tokens, bias_at_first=False)
    assert np.all(reps0[0, 0] == 0.0)
    for j in range(1, G):
        s = sum(0.5 ** (j - i + 1) * np.tanh(E[chain[i]]) for i in range(1, j + 1))
        assert np.allclose(reps0[0, j], np.tanh(s), rtol=0, atol=1e-14)


def test_rnn_verify_replays_the_drafted_states():
    # the verifier's q at a position equals the proposal's, which needs the
    # RNN state rebuilt from the drafted prefix: a keep-all verification of
    # the drafted tokens against P = the draft logits accepts everything
    rng = np.random.default_rng(23)
    R, G, V, r, H = 2, 4, 25, 3, 4
    E = rng.normal(0, 1, (V, r))
    W = rng.normal(0, 1, (V, r))
    U = rng.normal(0, 1, (R, G, V))
    rnn = dict(h=rng.normal(0, 1, (R, G, H)), W_rnn=rng.normal(0, 0.7, (3, r, 2 * r + H)))
    prev = rng.integers(0, V, R)
    out = O.propose(U, E, W, np.full((R, G), 0.9), prev, None, 1.0, 9, rnn=rnn)
    P = np.zeros((R, G + 1, V))
    for q in range(R):
        for t in range(G):
            P[q, t] = U[q, t] + W @ out["rep"][q, t]
    ver = O.verify(P, U, E, W, prev, out["tokens"], np.full(R, G), None, 1.0, 9, rnn=rnn)
    assert list(ver["accept_len"]) == [G] * R


# ---------------------------------------------------------------------------
# Markov top-16 candidate set ([TRAIN] Prefix reranker, 候选与前缀表示)
# ---------------------------------------------------------------------------

def test_top_k_by_hand():
    idx, val = O.top_k([0.5, 3.0, -1.0, 3.0, 2.0, 0.5], 4)
    assert list(idx) == [1, 3, 4, 0] and list(val) == [3.0, 3.0, 2.0, 0.5]   # ties: lower index
    idx, _ = O.top_k([1.0, 2.0], 5)                                          # K > V: everything
    assert list(idx) == [1, 0]


def test_candidates_without_markov_table_are_the_sorted_base_logits():
    rng = np.random.default_rng(11)
    R, G, V, r = 2, 3, 50, 4
    U = rng.normal(0, 1, (R, G, V))
    out = O.propose(U, np.zeros((V, r)), rng.normal(0, 1, (V, r)), np.full((R, G), 0.9),
                    [3, 7], candidates=16)
    for q in range(R):
        for j in range(G):
            ref = np.argsort(-U[q, j], kind="stable")[:16]
            assert list(out["cand_tok"][q, j]) == list(ref)
            assert np.array_equal(out["cand_logit"][q, j], U[q, j][ref])
            assert out["cand_tok"][q, j, 0] == out["tokens"][q, j]     # greedy = top-1


def test_candidates_follow_the_drafted_chain():
    # each position's set is the top of U_j + W E[x_{j-1}] with x the drafted token
    rng = np.random.default_rng(12)
    R, G, V, r = 1, 4, 60, 6
    U = rng.normal(0, 1, (R, G, V))
    E = rng.normal(0, 1, (V, r))
    W = rng.normal(0, 1, (V, r))
    out = O.propose(U, E, W, np.full((R, G), 0.9), [5], candidates=16)
    prev = 5
    for j in range(G):
        ell = U[0, j] + (E @ W.T)[prev]          # the dense V x V transition row
        ref = np.argsort(-ell, kind="stable")[:16]
        assert list(out["cand_tok"][0, j]) == list(ref)
        assert np.allclose(out["cand_logit"][0, j], ell[ref], atol=1e-12)
        prev = int(out["tokens"][0, j])
        assert prev == ref[0]


# ---------------------------------------------------------------------- AUROC

def _auroc_brute(score, label):
    pos = score[label]
    neg = score[~label]
    if pos.size == 0 or neg.size == 0:
        return 0.5
    gt = (pos[:, None] > neg[None, :]).sum()
    eq = (pos[:, None] == neg[None, :]).sum()
    return (gt + 0.5 * eq) / (pos.size * neg.size)


def test_auroc_against_brute_force_pairs():
    # every positive/negative pair counted by brute force (ties one half)
    rng = np.random.default_rng(21)
    for trial in range(20):
        M, G = int(rng.integers(1, 12)), int(rng.integers(1, 8))
        # few distinct confidence values so that ties occur
        conf = rng.choice([0.5, 0.8, 0.9, 1.0], size=(M, G)) if trial % 2 else rng.uniform(0, 1, (M, G))
        L = rng.integers(0, G + 1, size=M)
        a = np.cumprod(np.clip(conf, 0, 1), axis=1).reshape(-1)
        y = (np.arange(G)[None, :] < L[:, None]).reshape(-1)
        assert abs(O.auroc(conf, L) - _auroc_brute(a, y)) <= 1e-12


def test_auroc_closed_cases():
    G = 4
    conf = np.tile(np.array([0.9, 0.9, 0.9, 0.9]), (6, 1))
    # perfect ranking: survival falls along the block, acceptance ends at 2 for all
    assert O.auroc(conf, np.full(6, 2)) == 1.0
    # every score tied: one half
    assert O.auroc(np.ones((5, G)), np.array([0, 1, 2, 3, 4])) == 0.5
    # only positives or only negatives: one half by convention
    assert O.auroc(conf, np.full(6, G)) == 0.5
    assert O.auroc(conf, np.zeros(6, dtype=int)) == 0.5
    # reversed ranking is 0: the high-survival position is the negative one
    conf2 = np.array([[1.0, 1.0], [0.2, 1.0]])
    # scores a = [1, 1, .2, .2]; labels: request 0 accepts nothing, request 1 all
    assert O.auroc(conf2, np.array([0, 2])) == 0.0


def test_auroc_matches_a_library_implementation():
    metrics = pytest.importorskip("sklearn.metrics")
    rng = np.random.default_rng(22)
    conf = rng.beta(6, 2, size=(300, 7))
    L = rng.integers(0, 8, size=300)
    a = np.cumprod(conf, axis=1).reshape(-1)
    y = (np.arange(7)[None, :] < L[:, None]).reshape(-1)
    assert abs(O.auroc(conf, L) - metrics.roc_auc_score(y, a)) <= 1e-12
