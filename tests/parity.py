"""Element-by-element comparison of the CUDA path with the fp64 oracle.

Agreement rules:
  * token ids, accept lengths, next tokens and scheduler allocations are
    bit-exact, except where the oracle's decision variable has a top-2 margin
    below 1e-3 (draft tokens, greedy accept tests, correction / bonus draws)
    or an accept test whose uniform lies within 1e-6 of min(1, p/q); once a
    request's draft token is exempt, its later positions and its verification
    are exempt too (their inputs differ).  Exemptions are counted.
  * probabilities (q of the chosen token, overlaps) and tau_prob within 1e-4
    absolute; log-normalisers and logits within 1e-4 absolute.
"""

from __future__ import annotations

import numpy as np

MARGIN = 1e-3
ACCEPT_TIE = 1e-6
PROB_TOL = 1e-4
LOGIT_TOL = 1e-4


class Report:
    def __init__(self):
        self.checked = 0
        self.exempt = 0
        self.notes = []

    def __repr__(self):
        return f"checked={self.checked} exempt={self.exempt}"


def draft_exempt(margin: np.ndarray) -> np.ndarray:
    """[R, G] bool: position j of request r is exempt if any position <= j
    had a near-tie."""
    return np.minimum.accumulate(margin, axis=1) < MARGIN


def compare_propose(k, o, rep: Report | None = None, rows=None):
    """k: kernel outputs (numpy) for the rows `rows` (default all);
    o: oracle propose dict for the same rows, in the same order."""
    rep = rep or Report()
    tok_k = np.asarray(k["tokens"])
    ex = draft_exempt(o["margin"])
    R, G = tok_k.shape
    for r in range(R):
        for j in range(G):
            if ex[r, j]:
                rep.exempt += 1
                continue
            rep.checked += 1
            assert tok_k[r, j] == o["tokens"][r, j], f"token r={r} j={j}: {tok_k[r, j]} vs {o['tokens'][r, j]}"
            lk, lo = float(k["lse_q"][r, j]), float(o["lse_q"][r, j])
            assert abs(lk - lo) <= LOGIT_TOL, f"lse r={r} j={j}: {lk} vs {lo}"
            gk, go = float(k["logit_at_tok"][r, j]), float(o["logit_at_tok"][r, j])
            assert abs(gk - go) <= LOGIT_TOL, f"logit r={r} j={j}: {gk} vs {go}"
            qk, qo = np.exp(gk - lk), np.exp(go - lo)
            assert abs(qk - qo) <= PROB_TOL, f"q r={r} j={j}: {qk} vs {qo}"
    sk = np.asarray(k["survival"], dtype=np.float64)
    so = o["survival"].astype(np.float32).astype(np.float64)
    assert np.array_equal(sk, so), "survival differs from the fp64 product rounded to fp32"
    return rep


def compare_schedule(k_keep, k_theta, o, rep: Report | None = None):
    rep = rep or Report()
    if o["theta_gap"] < 1e-9:
        rep.exempt += 1
        rep.notes.append("scheduler near-tie")
        return rep
    rep.checked += 1
    assert np.array_equal(np.asarray(k_keep), o["keep_len"]), "keep_len differs"
    if k_theta is not None:
        assert abs(float(k_theta[0]) - o["theta"]) <= 1e-6 * abs(o["theta"]) + 1e-3
        assert int(round(float(k_theta[1]))) == o["B"]
    return rep


def compare_verify(k_acc, k_next, o, temperature, keep_len, draft_ex=None,
                   rep: Report | None = None):
    """draft_ex: [R] bool, requests whose kept draft prefix was exempt."""
    rep = rep or Report()
    R = len(k_acc)
    for r in range(R):
        if draft_ex is not None and draft_ex[r]:
            rep.exempt += 1
            continue
        tie = o["accept_gap"][r] < (MARGIN if temperature == 0.0 else ACCEPT_TIE)
        if tie:
            rep.exempt += 1
            continue
        rep.checked += 1
        assert int(k_acc[r]) == int(o["accept_len"][r]), \
            f"accept_len r={r}: {k_acc[r]} vs {o['accept_len'][r]} (keep {keep_len[r]})"
        if o["next_margin"][r] < MARGIN:
            rep.exempt += 1
            continue
        assert int(k_next[r]) == int(o["next_token"][r]), \
            f"next_token r={r}: {k_next[r]} vs {o['next_token'][r]}"
    return rep


def compare_overlap(k, o, rep: Report | None = None):
    rep = rep or Report()
    a_k, a_o = np.asarray(k["a"]), o["a"]
    assert np.max(np.abs(a_k - a_o)) <= PROB_TOL, f"a max err {np.max(np.abs(a_k - a_o))}"
    l1_k = np.asarray(k["l1"])
    assert np.max(np.abs(l1_k - o["l1"])) <= 2 * PROB_TOL
    assert np.max(np.abs(np.asarray(k["tau"]) - o["tau"])) <= PROB_TOL
    assert np.max(np.abs(np.asarray(k["accept_rate"]) - o["accept_rate"])) <= PROB_TOL
    assert abs(float(np.asarray(k["mean_tau"]).reshape(-1)[0]) - o["mean_tau"]) <= PROB_TOL
    # the identity sum min(p,q) = 1 - |p-q|_1 / 2 on the GPU outputs themselves
    assert np.max(np.abs(a_k - (1.0 - 0.5 * l1_k) * (a_k != 0))) <= 2 * PROB_TOL
    rep.checked += a_k.size
    return rep
