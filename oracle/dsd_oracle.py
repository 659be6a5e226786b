"""Plain fp64 CPU oracle for the DSpark draft/verify hot path.

TEST INFRASTRUCTURE ONLY.  This module is imported by the test-suite, by
``__graft_entry__.smoke()`` and by ``bench.py``'s CPU-baseline / reference leg.
The product path (the CUDA library under ``semi_autoregressive_draft_gb300``
and its binding) never imports, calls or links it, and there is no CPU
fallback anywhere in the product.

Everything here is written for a reader checking it against the pages by eye:
numpy in float64, loops over requests and positions, one library primitive per
step at most (a matrix-vector product, a sort).  Sources, by page title and
section:

  [TRAIN]  "Qwen3.8-Flash-Next DSpark 训练实验"
           -- 评估口径 / 离线指标 (overlap a_i, tau_prob, accept_rate@i)
           -- Baseline 架构 / Markov 顺序修正 (m_i, b_i, l_i = l_i^0 + b_i, greedy)
  [NOTES]  "DSpark notes" (h.sjds.net/a/571373)
           -- 2.2 Sequential Stage; 2.3 串行头的两种形态 (Markov head = low-rank
              factorisation of a V x V transition matrix)
  [READ]   "DSpark 论文精读：置信度调度推测解码、半自回归生成与大模型推理加速"
           -- 2.2 (biased logits, sampling), 2.3 (VanillaMarkov), 3.1 (prefix
              survival, overlap identity), 3.2 (hardware-aware prefix scheduler)
  [WALK]   "DeepSpec 训练全流程详解（以 Qwen3 + DSpark 为例）"
           -- 4.3 Propose, 4.4 Verify (rejection test, residual, bonus token)
           -- 3.4 (loss: CE, L1 alignment, confidence BCE, their weights)
  ([READ] 4.1 also gives the loss forward: position-decayed CE + L1 and the
  confidence BCE against the soft accept-rate label.)

Readings where the pages are silent or disagree (each one is listed with its
reason in the repository's design notes):
  * position 0 is biased by the Markov head using ``prev_tok`` ([TRAIN], m_1 =
    W_1[D]); ``bias_at_first=False`` gives the [READ] 2.3 behaviour instead;
  * no activation between the two Markov tables ([TRAIN]); ``act="silu"`` gives
    the [READ] 2.3 variant;
  * argmax ties go to the lowest token index;
  * temperature T divides the logits of both draft and target; T = 0 is greedy
    (argmax) for draft, accept test, correction and bonus;
  * random numbers: Philox4x32-10 (Salmon et al., SC'11) keyed by the 64-bit
    seed, counter (element group, position, request id, stream); streams
    0 draft Gumbel, 1 accept uniform, 2 residual Gumbel, 3 bonus Gumbel;
    u = ((w >> 9) + 0.5) * 2^-23, exactly representable in fp32 and in (0,1);
  * accept iff u < min(1, p/q) (strict);
  * an empty residual (sum <= 1e-12 * sum p) falls back to sampling p;
  * scheduler sort key (a desc, r asc, j asc); Theta must strictly improve;
    SPS table is 1-based (sps[B-1] = SPS(B)); B beyond the table is infeasible;
  * conf is clamped to [0, 1], and so is the scheduler's survival input;
  * RNN head: the output activation, unnamed on the page, is tanh; a
    position without a bias leaves the state at zero;
  * loss: every position of every row is valid (no loss mask), so [WALK]
    3.4's masked sum over all tokens divided by the total weight equals
    [READ] 4.1's per-position batch mean weighted by normalised w_j; the
    confidence label 1 - L1/2 is clamped to [0, 1] against rounding;
  * overlap: a_i is reported as sum(min(p,q)) unclamped; positions i >=
    valid_len have a_i = 0; a block is valid when valid_len >= 1.

Parity pins (what checks this oracle against something other than itself)
live in tests/test_oracle_pins.py; nothing in this file is "parity unpinned".
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Philox4x32-10, from its published definition (Salmon, Moraes, Dror, Shaw,
# "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): a 4-word counter is
# scrambled by 10 rounds; each round multiplies words 0 and 2 by fixed odd
# constants, swaps the high/low halves across the words and xors in the key;
# the 2-word key advances by a Weyl sequence between rounds.
# ---------------------------------------------------------------------------

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

STREAM_DRAFT = 0
STREAM_ACCEPT = 1
STREAM_RESIDUAL = 2
STREAM_BONUS = 3


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds.  Arguments are integers or integer arrays
    holding 32-bit values; returns the four output words as uint64 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for _ in range(10):
        p0 = m0 * c[0]                  # 32 x 32 -> 64 bits, exact in uint64
        p1 = m1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = np.uint64((int(k0) + PHILOX_W0) & 0xFFFFFFFF)
        k1 = np.uint64((int(k1) + PHILOX_W1) & 0xFFFFFFFF)
    return tuple(x & _MASK32 for x in c)


def seed_key(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniform_from_word(w):
    """u = ((w >> 9) + 0.5) * 2^-23, in (0, 1)."""
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def vocab_uniforms(seed: int, position: int, req: int, stream: int, V: int):
    """One uniform per vocabulary entry v: word (v mod 4) of
    Philox(counter = (v div 4, position, req, stream), key = seed)."""
    v = np.arange(V, dtype=np.uint64)
    k0, k1 = seed_key(seed)
    words = philox4x32_10(v >> np.uint64(2), position, req, stream, k0, k1)
    w = np.choose((v & np.uint64(3)).astype(np.int64), words)
    return uniform_from_word(w)


def vocab_gumbel(seed: int, position: int, req: int, stream: int, V: int):
    """Standard Gumbel noise g_v = -ln(-ln u_v)."""
    u = vocab_uniforms(seed, position, req, stream, V)
    return -np.log(-np.log(u))


def accept_uniform(seed: int, position: int, req: int) -> float:
    """The uniform of the accept test at one position ([WALK] 4.4: random())."""
    k0, k1 = seed_key(seed)
    w = philox4x32_10(0, position, req, STREAM_ACCEPT, k0, k1)[0]
    return float(uniform_from_word(w))


# ---------------------------------------------------------------------------
# Small numerical helpers, written out.
# ---------------------------------------------------------------------------

def logsumexp(x):
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)
    return float(m + np.log(np.sum(np.exp(x - m))))


def softmax(x):
    x = np.asarray(x, dtype=np.float64)
    return np.exp(x - logsumexp(x))


def top2_margin(z):
    """Gap between the largest and the second-largest entry (inf if V == 1)."""
    z = np.asarray(z, dtype=np.float64)
    if z.size < 2:
        return float("inf")
    i = int(np.argmax(z))
    rest = np.delete(z, i)
    return float(z[i] - np.max(rest))


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# a1: prefix survival  ([READ] 3.1: a_{r,j} = prod_{i<=j} c_{r,i})
# ---------------------------------------------------------------------------

def survival(conf):
    """a[r, j] = prod_{i <= j} clamp(c[r, i], 0, 1), in fp64.

    ``conf`` is [R, gamma].  Non-finite confidences are an error."""
    c = _f64(conf)
    if not np.all(np.isfinite(c)):
        raise ValueError("non-finite confidence")
    c = np.clip(c, 0.0, 1.0)
    R, G = c.shape
    a = np.empty((R, G), dtype=np.float64)
    for r in range(R):
        acc = 1.0
        for j in range(G):
            acc = acc * c[r, j]
            a[r, j] = acc
    return a


# ---------------------------------------------------------------------------
# a2/a3: Markov bias  ([TRAIN] Markov 顺序修正: m_i = W_1[t_{i-1}], b_i = W_2 m_i;
# [NOTES] 2.3: one table lookup plus one low-rank projection)
#
# Storage: E is the down table [V, r] (row t is the embedding of token t);
# W is the up projection stored [V, r] (row v is the weight vector producing
# logit bias v), i.e. b[v] = sum_k W[v, k] * m[k].
# ---------------------------------------------------------------------------

def markov_rep(E, prev: int, act: str = "none"):
    """m = act(E[prev]): the Markov representation of the previous token."""
    m = _f64(E[prev])
    if act == "silu":
        m = m / (1.0 + np.exp(-m))
    elif act != "none":
        raise ValueError(act)
    return m


def markov_bias(E, W, prev: int, act: str = "none"):
    return _f64(W) @ markov_rep(E, prev, act)


def gated_rep(E, W_g, h, prev: int, act: str = "none"):
    """The gated Markov head's representation ([READ] 2.3, GatedMarkovHead):
        m = act(E[prev]),  g = sigmoid(W_g [h; m]),  returns g * m
    W_g is [rank, H + rank] (the hidden-state columns first), h the backbone
    hidden state of this position [H]; the bias is then W (g * m)."""
    m = markov_rep(E, prev, act)
    z = _f64(W_g) @ np.concatenate([_f64(h), m])
    g = np.array([sigmoid(v) for v in z])
    return g * m


def rnn_step(E, W_rnn, h, s_prev, prev: int, act: str = "none"):
    """One step of the RNN head ([NOTES] 2.3, the second form, RNN 头;
    [READ] 2.3, the RNNHead row of the table of sequential heads):
        m = act(E[prev]),  u = [s_prev; m; h]
        g = sigmoid(W_g u)                      (gate: how much memory stays)
        c = tanh(W_c u)                         (candidate memory)
        s = g * s_prev + (1 - g) * c            (keep old, write new)
        o = tanh(W_o [s; m; h])                 (the updated input, projected)
    W_rnn is [3, rank, 2 rank + H] holding W_g, W_c, W_o, their columns in
    the order of the concatenation (state, Markov row, hidden state); h is
    the backbone hidden state of this position [H].  Returns (s, o); the
    head's bias is W o."""
    Wr = _f64(W_rnn)
    m = markov_rep(E, prev, act)
    hv = _f64(h)
    u = np.concatenate([s_prev, m, hv])
    g = np.array([sigmoid(v) for v in Wr[0] @ u])
    c = np.tanh(Wr[1] @ u)
    s = g * s_prev + (1.0 - g) * c
    o = np.tanh(Wr[2] @ np.concatenate([s, m, hv]))
    return s, o


def rnn_reps(E, W_rnn, h, prev_tok, tokens, bias_at_first=True, act="none"):
    """o[r, j] of every position of every request, the state starting at
    zero for each request ([NOTES] 2.3: the state is initialised to zero);
    the previous token of position j is prev_tok[r] for j = 0 and
    tokens[r, j-1] after it.  A position without a bias (j = 0 when not
    bias_at_first) has o = 0 and leaves the state at zero."""
    h = np.asarray(h)
    R, G = np.asarray(tokens).shape
    rank = np.asarray(W_rnn).shape[1]
    out = np.zeros((R, G, rank))
    for r in range(R):
        s = np.zeros(rank)
        for j in range(G):
            if j == 0 and not bias_at_first:
                continue
            prev = int(prev_tok[r]) if j == 0 else int(tokens[r, j - 1])
            s, out[r, j] = rnn_step(E, W_rnn, h[r, j], s, prev, act)
    return out


def head_bias(E, W, prev: int, act="none", gate=None, r=0, j=0):
    """Bias of the vanilla head (gate None) or of the gated head, gate =
    dict(h=[R, gamma, H], W_g=[rank, H + rank]) at request r, position j."""
    if gate is None:
        return markov_bias(E, W, prev, act)
    return _f64(W) @ gated_rep(E, gate["W_g"], np.asarray(gate["h"])[r, j], prev, act)


# ---------------------------------------------------------------------------
# a2-a4: sequential propose  ([TRAIN] Markov 顺序修正; [READ] 2.2, 2.3)
# ---------------------------------------------------------------------------

def top_k(ell, K):
    """The K largest entries of ell, largest first; equal values in index
    order (lowest first).  Returns (indices, values)."""
    ell = np.asarray(ell, dtype=np.float64)
    order = np.lexsort((np.arange(ell.size), -ell))[:K]
    return order, ell[order]


def propose(U, E, W, conf, prev_tok, req_id=None, temperature=0.0, seed=0,
            bias_at_first=True, act="none", gate=None, candidates=0, rnn=None):
    """Sequential Markov-head proposal for a batch of R requests.

    For each request r and position j = 0..gamma-1:
        prev  = prev_tok[r] if j == 0 else x[r, j-1]
        l     = U[r, j] + b(prev)        (b omitted at j = 0 if not bias_at_first)
        T = 0: x = argmax l,              lse = logsumexp(l),   l(x)
        T > 0: x = argmax l/T + g,        lse = logsumexp(l/T), l(x)/T
    where g is the stream-0 Gumbel noise of (seed, j, req_id[r]).

    Returns a dict with tokens [R,G] int, lse_q [R,G], logit_at_tok [R,G],
    survival [R,G] (fp64) and margin [R,G] (top-2 gap of the decision
    variable, for the near-tie exemption rule).

    With candidates = K > 0 also the Markov candidate set of every position
    ([TRAIN] Prefix reranker, 候选与前缀表示: C_i = Top16(l_i) of the Markov-
    corrected scores, with the tokens drafted in this round as predecessors): cand_tok [R,G,K] and
    cand_logit [R,G,K] (the biased logits l, largest first, ties by lowest
    token index; token -1 and logit -inf past V when V < K) and cand_gap [R,G] (the gap between the K-th and the
    (K+1)-th largest l, for the near-tie exemption of the set's boundary).

    gate = dict(h, W_g) selects the gated Markov head, rnn = dict(h, W_rnn)
    the RNN head (rnn_step); then the result also holds rep [R,G,rank], the
    representation that W multiplies (g * m, or o)."""
    U = np.asarray(U)
    R, G, V = U.shape
    if req_id is None:
        req_id = np.arange(R)
    T = float(temperature)
    tokens = np.zeros((R, G), dtype=np.int64)
    lse_q = np.zeros((R, G))
    logit_at_tok = np.zeros((R, G))
    margin = np.zeros((R, G))
    K = int(candidates)
    cand_tok = np.zeros((R, G, K), dtype=np.int64)
    cand_logit = np.zeros((R, G, K))
    cand_gap = np.full((R, G), np.inf)
    rank = np.asarray(E).shape[1]
    rep = np.zeros((R, G, rank))
    for r in range(R):
        prev = int(prev_tok[r])
        s_rnn = np.zeros(rank)
        for j in range(G):
            ell = _f64(U[r, j])
            if j > 0 or bias_at_first:
                if rnn is not None:
                    s_rnn, rep[r, j] = rnn_step(E, rnn["W_rnn"], np.asarray(rnn["h"])[r, j],
                                                s_rnn, prev, act)
                    ell = ell + _f64(W) @ rep[r, j]
                else:
                    if gate is not None:
                        rep[r, j] = gated_rep(E, gate["W_g"], np.asarray(gate["h"])[r, j], prev,
                                              act)
                    ell = ell + head_bias(E, W, prev, act, gate, r, j)
            if T == 0.0:
                z = ell
                lse_q[r, j] = logsumexp(ell)
            else:
                s = ell / T
                z = s + vocab_gumbel(seed, j, int(req_id[r]), STREAM_DRAFT, V)
                lse_q[r, j] = logsumexp(s)
            if K:
                idx, val = top_k(ell, K + 1)
                n = min(K, idx.size)
                cand_tok[r, j] = -1                 # a vocabulary smaller than K:
                cand_logit[r, j] = -np.inf          # the missing entries are -1 / -inf
                cand_tok[r, j, :n] = idx[:n]
                cand_logit[r, j, :n] = val[:n]
                if idx.size > K:
                    cand_gap[r, j] = val[K - 1] - val[K]
            x = int(np.argmax(z))              # first maximum: lowest index
            tokens[r, j] = x
            margin[r, j] = top2_margin(z)
            logit_at_tok[r, j] = ell[x] if T == 0.0 else ell[x] / T
            prev = x
    out = dict(tokens=tokens, lse_q=lse_q, logit_at_tok=logit_at_tok,
               survival=survival(conf), margin=margin)
    if K:
        out.update(cand_tok=cand_tok, cand_logit=cand_logit, cand_gap=cand_gap)
    if gate is not None or rnn is not None:
        out.update(rep=rep)
    return out


# ---------------------------------------------------------------------------
# a5: hardware-aware batch-global prefix scheduler  ([READ] 3.2)
# ---------------------------------------------------------------------------

def schedule(a, sps):
    """Greedy global allocation maximising Theta = tau * SPS(B).

    a is [R, gamma] (prefix survival, non-increasing in j); sps[B-1] = SPS(B).
    A survival is a product of probabilities, so values outside [0, 1] are
    clamped to it (the reading taken for confidences, applied to the
    scheduler's own input).
    Start from l_r = 0: B = R, tau = R, Theta* = R * SPS(R).  Visit the
    (r, j) items in order of a descending (ties: r, then j ascending); each
    visit adds one verify slot (B += 1) and its expected token (tau += a).
    Keep the cut with the largest Theta (strictly larger wins, so the
    smallest B attaining the maximum is kept).  Items beyond the SPS table
    are infeasible.  keep_len[r] = number of kept items of request r.

    Returns dict(keep_len [R] int, theta, B, theta_gap) where theta_gap is the
    relative gap between Theta* and the best Theta at any other cut (used to
    count near-ties)."""
    a = np.clip(_f64(a), 0.0, 1.0)
    sps = _f64(sps)
    R, G = a.shape
    n_sps = sps.shape[0]
    if R < 1 or R > n_sps:
        raise ValueError("R outside the SPS table")
    items = sorted(((a[r, j], r, j) for r in range(R) for j in range(G)),
                   key=lambda it: (-it[0], it[1], it[2]))
    tau = float(R)
    best_theta = R * sps[R - 1]
    best_k = 0
    thetas = [best_theta]
    for k, (av, r, j) in enumerate(items, start=1):
        B = R + k
        if B > n_sps:
            break
        tau = tau + av
        theta = tau * sps[B - 1]
        thetas.append(theta)
        if theta > best_theta:
            best_theta = theta
            best_k = k
    keep_len = np.zeros(R, dtype=np.int64)
    for (av, r, j) in items[:best_k]:
        keep_len[r] += 1
    others = [t for k, t in enumerate(thetas) if k != best_k]
    gap = (best_theta - max(others)) / abs(best_theta) if others and best_theta != 0 else float("inf")
    return dict(keep_len=keep_len, theta=float(best_theta), B=R + best_k,
                theta_gap=float(gap), sorted_items=items)


# ---------------------------------------------------------------------------
# a6/a7: target verification  ([WALK] 4.4; [READ] 2.1, 3.1)
# ---------------------------------------------------------------------------

def _draft_logits(U, E, W, prev_tok, tokens, r, t, bias_at_first, act, gate=None, rnn=None):
    ell = _f64(U[r, t])
    prev = int(prev_tok[r]) if t == 0 else int(tokens[r, t - 1])
    if t > 0 or bias_at_first:
        if rnn is not None:
            # the RNN state at t replays the recursion over the drafted tokens
            o = rnn_reps(E, rnn["W_rnn"], np.asarray(rnn["h"])[r:r + 1],
                         np.asarray(prev_tok)[r:r + 1], np.asarray(tokens)[r:r + 1, :t + 1],
                         bias_at_first, act)[0, t]
            ell = ell + _f64(W) @ o
        else:
            ell = ell + head_bias(E, W, prev, act, gate, r, t)
    return ell


def accept_probability(p_x, q_x):
    """[WALK] 4.4 (the accept test of the verify step): the draft token x is
    kept with probability min(1, p(x) / q(x))."""
    return min(1.0, p_x / q_x)


def correction_weights(p, q):
    """[WALK] 4.4: after a rejection the next token is drawn from the residual
    max(0, p - q), renormalised.  Returns the unnormalised weights and whether
    the empty-residual reading applied: if sum(max(0, p - q)) <= 1e-12 sum(p),
    which only rounding can produce, the draw falls back to p itself."""
    res = np.maximum(0.0, p - q)
    if np.sum(res) <= 1e-12 * np.sum(p):
        return p, True
    return res, False


def verify(P, U, E, W, prev_tok, tokens, keep_len, req_id=None,
           temperature=0.0, seed=0, bias_at_first=True, act="none", gate=None, rnn=None):
    """Rejection verification of the kept prefix of every request.

    P is [R, gamma+1, V]: row t scores draft token x_t, row keep_len[r] gives
    the bonus distribution.  The draft distribution q_t = softmax(l_t / T) is
    recomputed here from U, E, W and the draft tokens (its definition).

    T > 0, for t = 0..keep_len-1: accept x_t iff u_t < min(1, p_t(x_t)/q_t(x_t))
    (u_t: stream-1 uniform of (seed, t, req)); stop at the first rejection k.
    If k < keep_len the next token is drawn from norm(max(0, p_k - q_k)) by
    Gumbel-max on stream 2; otherwise the bonus token is drawn from p at row
    keep_len by Gumbel-max on stream 3.
    T = 0: accept iff x_t == argmax P[r, t]; the correction / bonus is argmax P.

    Returns dict(accept_len [R], next_token [R]) plus diagnostics:
    accept_gap [R] (smallest |u - min(1,p/q)| over the tests taken, or the
    smallest argmax margin in greedy mode) and next_margin [R]."""
    P = np.asarray(P)
    R = P.shape[0]
    V = P.shape[2]
    if req_id is None:
        req_id = np.arange(R)
    T = float(temperature)
    accept_len = np.zeros(R, dtype=np.int64)
    next_token = np.zeros(R, dtype=np.int64)
    accept_gap = np.full(R, np.inf)
    next_margin = np.zeros(R)
    for r in range(R):
        L = int(keep_len[r])
        req = int(req_id[r])
        k = L
        p_k = q_k = None
        for t in range(L):
            x = int(tokens[r, t])
            if T == 0.0:
                row = _f64(P[r, t])
                accept_gap[r] = min(accept_gap[r], top2_margin(row))
                ok = int(np.argmax(row)) == x
            else:
                p = softmax(_f64(P[r, t]) / T)
                q = softmax(_draft_logits(U, E, W, prev_tok, tokens, r, t,
                                          bias_at_first, act, gate, rnn) / T)
                accept_prob = accept_probability(p[x], q[x])
                u = accept_uniform(seed, t, req)
                accept_gap[r] = min(accept_gap[r], abs(u - accept_prob))
                ok = u < accept_prob
                if not ok:
                    p_k, q_k = p, q
            if not ok:
                k = t
                break
        if k < L:
            if T == 0.0:
                z = _f64(P[r, k])
            else:
                w, _ = correction_weights(p_k, q_k)
                g = vocab_gumbel(seed, k, req, STREAM_RESIDUAL, V)
                with np.errstate(divide="ignore"):
                    z = np.where(w > 0.0, np.log(w), -np.inf) + g
        else:
            if T == 0.0:
                z = _f64(P[r, L])
            else:
                z = _f64(P[r, L]) / T + vocab_gumbel(seed, L, req, STREAM_BONUS, V)
        accept_len[r] = k
        next_token[r] = int(np.argmax(z))
        finite = z[np.isfinite(z)]
        next_margin[r] = top2_margin(finite) if finite.size > 1 else float("inf")
    return dict(accept_len=accept_len, next_token=next_token,
                accept_gap=accept_gap, next_margin=next_margin)


# ---------------------------------------------------------------------------
# a8: offline overlap metrics  ([TRAIN] 评估口径 / 离线指标; [READ] 3.1)
# ---------------------------------------------------------------------------

def overlap(P_logits, Q_logits, valid_len):
    """Teacher-forced overlap metrics of N blocks of gamma positions.

    For each block n and valid position i < valid_len[n]:
        p = softmax(P[n, i]), q = softmax(Q[n, i])
        a[n, i]  = sum_v min(p, q)
        l1[n, i] = sum_v |p - q|        (so a = 1 - l1/2 by the identity)
    invalid positions have a = 0 (and l1 = 0).
        tau[n] = 1 + sum_i prod_{j <= i} a[n, j]
        accept_rate[i] = mean of a[n, i] over blocks with position i valid
        mean_tau = mean of tau over valid blocks (valid_len >= 1)
    Empty averages are reported as 0."""
    P = np.asarray(P_logits)
    Q = np.asarray(Q_logits)
    N, G, V = P.shape
    vl = np.asarray(valid_len).astype(np.int64)
    a = np.zeros((N, G))
    l1 = np.zeros((N, G))
    tau = np.zeros(N)
    for n in range(N):
        L = int(vl[n])
        for i in range(min(max(L, 0), G)):
            p = softmax(_f64(P[n, i]))
            q = softmax(_f64(Q[n, i]))
            a[n, i] = np.sum(np.minimum(p, q))
            l1[n, i] = np.sum(np.abs(p - q))
        acc = 1.0
        t = 1.0
        for i in range(G):
            acc = acc * a[n, i]
            t = t + acc
        tau[n] = t
    accept_rate = np.zeros(G)
    for i in range(G):
        sel = vl > i
        accept_rate[i] = float(np.mean(a[sel, i])) if np.any(sel) else 0.0
    valid = vl >= 1
    mean_tau = float(np.mean(tau[valid])) if np.any(valid) else 0.0
    return dict(a=a, l1=l1, tau=tau, accept_rate=accept_rate, mean_tau=mean_tau)


# ---------------------------------------------------------------------------
# Teacher-forced Markov bias and the DSpark loss forward  ([READ] 2.3
# VanillaMarkov.apply_block_logits: the bias of every block position at once
# from known previous tokens; [READ] 4.1 位置指数衰减与分布 L1 对齐损失)
# ---------------------------------------------------------------------------

def position_weights(gamma: int, decay: float = 4.0):
    """w_j = exp(-j / decay), normalised to sum 1 ([READ] 4.1)."""
    w = np.exp(-np.arange(gamma, dtype=np.float64) / decay)
    return w / np.sum(w)


def bce_with_logits(z, y):
    """Binary cross-entropy of the logit z against the soft label y:
    -(y log sigma(z) + (1 - y) log(1 - sigma(z))), with
    log sigma(z) = -log(1 + e^-z) and log(1 - sigma(z)) = -log(1 + e^z)."""
    z = float(z)
    y = float(y)
    log_sig = -np.logaddexp(0.0, -z)
    log_one_minus = -np.logaddexp(0.0, z)
    return -(y * log_sig + (1.0 - y) * log_one_minus)


def loss_forward(U, E, W, prev_tokens, P, target_tokens, conf_logits,
                 bias_at_first=True, act="none", ce_alpha=0.1, l1_alpha=0.9,
                 conf_alpha=1.0, decay=4.0):
    """DSpark loss forward over B blocks of gamma teacher-forced positions.

    For each block b and position j (prev_tokens[b, j] is the known token
    before position j; position 0 is biased unless bias_at_first is False):
        l[v]   = U[b, j, v] + b_j[v],  b_j = W E[prev_tokens[b, j]]
        q      = softmax(l),  p = softmax(P[b, j])
        l1     = sum_v |p - q|
        a      = clamp(1 - l1 / 2, 0, 1)          (soft accept-rate label)
        ce     = logsumexp(l) - l[target_tokens[b, j]]     (-log q(x*))
        bce    = BCE(conf_logits[b, j], a)
    Aggregates with w = position_weights(gamma, decay):
        ce_loss   = sum_j w_j mean_b ce[b, j]
        l1_loss   = sum_j w_j mean_b l1[b, j]
        conf_loss = mean_{b, j} bce[b, j]
        loss      = ce_alpha ce_loss + l1_alpha l1_loss + conf_alpha conf_loss"""
    U = np.asarray(U)
    B, G, V = U.shape
    prev = np.asarray(prev_tokens).astype(np.int64)
    tgt = np.asarray(target_tokens).astype(np.int64)
    z = _f64(conf_logits)
    l1 = np.zeros((B, G))
    a = np.zeros((B, G))
    ce = np.zeros((B, G))
    bce = np.zeros((B, G))
    for b in range(B):
        for j in range(G):
            l = _f64(U[b, j])
            if j > 0 or bias_at_first:
                l = l + markov_bias(E, W, int(prev[b, j]), act)
            q = softmax(l)
            p = softmax(_f64(P[b, j]))
            l1[b, j] = np.sum(np.abs(p - q))
            a[b, j] = min(1.0, max(0.0, 1.0 - 0.5 * l1[b, j]))
            ce[b, j] = logsumexp(l) - l[int(tgt[b, j])]
            bce[b, j] = bce_with_logits(z[b, j], a[b, j])
    w = position_weights(G, decay)
    ce_loss = float(np.sum(w * np.mean(ce, axis=0))) if B else 0.0
    l1_loss = float(np.sum(w * np.mean(l1, axis=0))) if B else 0.0
    conf_loss = float(np.mean(bce)) if B else 0.0
    loss = ce_alpha * ce_loss + l1_alpha * l1_loss + conf_alpha * conf_loss
    return dict(l1=l1, accept=a, ce=ce, bce=bce, ce_loss=ce_loss, l1_loss=l1_loss,
                conf_loss=conf_loss, loss=loss)


# ---------------------------------------------------------------------------
# One whole draft-verify cycle (propose -> schedule -> verify), as the pages'
# serving loop runs it ([WALK] 4.2), used by the cycle parity tests and the
# CPU baseline.
# ---------------------------------------------------------------------------

def cycle(U, E, W, conf, prev_tok, P, sps, req_id=None, temperature=0.0,
          seed=0, bias_at_first=True, act="none", keep_len=None, gate=None, rnn=None):
    prop = propose(U, E, W, conf, prev_tok, req_id, temperature, seed,
                   bias_at_first, act, gate, rnn=rnn)
    a32 = prop["survival"].astype(np.float32)       # the schedule's input type
    sch = schedule(a32, sps)
    kl = sch["keep_len"] if keep_len is None else np.asarray(keep_len)
    ver = verify(P, U, E, W, prev_tok, prop["tokens"], kl, req_id,
                 temperature, seed, bias_at_first, act, gate, rnn)
    return dict(propose=prop, schedule=sch, verify=ver, keep_len=kl)


# ---------------------------------------------------------------------------
# Confidence side: the confidence head, static threshold truncation and the
# calibration metrics of the survival probabilities
# ([TRAIN] Confidence head 与训练目标; [WALK] 4.3 Propose;
#  [READ] 3.1 prefix survival and its monitoring, 5 reliability diagram)
# ---------------------------------------------------------------------------

def sigmoid(z):
    """1 / (1 + e^-z), written per sign so neither branch overflows."""
    z = float(z)
    if z >= 0.0:
        return 1.0 / (1.0 + np.exp(-z))
    e = np.exp(z)
    return e / (1.0 + e)


def confidence_head(h, E, w_c, b_c, prev_tok, tokens):
    """Per-position confidence of the drafted tokens ([TRAIN] Confidence head):
        s[r, j] = w_c . [h[r, j]; m[r, j]] + b_c,   c[r, j] = sigmoid(s[r, j])
    with m[r, j] = E[t_{j-1}] the Markov table row of the token before
    position j (the anchor prev_tok[r] at j = 0, the drafted tokens[r, j-1]
    after it) and w_c of length H + r (h part first).  Returns the logits s,
    the confidences c and the prefix survival a = survival(c)."""
    h = _f64(h)
    R, G, H = h.shape
    w = _f64(w_c)
    rank = np.asarray(E).shape[1]
    if w.shape != (H + rank,):
        raise ValueError("w_c must have H + rank entries")
    s = np.zeros((R, G))
    c = np.zeros((R, G))
    for r in range(R):
        for j in range(G):
            t = int(prev_tok[r]) if j == 0 else int(tokens[r, j - 1])
            x = np.concatenate([h[r, j], _f64(E[t])])
            s[r, j] = float(np.dot(w, x)) + float(b_c)
            c[r, j] = sigmoid(s[r, j])
    return dict(logit=s, conf=c, survival=survival(c))


def threshold_keep(conf, threshold):
    """Static confidence truncation ([WALK] 4.3: proposal_len =
    min(block, first position whose confidence is below the threshold)):
    keep[r] = number of leading positions j with conf[r, j] >= threshold.
    A threshold of 0 keeps every position.  The threshold is an fp32
    argument of the library call, so it is rounded to fp32 here too and the
    comparison is the fp32 one (exact in fp64 after widening both)."""
    c = _f64(conf)
    threshold = float(np.float32(threshold))
    R, G = c.shape
    keep = np.zeros(R, dtype=np.int64)
    for r in range(R):
        k = 0
        while k < G and c[r, k] >= threshold:
            k += 1
        keep[r] = k
    return keep


def calibration(conf, accept_len, n_bins=10):
    """Calibration of predicted survival against realised acceptance
    ([READ] 3.1: per-step error and the cumulative-product bias; [READ] 5:
    reliability diagram and ECE).  conf [M, gamma] are the predicted per-step
    confidences (clamped to [0, 1]); accept_len [M] the accepted prefix
    lengths of full-block verification.  With a = survival(conf):
      realised survival     y[r, j] = 1 if j < accept_len[r] else 0
      tested positions      j <= accept_len[r] (and j < gamma), whose
                            realised step outcome is y[r, j]
      abs_error    = mean over tested positions of |conf - y|
      cumprod_bias = mean over all positions of (a - y)   (> 0: optimistic)
      pos_pred[j], pos_real[j] = means over requests of a[:, j] and y[:, j]
      reliability bins of a: b = min(floor(a n_bins), n_bins - 1); per bin
      the count, the mean of a and the mean of y (0 for an empty bin)
      ece = sum_b count_b / (M gamma) |mean a_b - mean y_b|
    Empty means are 0."""
    c = np.clip(_f64(conf), 0.0, 1.0)
    M, G = c.shape
    L = np.asarray(accept_len).astype(np.int64)
    if np.any(L < 0) or np.any(L > G):
        raise ValueError("accept_len outside 0..gamma")
    a = survival(c)
    cnt = np.zeros(n_bins, dtype=np.int64)
    sp = np.zeros(n_bins)
    sr = np.zeros(n_bins)
    err_sum, n_tested, bias_sum = 0.0, 0, 0.0
    pos_pred = np.zeros(G)
    pos_real = np.zeros(G)
    for r in range(M):
        for j in range(G):
            y = 1.0 if j < L[r] else 0.0
            if j <= L[r]:
                err_sum += abs(c[r, j] - y)
                n_tested += 1
            bias_sum += a[r, j] - y
            pos_pred[j] += a[r, j]
            pos_real[j] += y
            b = min(int(np.floor(a[r, j] * n_bins)), n_bins - 1)
            cnt[b] += 1
            sp[b] += a[r, j]
            sr[b] += y
    total = M * G
    mean_pred = np.where(cnt > 0, sp / np.maximum(cnt, 1), 0.0)
    mean_real = np.where(cnt > 0, sr / np.maximum(cnt, 1), 0.0)
    ece = float(np.sum(cnt / total * np.abs(mean_pred - mean_real))) if total else 0.0
    return dict(count=cnt, mean_pred=mean_pred, mean_real=mean_real, ece=ece,
                abs_error=err_sum / n_tested if n_tested else 0.0,
                cumprod_bias=bias_sum / total if total else 0.0,
                n_tested=n_tested,
                pos_pred=pos_pred / M if M else pos_pred,
                pos_real=pos_real / M if M else pos_real)


def auroc(conf, accept_len):
    """Ranking quality of predicted survival ([READ] 5: the raw confidence
    head's AUROC beside its reliability diagram).  Reading: over all (r, j)
    positions, the score is the predicted prefix survival a[r, j] (fp64
    product of the clamped confidences, as in calibration) and the label the
    realised survival y[r, j] = (j < accept_len[r]).  AUROC is the
    probability that a random positive outscores a random negative, a tie
    counting one half (the Mann-Whitney statistic over all pairs).  With no
    positive or no negative it is 0.5.  Written with a stable sort: within a
    run of equal scores each positive meets the run's negatives as ties."""
    c = np.clip(_f64(conf), 0.0, 1.0)
    M, G = c.shape
    L = np.asarray(accept_len).astype(np.int64)
    a = survival(c).reshape(-1)
    y = (np.arange(G)[None, :] < L[:, None]).reshape(-1)
    n_pos = int(y.sum())
    n_neg = y.size - n_pos
    if n_pos == 0 or n_neg == 0:
        return 0.5
    order = np.argsort(a, kind="stable")
    a_s, y_s = a[order], y[order]
    u = 0.0
    neg_below = 0            # negatives with a strictly smaller score
    i = 0
    while i < a_s.size:
        k = i
        while k < a_s.size and a_s[k] == a_s[i]:
            k += 1
        pos_run = int(y_s[i:k].sum())
        neg_run = (k - i) - pos_run
        u += pos_run * (neg_below + 0.5 * neg_run)
        neg_below += neg_run
        i = k
    return u / (n_pos * n_neg)

