"""dsd_propose_candidates (the Markov top-16 candidate set along the drafted
chain) against the oracle's propose(candidates=16), through the C ABI.

Agreement: the 16 biased logits of a set within 1e-4 (fp32 sums of exact
products, as for the draft logits); a token must equal the oracle's at its
rank unless an oracle logit within 1e-3 lies next to it (then it must be one
of those near-equal tokens), and the 16th is exempt when the 16th and 17th
oracle logits are within 1e-3.  Rows after a near-tie of the drafted chain
are exempt (their predecessors differ)."""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
K = 16
TIE = 1e-3


@pytest.fixture(scope="module")
def dsd():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from semi_autoregressive_draft_gb300 import build as b

    b.build()
    import semi_autoregressive_draft_gb300 as m

    return m


def host(x):
    return {k: synth.to_numpy(v) for k, v in x.items() if isinstance(v, torch.Tensor)}


def compare_candidates(k, o, rows_exempt):
    R, G = k["tokens"].shape
    checked = 0
    for r in range(R):
        for j in range(G):
            if rows_exempt[r, j]:
                continue
            kt, kv = k["cand_tok"][r, j], k["cand_logit"][r, j]
            ot, ov = o["cand_tok"][r, j], o["cand_logit"][r, j]
            n = int(np.isfinite(ov).sum())        # fewer than K when V < K
            assert np.array_equal(kt[n:], ot[n:]) and np.all(np.isinf(kv[n:]))
            assert np.max(np.abs(kv[:n] - ov[:n])) <= parity.LOGIT_TOL, (r, j)
            for t in range(n):
                if t == n - 1 and o["cand_gap"][r, j] < TIE:
                    continue
                near = np.abs(ov - ov[t]) < TIE
                if near.sum() == 1:
                    assert kt[t] == ot[t], (r, j, t, kt, ot)
                else:
                    assert kt[t] in set(ot[near].tolist()), (r, j, t)
            assert len(set(kt[:n].tolist())) == n   # no token twice
            checked += 1
    return checked


def run(dsd, spec, n_sample=None, seed_idx=0, engine="simt"):
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, engine=engine)
    T = spec.temperature
    out = ctx.propose_candidates(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                                 req_id=x["req_id"], temperature=T, seed=x["seed"])
    plain = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], req_id=x["req_id"],
                        temperature=T, seed=x["seed"])
    assert ctx.sync_status() == 0
    k = {n: t.cpu().numpy() for n, t in out.items()}
    ctx.close()
    h = host(x)
    idx = np.arange(spec.R) if n_sample is None else \
        np.sort(np.random.default_rng(70 + seed_idx).choice(spec.R, n_sample, replace=False))
    rid = h["req_id"].astype(np.int64)[idx]
    o = O.propose(h["U"][idx], h["E"], h["W"], h["conf"][idx], h["prev_tok"][idx], rid, T,
                  x["seed"], candidates=K)
    ks = {n: v[idx] for n, v in k.items()}
    parity.compare_propose(ks, o)
    ex = parity.draft_exempt(o["margin"])
    # a position's set depends on the previous tokens only
    rows_ex = np.zeros_like(ex)
    rows_ex[:, 1:] = ex[:, :-1]
    assert compare_candidates(ks, o, rows_ex) > 0
    return k, plain


@pytest.mark.parametrize("temperature,dtype", [(0.0, "bf16"), (1.0, "bf16"), (0.0, "f32"),
                                               (0.7, "f32")])
def test_candidates_small(dsd, temperature, dtype):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=71,
                        dtype=dtype, r=64, V=2568, R=19, ew_std=0.3)
    k, plain = run(dsd, spec)
    # the proposal itself is the plain head's, and greedy picks the top candidate
    assert torch.equal(plain["tokens"].cpu(), torch.as_tensor(k["tokens"]))
    if temperature == 0.0:
        assert np.array_equal(k["cand_tok"][:, :, 0], k["tokens"])


def test_candidates_tiny_vocabulary_and_capacity(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["tiny"], seed=72, V=8, r=8, R=3, ew_std=0.3)
    k, _ = run(dsd, spec)
    assert np.all(k["cand_tok"][:, :, 8:] == -1)
    assert np.all(np.isinf(k["cand_logit"][:, :, 8:]))
    x = synth.cycle_inputs(synth.scaled(synth.CYCLE_SPECS["greedy"], seed=73, V=1032, r=64,
                                        R=33), device=DEV)
    ctx = dsd.Context(1032, 64, 7, 33, dtype="bf16")
    with pytest.raises(dsd.DsdError):
        ctx.propose_candidates(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"])
    ctx.close()


def test_candidates_full_size_sampled_requests(dsd):
    # the greedy workload: R = 16, V = 151936, rank 256
    run(dsd, synth.CYCLE_SPECS["greedy"], n_sample=4)


@pytest.mark.parametrize("R,rank,temperature", [(19, 64, 0.0), (19, 256, 1.0), (32, 128, 0.0),
                                                (1, 64, 0.6)])
def test_candidates_on_the_tensor_cores(dsd, R, rank, temperature):
    # the tensor-core engine's repeated-rows kernel keeps the lists (21 tiles
    # of 128 with an 8-row tail; one request; the 32-request maximum)
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=74 + R,
                        r=rank, V=2568, R=R, ew_std=0.3)
    k, plain = run(dsd, spec, engine="tcgen05")
    assert torch.equal(plain["tokens"].cpu(), torch.as_tensor(k["tokens"]))
    if temperature == 0.0:
        assert np.array_equal(k["cand_tok"][:, :, 0], k["tokens"])


def test_candidates_on_the_tensor_cores_full_size_sampled_requests(dsd):
    # the greedy workload (R = 16, V = 151936, rank 256) on AUTO, which takes
    # the tensor-core engine
    run(dsd, synth.CYCLE_SPECS["greedy"], n_sample=4, engine="auto")


def test_candidates_on_the_tensor_cores_one_position(dsd):
    # gamma = 1: one launch for the one step (no per-position counter)
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=0.0, seed=79, r=64, V=2568,
                        R=7, G=1, ew_std=0.3)
    k, plain = run(dsd, spec, engine="tcgen05")
    assert np.array_equal(k["cand_tok"][:, :, 0], k["tokens"])
