"""dsd_propose_rnn / dsd_verify_rnn (the RNN head on the CUDA-core engine)
against the oracle's propose / verify with the RNN head, through the C ABI.
Same agreement rules as the plain head: tokens, keep and accept lengths
bit-exact outside counted near-ties; log-normalisers and logits within 1e-4.
The head adds fp32 dot products of 2 rank + H terms per gate, candidate and
output (relative rounding ~1e-6) and a seven-step fp32 recursion before the
bias projection; its output o_j is compared within 1e-4 on every position
whose drafted prefix matches the oracle's."""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
SMALL = dict(V=2568, R=19, ew_std=0.3)
REP_TOL = 1e-4


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


def run_rnn(dsd, spec, rx, bias_at_first=True, keep_all=False, act="none",
            engine="auto"):
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, act=act,
                      bias_at_first=bias_at_first, engine=engine)
    T = spec.temperature
    prop = ctx.propose_rnn(x["U"], x["E"], x["W"], rx["h"], rx["W_rnn"], x["conf"], x["prev_tok"],
                           req_id=x["req_id"], temperature=T, seed=x["seed"])
    sch = ctx.schedule(prop["survival"], x["sps"])
    keep = torch.full_like(sch["keep_len"], spec.G) if keep_all else sch["keep_len"]
    ver = ctx.verify_rnn(x["P"], prop["tokens"], keep, rnn_rep=prop["rnn_rep"], U=x["U"],
                         E=x["E"], W=x["W"], prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                         logit_at_tok=prop["logit_at_tok"], req_id=x["req_id"], temperature=T,
                         seed=x["seed"])
    assert ctx.sync_status() == 0
    k = {n: t.cpu().numpy() for n, t in {**prop, **sch, **ver}.items()}
    k["keep_used"] = keep.cpu().numpy()
    ctx.close()
    return x, k


def check_rnn(spec, x, rx, k, bias_at_first=True, act="none"):
    h = host(x)
    rnn = dict(h=synth.to_numpy(rx["h"]), W_rnn=synth.to_numpy(rx["W_rnn"]))
    rid = h["req_id"].astype(np.int64)
    T = spec.temperature
    prop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"], rid, T, x["seed"],
                     bias_at_first, act, rnn=rnn)
    rep = parity.compare_propose(k, prop)
    keep = k["keep_used"]
    ver = O.verify(h["P"], h["U"], h["E"], h["W"], h["prev_tok"], prop["tokens"], keep, rid, T,
                   x["seed"], bias_at_first, act, rnn=rnn)
    ex = parity.draft_exempt(prop["margin"])
    draft_ex = np.array([ex[r, :keep[r] + 1].any() if keep[r] < spec.G else ex[r].any()
                         for r in range(spec.R)])
    parity.compare_verify(k["accept_len"], k["next_token"], ver, T, keep, draft_ex)
    assert rep.exempt <= 0.05 * (rep.checked + rep.exempt) + 1, f"too many exemptions: {rep}"
    # o_j of every position whose predecessors match the oracle's
    compared = 0
    for q in range(spec.R):
        for j in range(spec.G):
            if j > 0 and ex[q, :j].any():
                break
            assert np.max(np.abs(k["rnn_rep"][q, j] - prop["rep"][q, j])) <= REP_TOL, (q, j)
            compared += 1
    assert compared > 0
    return rep


@pytest.mark.parametrize("temperature,keep_all", [(0.0, False), (1.0, False), (1.0, True),
                                                  (0.6, False)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_rnn_cycle_small(dsd, temperature, keep_all, dtype):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=81,
                        p_noise=1.0 if temperature else 0.5, dtype=dtype, r=64, **SMALL)
    rx = synth.rnn_inputs(spec.R, spec.G, 328, spec.r, spec.ew_std, seed=82, dtype=dtype,
                          device=DEV)
    x, k = run_rnn(dsd, spec, rx, keep_all=keep_all)
    check_rnn(spec, x, rx, k)


def test_rnn_no_bias_at_first_and_silu(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=83, p_noise=1.0,
                        r=64, **SMALL)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=84, device=DEV)
    x, k = run_rnn(dsd, spec, rx, bias_at_first=False, act="silu")
    check_rnn(spec, x, rx, k, bias_at_first=False, act="silu")
    assert np.all(k["rnn_rep"][:, 0] == 0.0)


def test_rnn_repeated_calls_reset_the_state(dsd):
    # the recurrent state starts from zero in every call: two calls on the
    # same context give the same result
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=85, p_noise=1.0,
                        r=64, **SMALL)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=86, device=DEV)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype)
    outs = [ctx.propose_rnn(x["U"], x["E"], x["W"], rx["h"], rx["W_rnn"], x["conf"],
                            x["prev_tok"], req_id=x["req_id"], temperature=1.0, seed=x["seed"])
            for _ in range(2)]
    assert ctx.sync_status() == 0
    for n in ("tokens", "lse_q", "rnn_rep"):
        assert torch.equal(outs[0][n], outs[1][n]), n
    ctx.close()


def test_rnn_full_size_sampled_requests(dsd):
    # the greedy workload (R = 16, V = 151936, rank 256) with H = 2560
    spec = synth.CYCLE_SPECS["greedy"]
    rx = synth.rnn_inputs(spec.R, spec.G, 2560, spec.r, spec.ew_std, seed=87, device=DEV)
    x, k = run_rnn(dsd, spec, rx)
    idx = np.array([0, 6, 13, 15])
    h = host(x)
    rnn = dict(h=synth.to_numpy(rx["h"])[idx], W_rnn=synth.to_numpy(rx["W_rnn"]))
    rid = h["req_id"].astype(np.int64)[idx]
    prop = O.propose(h["U"][idx], h["E"], h["W"], h["conf"][idx], h["prev_tok"][idx], rid, 0.0,
                     x["seed"], True, "none", rnn=rnn)
    parity.compare_propose({n: k[n][idx] for n in ("tokens", "lse_q", "logit_at_tok",
                                                     "survival")}, prop)
    ex = parity.draft_exempt(prop["margin"])
    for qi in range(len(idx)):
        for j in range(spec.G):
            if j > 0 and ex[qi, :j].any():
                break
            assert np.max(np.abs(k["rnn_rep"][idx[qi], j] - prop["rep"][qi, j])) <= REP_TOL


def test_rnn_errors(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=88, r=64, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=89, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    with pytest.raises(dsd.DsdError):   # H not a multiple of 8
        ctx.propose_rnn(x["U"], x["E"], x["W"], rx["h"][:, :, :60].contiguous(),
                        rx["W_rnn"][:, :, 4:].contiguous(), x["conf"], x["prev_tok"])
    h = rx["h"].clone()
    h[3, 2, 7] = float("nan")
    ctx.propose_rnn(x["U"], x["E"], x["W"], h, rx["W_rnn"], x["conf"], x["prev_tok"])
    assert ctx.sync_status() == -6
    ctx.close()


@pytest.mark.parametrize("engine,R,temperature", [("simt", 19, 1.0), ("tcgen05", 70, 1.0),
                                                  ("tcgen05", 19, 0.0)])
def test_rnn_on_each_engine(dsd, engine, R, temperature):
    # the CUDA-core engine, and the tensor-core engine's split mode
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=80 + R,
                        p_noise=1.0, r=64, R=R, V=2568, ew_std=0.3)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=81, device=DEV)
    x, k = run_rnn(dsd, spec, rx, engine=engine)
    check_rnn(spec, x, rx, k)



def test_rnn_in_launch_step_matches_the_step_kernels(dsd):
    # the tensor-core engine runs the state and output phases inside its
    # one-launch proposal, the CUDA-core engine the standalone step kernels;
    # the same warp routines, so equal drafted prefixes give equal bits
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=85, p_noise=1.0,
                        r=64, R=40, V=2568, ew_std=0.3)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=86, device=DEV)
    _, kt = run_rnn(dsd, spec, rx, engine="tcgen05")
    _, ks = run_rnn(dsd, spec, rx, engine="simt")
    same = 0
    for q in range(spec.R):
        for j in range(spec.G):
            if np.array_equal(kt["tokens"][q, :j], ks["tokens"][q, :j]):
                same += 1
                assert np.array_equal(kt["rnn_rep"][q, j].view(np.uint32),
                                      ks["rnn_rep"][q, j].view(np.uint32)), (q, j)
    assert same >= 0.9 * spec.R * spec.G, same


@pytest.mark.parametrize("G", [1, 2])
def test_rnn_short_blocks_on_the_tensor_cores(dsd, G):
    # gamma = 1: the standalone state and output kernels before one step
    # launch; gamma = 2: both phases inside the one-launch proposal
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=87 + G, p_noise=1.0,
                        r=64, R=19, G=G, V=2568, ew_std=0.3)
    rx = synth.rnn_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=88, device=DEV)
    x, k = run_rnn(dsd, spec, rx, engine="tcgen05")
    check_rnn(spec, x, rx, k)
