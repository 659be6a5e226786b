"""dsd_propose_gated / dsd_verify_gated (the gated Markov head on the
CUDA-core engine) against the oracle's propose / verify with the gate,
through the C ABI.  Same agreement rules as the plain head: tokens, keep and
accept lengths bit-exact outside counted near-ties; log-normalisers and
logits within 1e-4.  The gate adds an fp32 dot product of H + rank terms
per gate (relative rounding ~1e-6) before the bias GEMV."""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
SMALL = dict(V=2568, R=19, ew_std=0.3)


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


def run_gated(dsd, spec, gx, bias_at_first=True, keep_all=False, act="none",
              engine="auto"):
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, act=act,
                      bias_at_first=bias_at_first, engine=engine)
    T = spec.temperature
    prop = ctx.propose_gated(x["U"], x["E"], x["W"], gx["h"], gx["W_g"], x["conf"], x["prev_tok"],
                             req_id=x["req_id"], temperature=T, seed=x["seed"])
    sch = ctx.schedule(prop["survival"], x["sps"])
    keep = torch.full_like(sch["keep_len"], spec.G) if keep_all else sch["keep_len"]
    ver = ctx.verify_gated(x["P"], prop["tokens"], keep, gated_rep=prop["gated_rep"], U=x["U"],
                           E=x["E"], W=x["W"], prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                           logit_at_tok=prop["logit_at_tok"], req_id=x["req_id"], temperature=T,
                           seed=x["seed"])
    assert ctx.sync_status() == 0
    k = {n: t.cpu().numpy() for n, t in {**prop, **sch, **ver}.items()}
    k["keep_used"] = keep.cpu().numpy()
    ctx.close()
    return x, k


def check_gated(spec, x, gx, k, bias_at_first=True, act="none"):
    h = host(x)
    gate = dict(h=synth.to_numpy(gx["h"]), W_g=synth.to_numpy(gx["W_g"]))
    rid = h["req_id"].astype(np.int64)
    T = spec.temperature
    prop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"], rid, T, x["seed"],
                     bias_at_first, act, gate)
    rep = parity.compare_propose(k, prop)
    keep = k["keep_used"]
    ver = O.verify(h["P"], h["U"], h["E"], h["W"], h["prev_tok"], prop["tokens"], keep, rid, T,
                   x["seed"], bias_at_first, act, gate)
    ex = parity.draft_exempt(prop["margin"])
    draft_ex = np.array([ex[r, :keep[r] + 1].any() if keep[r] < spec.G else ex[r].any()
                         for r in range(spec.R)])
    parity.compare_verify(k["accept_len"], k["next_token"], ver, T, keep, draft_ex)
    assert rep.exempt <= 0.05 * (rep.checked + rep.exempt) + 1, f"too many exemptions: {rep}"
    # the gated representation of every position, against its definition
    G, r = spec.G, spec.r
    for q in range(spec.R):
        prev = int(h["prev_tok"][q])
        for j in range(G):
            if j == 0 and not bias_at_first:
                ref = np.zeros(r)
            else:
                ref = O.gated_rep(h["E"], gate["W_g"], gate["h"][q, j], prev, act)
            assert np.max(np.abs(k["gated_rep"][q, j] - ref)) <= 1e-4, (q, j)
            prev = int(prop["tokens"][q, j])
    return rep


@pytest.mark.parametrize("temperature,keep_all", [(0.0, False), (1.0, False), (1.0, True),
                                                  (0.6, False)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gated_cycle_small(dsd, temperature, keep_all, dtype):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=61,
                        p_noise=1.0 if temperature else 0.5, dtype=dtype, r=64, **SMALL)
    gx = synth.gate_inputs(spec.R, spec.G, 328, spec.r, spec.ew_std, seed=62, dtype=dtype,
                           device=DEV)
    x, k = run_gated(dsd, spec, gx, keep_all=keep_all)
    check_gated(spec, x, gx, k)


def test_gated_no_bias_at_first_and_silu(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=63, p_noise=1.0,
                        r=64, **SMALL)
    gx = synth.gate_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=64, device=DEV)
    x, k = run_gated(dsd, spec, gx, bias_at_first=False, act="silu")
    check_gated(spec, x, gx, k, bias_at_first=False, act="silu")
    assert np.all(k["gated_rep"][:, 0] == 0.0)


def test_zero_gate_is_the_plain_head_on_half_the_table(dsd):
    # W_g = 0 opens every gate half way: the gated head on E equals the plain
    # head on E / 2 (exact in bf16), token for token
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=65, p_noise=1.0,
                        r=64, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine="simt")
    h = torch.randn((spec.R, spec.G, 64), device=DEV).to(torch.bfloat16)
    Wg = torch.zeros((spec.r, 64 + spec.r), device=DEV, dtype=torch.bfloat16)
    a = ctx.propose_gated(x["U"], x["E"], x["W"], h, Wg, x["conf"], x["prev_tok"],
                          req_id=x["req_id"], temperature=1.0, seed=x["seed"])
    b = ctx.propose(x["U"], (x["E"].float() * 0.5).to(torch.bfloat16), x["W"], x["conf"],
                    x["prev_tok"], req_id=x["req_id"], temperature=1.0, seed=x["seed"])
    assert ctx.sync_status() == 0
    assert torch.equal(a["tokens"], b["tokens"])
    assert torch.allclose(a["lse_q"], b["lse_q"], atol=1e-5)
    ctx.close()


def test_gated_full_size_sampled_requests(dsd):
    # the greedy workload (R = 16, V = 151936, rank 256) with H = 2560
    spec = synth.CYCLE_SPECS["greedy"]
    gx = synth.gate_inputs(spec.R, spec.G, 2560, spec.r, spec.ew_std, seed=66, device=DEV)
    x, k = run_gated(dsd, spec, gx)
    idx = np.array([0, 5, 11, 15])
    h = host(x)
    gate = dict(h=synth.to_numpy(gx["h"])[idx], W_g=synth.to_numpy(gx["W_g"]))
    rid = h["req_id"].astype(np.int64)[idx]
    prop = O.propose(h["U"][idx], h["E"], h["W"], h["conf"][idx], h["prev_tok"][idx], rid, 0.0,
                     x["seed"], True, "none", gate)
    parity.compare_propose({n: k[n][idx] for n in ("tokens", "lse_q", "logit_at_tok",
                                                     "survival")}, prop)


def test_gated_errors(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=67, r=64, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    gx = synth.gate_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=68, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    with pytest.raises(dsd.DsdError):   # H not a multiple of 8
        ctx.propose_gated(x["U"], x["E"], x["W"], gx["h"][:, :, :60].contiguous(),
                          gx["W_g"][:, 4:].contiguous(), x["conf"], x["prev_tok"])
    h = gx["h"].clone()
    h[3, 2, 7] = float("nan")
    ctx.propose_gated(x["U"], x["E"], x["W"], h, gx["W_g"], x["conf"], x["prev_tok"])
    assert ctx.sync_status() == -6
    ctx.close()


@pytest.mark.parametrize("engine,R,temperature", [("simt", 19, 1.0), ("simt", 19, 0.0),
                                                  ("tcgen05", 100, 1.0), ("tcgen05", 64, 0.0)])
def test_gated_on_each_engine(dsd, engine, R, temperature):
    # the CUDA-core engine, and the tensor-core engine's split mode (hi and
    # lo bf16 parts of the fp32 representation, 64-request M-tiles: R = 100
    # takes two, one of them partial)
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=69 + R,
                        p_noise=1.0, r=128, R=R, V=2568, ew_std=0.3)
    gx = synth.gate_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=70, device=DEV)
    x, k = run_gated(dsd, spec, gx, engine=engine)
    check_gated(spec, x, gx, k)



def test_gated_in_launch_step_matches_the_step_kernels(dsd):
    # the tensor-core engine runs the gate inside its one-launch proposal;
    # the CUDA-core engine runs the standalone step kernel.  Both compute each
    # output with the same warp routine, so wherever the drafted prefix is the
    # same the representation is the same bit for bit.
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=75, p_noise=1.0,
                        r=128, R=40, V=2568, ew_std=0.3)
    gx = synth.gate_inputs(spec.R, spec.G, 96, spec.r, spec.ew_std, seed=76, device=DEV)
    _, kt = run_gated(dsd, spec, gx, engine="tcgen05")
    _, ks = run_gated(dsd, spec, gx, engine="simt")
    same = 0
    for q in range(spec.R):
        for j in range(spec.G):
            if np.array_equal(kt["tokens"][q, :j], ks["tokens"][q, :j]):
                same += 1
                assert np.array_equal(kt["gated_rep"][q, j].view(np.uint32),
                                      ks["gated_rep"][q, j].view(np.uint32)), (q, j)
    assert same >= 0.9 * spec.R * spec.G, same


@pytest.mark.parametrize("G", [1, 2])
def test_gated_short_blocks_on_the_tensor_cores(dsd, G):
    # gamma = 1: one launch per draft step with the standalone gate kernel
    # before it; gamma = 2: the one-launch proposal with its in-launch gate
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=77 + G, p_noise=1.0,
                        r=128, R=19, G=G, V=2568, ew_std=0.3)
    gx = synth.gate_inputs(spec.R, spec.G, 64, spec.r, spec.ew_std, seed=78, device=DEV)
    x, k = run_gated(dsd, spec, gx, engine="tcgen05")
    check_gated(spec, x, gx, k)
