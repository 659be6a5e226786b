"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the
same seeded inputs.  Small cases span several vocabulary tiles with a ragged
tail and request counts that are not multiples of the CTA batching; the
full-size workloads are checked on sampled requests / blocks."""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


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


def run_cycle(dsd, spec, engine="auto", act="none", bias_at_first=True, keep_all=False):
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, act=act,
                      bias_at_first=bias_at_first, engine=engine)
    T = spec.temperature
    prop = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], req_id=x["req_id"],
                       temperature=T, seed=x["seed"])
    sch = ctx.schedule(prop["survival"], x["sps"])
    keep = sch["keep_len"]
    if keep_all:
        keep = torch.full_like(keep, spec.G)
    ver = ctx.verify(x["P"], prop["tokens"], keep, U=x["U"], E=x["E"], W=x["W"],
                     prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                     logit_at_tok=prop["logit_at_tok"], req_id=x["req_id"], temperature=T,
                     seed=x["seed"])
    assert ctx.sync_status() == 0
    k = {n: t.cpu().numpy() for n, t in {**prop, **sch, **ver}.items()}
    k["keep_used"] = keep.cpu().numpy()
    ctx.close()
    return x, k


def oracle_cycle(spec, x, act="none", bias_at_first=True, keep_all=False):
    h = host(x)
    rid = h["req_id"].astype(np.int64)
    T = spec.temperature
    prop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"], rid, T, x["seed"],
                     bias_at_first, act)
    sch = O.schedule(prop["survival"].astype(np.float32), h["sps"])
    keep = np.full(spec.R, spec.G) if keep_all else sch["keep_len"]
    ver = O.verify(h["P"], h["U"], h["E"], h["W"], h["prev_tok"], prop["tokens"], keep, rid, T,
                   x["seed"], bias_at_first, act)
    return prop, sch, ver, keep


def check_cycle(spec, x, k, act="none", bias_at_first=True, keep_all=False, max_exempt=0.05):
    prop, sch, ver, keep = oracle_cycle(spec, x, act, bias_at_first, keep_all)
    rep = parity.compare_propose(k, prop)
    parity.compare_schedule(k["keep_len"], k["theta_B"], sch)
    ex = parity.draft_exempt(prop["margin"])
    draft_ex = np.array([ex[r, :keep[r] + 1].any() if keep[r] < spec.G else ex[r].any()
                         for r in range(spec.R)])
    if not draft_ex.any():
        assert np.array_equal(k["keep_used"], keep)
    vrep = parity.compare_verify(k["accept_len"], k["next_token"], ver, spec.temperature, keep,
                                 draft_ex)
    total = rep.checked + rep.exempt
    assert rep.exempt <= max_exempt * total + 1, f"too many exemptions: {rep}"
    return rep, vrep, ver


SMALL = dict(V=2568, R=19, ew_std=0.3)        # 21 tiles of 128 with an 8-row tail


@pytest.mark.parametrize("engine", ["simt", "auto"])
@pytest.mark.parametrize("temperature", [0.0, 1.0, 0.6])
def test_cycle_bf16_small(dsd, engine, temperature):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=21,
                        p_noise=1.0 if temperature else 0.5, **SMALL)
    x, k = run_cycle(dsd, spec, engine)
    check_cycle(spec, x, k)


@pytest.mark.parametrize("R,V,rank,temperature", [
    (129, 2568, 256, 0.0),     # second M-tile with one request, ragged vocabulary tail
    (256, 1032, 256, 1.0),     # two full M-tiles, sampled
    (300, 1544, 256, 0.0),     # three M-tiles
    (40, 3080, 128, 0.0),      # rank 128
    (16, 4104, 64, 1.0),       # rank 64, smallest batch AUTO sends to this engine
])
def test_cycle_mma_shapes(dsd, R, V, rank, temperature):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=R, V=V, r=rank, ew_std=0.3,
                        temperature=temperature, seed=100 + R, n_sps=None)
    x, k = run_cycle(dsd, spec, engine="mma")
    check_cycle(spec, x, k)


def test_mma_and_simt_engines_agree(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=64, V=2568, ew_std=0.3, seed=33)
    x = synth.cycle_inputs(spec, device=DEV)
    outs = []
    for engine in ("simt", "mma"):
        ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine=engine)
        o = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1)
        assert ctx.sync_status() == 0
        assert ctx.last_engine() == engine
        outs.append({n: t.cpu().numpy() for n, t in o.items()})
        ctx.close()
    h = host(x)
    prop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"],
                     h["req_id"].astype(np.int64), 0.0, 1)
    ok = ~parity.draft_exempt(prop["margin"])
    assert np.array_equal(outs[0]["tokens"][ok], outs[1]["tokens"][ok])
    assert np.max(np.abs(outs[0]["lse_q"] - outs[1]["lse_q"])[ok]) <= parity.LOGIT_TOL


@pytest.mark.parametrize("R,V,rank,temperature", [
    (129, 2568, 256, 0.0),     # CTA pair, second M-tile with one request, ragged vocabulary tail
    (256, 1032, 256, 1.0),     # CTA pair, two full M-tiles, sampled
    (256, 2600, 256, 0.0),     # CTA pair, last tile ends in a ragged second U box
    (200, 4104, 256, 1.0),     # CTA pair, partial second M-tile, sampled
    (140, 3080, 64, 0.0),      # CTA pair at rank 64 (one K-chunk per half-box stage)
    (450, 2568, 128, 1.0),     # four M-tiles: two CTA pairs per range, rank 128
    (512, 1032, 256, 0.0),     # four full M-tiles
    (300, 1544, 256, 0.0),     # three M-tiles: single CTAs (an odd count)
    (40, 3080, 128, 0.0),      # rank 128
    (16, 4104, 64, 1.0),       # rank 64
    (64, 2600, 256, 1.0),      # the largest batch whose rows 64..127 repeat rows 0..63
    (65, 1032, 256, 0.0),      # one request more: no repeated rows
])
def test_cycle_tc_shapes(dsd, R, V, rank, temperature):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=R, V=V, r=rank, ew_std=0.3,
                        temperature=temperature, seed=200 + R, n_sps=None)
    x, k = run_cycle(dsd, spec, engine="tcgen05")
    check_cycle(spec, x, k)


@pytest.mark.parametrize("R,G,temperature", [
    (256, 16, 0.0),    # CTA pairs, the largest gamma: every position counter of one launch
    (256, 2, 1.0),     # CTA pairs, one counter, sampled
    (256, 1, 0.0),     # one position: a single launch without counters
    (64, 16, 1.0),     # single CTAs with repeated rows, sampled
    (100, 16, 0.0),    # single CTAs, no repeated rows
    (1, 16, 0.0),      # one request
])
def test_cycle_tc_gamma_range(dsd, R, G, temperature):
    # all draft positions in one launch, the CTAs meeting at a counter per
    # position, from one position up to the largest gamma
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=R, G=G, V=1544, ew_std=0.3,
                        temperature=temperature, seed=400 + R + G, n_sps=None)
    x, k = run_cycle(dsd, spec, engine="tcgen05")
    check_cycle(spec, x, k)


@pytest.mark.parametrize("R,V,rank", [
    (19, 2568, 256),     # one 64-row block of the rejection list, ragged vocabulary tail
    (100, 1544, 128),    # two blocks, rank 128
    (200, 4104, 256),    # four blocks, the last partial
    (7, 1032, 64),       # a handful of rows, rank 64
])
def test_residual_pass_on_tensor_cores(dsd, R, V, rank):
    # every drafted position is verified (keep_len = gamma) at T = 1, so most
    # requests reject somewhere and take the residual draw of the tensor-core
    # residual pass; accept lengths and next tokens against the oracle
    spec = synth.scaled(synth.CYCLE_SPECS["sampled"], R=R, V=V, r=rank, ew_std=0.3,
                        seed=300 + R, n_sps=None)
    x, k = run_cycle(dsd, spec, engine="tcgen05", keep_all=True)
    check_cycle(spec, x, k, keep_all=True)
    assert (k["accept_len"] < spec.G).sum() >= max(1, R // 4)


def test_tc_mma_simt_engines_agree(dsd):
    """Tokens identical and lse within tolerance across the three engines at
    two full M-tiles, on rows whose top-2 margin is not a near tie."""
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=256, V=4104, ew_std=0.3, seed=35)
    x = synth.cycle_inputs(spec, device=DEV)
    outs = []
    for engine in ("simt", "mma", "tcgen05"):
        ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine=engine)
        o = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1)
        assert ctx.sync_status() == 0
        assert ctx.last_engine() == engine
        outs.append({n: t.cpu().numpy() for n, t in o.items()})
        ctx.close()
    h = host(x)
    prop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"],
                     h["req_id"].astype(np.int64), 0.0, 1)
    ok = ~parity.draft_exempt(prop["margin"])
    for o in outs[1:]:
        assert np.array_equal(outs[0]["tokens"][ok], o["tokens"][ok])
        assert np.max(np.abs(outs[0]["lse_q"] - o["lse_q"])[ok]) <= parity.LOGIT_TOL


def test_tc_engine_rejects_unsupported_config_before_any_launch(dsd):
    # rank 32: a valid context, but the tensor-core engine needs a multiple of 64
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=16, V=1032, r=32, seed=34)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine="tcgen05")
    n0 = ctx.launch_count()
    with pytest.raises(dsd.DsdError) as ei:
        ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1)
    assert ei.value.code == -9
    assert ctx.launch_count() == n0
    ctx.close()


def test_cycle_bf16_no_pruning_covers_all_positions(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["sampled"], seed=22, **SMALL)
    x, k = run_cycle(dsd, spec, keep_all=True)
    _, vrep, ver = check_cycle(spec, x, k, keep_all=True)
    assert vrep.checked > 0
    # every accept length 0..gamma is possible; some rejections happened
    assert (ver["accept_len"] < spec.G).any()


def test_cycle_f32_tiny_config(dsd):
    spec = synth.CYCLE_SPECS["tiny"]
    x, k = run_cycle(dsd, spec)
    check_cycle(spec, x, k)
    assert k["keep_len"].tolist() == [7]      # constant SPS over B <= 8 keeps all


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_cycle_f32_rank32_ragged(dsd, temperature):
    spec = synth.scaled(synth.CYCLE_SPECS["tiny"], R=5, V=1000, ew_std=0.5,
                        temperature=temperature, seed=23)
    x, k = run_cycle(dsd, spec)
    check_cycle(spec, x, k)


@pytest.mark.parametrize("act,baf", [("silu", True), ("none", False)])
def test_cycle_variants(dsd, act, baf):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=24, temperature=1.0, **SMALL)
    x, k = run_cycle(dsd, spec, act=act, bias_at_first=baf)
    check_cycle(spec, x, k, act=act, bias_at_first=baf)


@pytest.mark.parametrize("R,temperature,rank", [(19, 1.0, 256), (100, 0.0, 128), (130, 1.0, 64)])
def test_silu_on_the_tensor_core_split_mode(dsd, R, temperature, rank):
    # SiLU rows are not bf16: the tensor-core engine feeds their hi and lo
    # bf16 parts (64-request M-tiles: R = 130 takes three)
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=26 + R, temperature=temperature, R=R,
                        V=2568, ew_std=0.3, r=rank)
    x, k = run_cycle(dsd, spec, engine="tcgen05", act="silu")
    check_cycle(spec, x, k, act="silu")


def test_single_position_and_single_request(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=1, G=1, V=1032, ew_std=0.5, seed=25)
    x, k = run_cycle(dsd, spec)
    check_cycle(spec, x, k)


def test_propose_is_deterministic_and_keyed_by_request_id(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["sampled"], seed=26, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    a = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 1.0, 7)
    b = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 1.0, 7)
    assert torch.equal(a["tokens"], b["tokens"]) and torch.equal(a["lse_q"], b["lse_q"])
    perm = torch.randperm(spec.R, generator=torch.Generator().manual_seed(0)).to(DEV)
    c = ctx.propose(x["U"][perm].contiguous(), x["E"], x["W"], x["conf"][perm].contiguous(),
                    x["prev_tok"][perm].contiguous(), x["req_id"][perm].contiguous(), 1.0, 7)
    assert torch.equal(c["tokens"], a["tokens"][perm])
    assert ctx.sync_status() == 0
    ctx.close()


def test_schedule_against_oracle_random_tables(dsd):
    rng = np.random.default_rng(27)
    ctx = dsd.Context(4096, 64, 7, 300, dtype="bf16")
    for trial in range(12):
        R = int(rng.integers(1, 300))
        conf = rng.beta(rng.uniform(1, 10), 2, size=(R, 7)).astype(np.float32)
        if trial % 3 == 0:
            conf[:, 2:] = 1.0                 # equal survivals within a request
        if trial % 4 == 1:
            conf = np.round(conf * 4) / 4     # many exact ties across requests
        n = int(rng.integers(R, R * 8 + 2))
        B = np.arange(1, n + 1)
        knee = rng.uniform(0, n)
        sps = (1.0 / (1e-3 + rng.uniform(1e-6, 1e-4) * np.maximum(0, B - knee))).astype(np.float32)
        surv = O.survival(conf).astype(np.float32)
        out = ctx.schedule(torch.as_tensor(surv, device=DEV), torch.as_tensor(sps, device=DEV))
        ref = O.schedule(surv, sps)
        parity.compare_schedule(out["keep_len"].cpu().numpy(), out["theta_B"].cpu().numpy(), ref)
    with pytest.raises(dsd.DsdError):
        ctx.schedule(torch.ones((10, 7), device=DEV), torch.ones(5, device=DEV))
    assert ctx.sync_status() == 0
    ctx.close()


def test_schedule_unsorted_clamped_and_maximum_size(dsd):
    # any survival table: runs that are not sorted, values outside [0, 1]
    # (clamped on both sides), exact ties, and the largest table R * gamma =
    # 4096 the scheduler holds
    rng = np.random.default_rng(29)
    for R, G in ((512, 8), (37, 5), (1, 16), (585, 7)):
        ctx = dsd.Context(4096, 64, G, R, dtype="bf16")
        for trial in range(3):
            surv = rng.uniform(-0.2, 1.2, size=(R, G)).astype(np.float32)
            if trial == 1:
                surv = np.round(surv * 8) / 8            # many exact ties
            if trial == 2:
                surv = np.sort(surv, axis=1)             # ascending runs
            n = R * (G + 1)
            B = np.arange(1, n + 1)
            sps = (1.0 / (1e-3 + rng.uniform(1e-6, 1e-4) * np.maximum(0, B - rng.uniform(0, n)))
                   ).astype(np.float32)
            out = ctx.schedule(torch.as_tensor(surv, device=DEV), torch.as_tensor(sps, device=DEV))
            ref = O.schedule(surv, sps)
            parity.compare_schedule(out["keep_len"].cpu().numpy(), out["theta_B"].cpu().numpy(),
                                    ref)
        assert ctx.sync_status() == 0
        bad = torch.full((R, G), 0.5, device=DEV)
        bad[0, 0] = float("nan")
        ctx.schedule(bad, torch.ones(R * (G + 1), device=DEV))
        assert ctx.sync_status() == -6
        ctx.close()


def test_repeated_verify_calls_on_one_context(dsd):
    # the per-request item counters return to zero after every call: the
    # same context verifies several keep patterns in a row
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=1.0, seed=31, p_noise=1.0,
                        r=64, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype)
    prop = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], req_id=x["req_id"],
                       temperature=1.0, seed=x["seed"])
    h = host(x)
    rid = h["req_id"].astype(np.int64)
    oprop = O.propose(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"], rid, 1.0, x["seed"])
    parity.compare_propose({n: t.cpu().numpy() for n, t in prop.items()}, oprop)
    ex = parity.draft_exempt(oprop["margin"])
    rng = np.random.default_rng(32)
    for trial in range(4):
        for T in (1.0, 0.0):
            keep = rng.integers(0, spec.G + 1, size=spec.R).astype(np.int32)
            if trial == 0:
                keep[:] = spec.G
            ver = ctx.verify(x["P"], prop["tokens"], torch.as_tensor(keep, device=DEV), U=x["U"],
                             E=x["E"], W=x["W"], prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                             logit_at_tok=prop["logit_at_tok"], req_id=x["req_id"],
                             temperature=T, seed=x["seed"])
            # T = 0: greedy verification of the sampled proposal (only the
            # argmax of each target row decides)
            over = O.verify(h["P"], h["U"], h["E"], h["W"], h["prev_tok"], oprop["tokens"], keep,
                            rid, T, x["seed"])
            draft_ex = np.array([ex[r, :keep[r] + 1].any() if keep[r] < spec.G else ex[r].any()
                                 for r in range(spec.R)])
            parity.compare_verify(ver["accept_len"].cpu().numpy(), ver["next_token"].cpu().numpy(),
                                  over, T, keep, draft_ex)
    assert ctx.sync_status() == 0
    ctx.close()


def test_verify_greedy_hand_case(dsd):
    P = torch.zeros((1, 4, 8), dtype=torch.float32)
    P[0, 0, 0] = 5
    P[0, 1, 3] = 4
    P[0, 2, 1] = 6
    P[0, 3, 3] = 9
    ctx = dsd.Context(8, 8, 3, 1, dtype="f32")
    tokens = torch.tensor([[0, 3, 2]], dtype=torch.int32, device=DEV)
    for kl, acc, nxt in [(3, 2, 1), (2, 2, 1), (1, 1, 3), (0, 0, 0)]:
        out = ctx.verify(P.to(DEV), tokens, torch.tensor([kl], dtype=torch.int32, device=DEV))
        assert (int(out["accept_len"][0]), int(out["next_token"][0])) == (acc, nxt)
    assert ctx.sync_status() == 0
    ctx.close()


# (9, 2568) and (3, 1000): ragged last slices of the eight-CTA split;
# (64, 2568): many clusters resident per SM; (2, 240000): a large vocabulary
# (60 KB slices).
@pytest.mark.parametrize("N,V", [(9, 2568), (3, 1000), (64, 2568), (2, 240000)])
def test_overlap_small(dsd, N, V):
    spec = synth.OverlapSpec(N=N, V=V, ragged_frac=0.5, seed=28)
    ox = synth.overlap_inputs(spec, device=DEV)
    ox["valid_len"][0] = 0
    ctx = dsd.Context(V, 64, spec.G, 8, dtype="bf16")
    out = ctx.overlap(ox["P"], ox["Q"], ox["valid_len"])
    assert ctx.sync_status() == 0
    ref = O.overlap(synth.to_numpy(ox["P"]), synth.to_numpy(ox["Q"]), synth.to_numpy(ox["valid_len"]))
    parity.compare_overlap({k: v.cpu().numpy() for k, v in out.items()}, ref)
    # empty call
    e = ctx.overlap(ox["P"][:0], ox["Q"][:0], ox["valid_len"][:0])
    assert float(e["mean_tau"][0]) == 0.0 and torch.all(e["accept_rate"] == 0)
    ctx.close()


def test_overlap_masked_and_nonfinite(dsd):
    """-inf logits (a masked vocabulary range) are zero-probability entries;
    a NaN logit on a valid position is reported as non-finite."""
    spec = synth.OverlapSpec(N=5, V=2568, ragged_frac=0.0, seed=31)
    ox = synth.overlap_inputs(spec, device=DEV)
    P, Q = ox["P"].clone(), ox["Q"].clone()
    P[0, 0, :700] = float("-inf")          # whole 16-byte chunks of several threads
    Q[0, 0, 1000:1800] = float("-inf")
    P[1, 2, ::3] = float("-inf")
    Q[1, 2, 1::3] = float("-inf")
    ctx = dsd.Context(spec.V, 64, spec.G, 8, dtype="bf16")
    out = ctx.overlap(P, Q, ox["valid_len"])
    assert ctx.sync_status() == 0
    ref = O.overlap(synth.to_numpy(P), synth.to_numpy(Q), synth.to_numpy(ox["valid_len"]))
    parity.compare_overlap({k: v.cpu().numpy() for k, v in out.items()}, ref)
    P[2, 1, 17] = float("nan")
    ctx.overlap(P, Q, ox["valid_len"])
    assert ctx.sync_status() == -6
    ctx.close()


def test_nonfinite_logits_are_reported(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=29, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    x["U"][3, 2, 100] = float("nan")
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1)
    assert ctx.sync_status() == -6
    assert ctx.sync_status() == 0           # status is cleared after reading
    ctx.close()


def test_empty_batch_is_a_noop(dsd):
    ctx = dsd.Context(1032, 64, 7, 4, dtype="bf16")
    z = torch.empty((0, 7, 1032), dtype=torch.bfloat16, device=DEV)
    e = torch.zeros((1032, 64), dtype=torch.bfloat16, device=DEV)
    out = ctx.propose(z, e, e, torch.empty((0, 7), device=DEV),
                      torch.empty((0,), dtype=torch.int32, device=DEV))
    assert out["tokens"].numel() == 0
    assert ctx.sync_status() == 0
    ctx.close()


# ----------------------------------------------------------- full-size checks

def _subset(x, idx):
    return {k: (v[idx].contiguous() if isinstance(v, torch.Tensor) and k in
                ("U", "P", "conf", "prev_tok", "req_id") else v) for k, v in x.items()}


@pytest.mark.parametrize("name,n_sample", [("greedy", 16), ("sampled", 6), ("highconc", 6)])
def test_full_size_cycle_sampled_requests(dsd, name, n_sample):
    spec = synth.CYCLE_SPECS[name]
    x, k = run_cycle(dsd, spec)
    rng = np.random.default_rng(30)
    idx = np.sort(rng.choice(spec.R, size=n_sample, replace=False))
    h = host(x)
    rid = h["req_id"].astype(np.int64)
    T = spec.temperature
    # schedule over the whole batch needs only the (cheap) survivals
    surv = O.survival(h["conf"]).astype(np.float32)
    sch = O.schedule(surv, h["sps"])
    parity.compare_schedule(k["keep_len"], k["theta_B"], sch)
    hs = {n: v[idx] for n, v in h.items() if n in ("U", "P", "conf", "prev_tok")}
    prop = O.propose(hs["U"], h["E"], h["W"], hs["conf"], hs["prev_tok"], rid[idx], T, x["seed"])
    kk = {n: k[n][idx] for n in ("tokens", "lse_q", "logit_at_tok", "survival")}
    parity.compare_propose(kk, prop)
    keep = sch["keep_len"][idx]
    ver = O.verify(hs["P"], hs["U"], h["E"], h["W"], hs["prev_tok"], prop["tokens"], keep,
                   rid[idx], T, x["seed"])
    ex = parity.draft_exempt(prop["margin"])
    draft_ex = np.array([ex[i, :min(keep[i] + 1, spec.G)].any() for i in range(len(idx))])
    parity.compare_verify(k["accept_len"][idx], k["next_token"][idx], ver, T, keep, draft_ex)


def test_full_size_overlap_sampled_blocks(dsd):
    spec = synth.OverlapSpec()
    ox = synth.overlap_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, 64, spec.G, 8, dtype="bf16")
    out = ctx.overlap(ox["P"], ox["Q"], ox["valid_len"])
    assert ctx.sync_status() == 0
    rng = np.random.default_rng(31)
    vl = synth.to_numpy(ox["valid_len"])
    ragged = np.flatnonzero(vl < spec.G)
    idx = np.sort(np.concatenate([rng.choice(spec.N, 10, replace=False), ragged[:4]]))
    ref = O.overlap(synth.to_numpy(ox["P"][idx]), synth.to_numpy(ox["Q"][idx]), vl[idx])
    a_k = out["a"].cpu().numpy()[idx]
    assert np.max(np.abs(a_k - ref["a"])) <= parity.PROB_TOL
    assert np.max(np.abs(out["tau"].cpu().numpy()[idx] - ref["tau"])) <= parity.PROB_TOL
    # aggregates over all blocks from the kernel's own per-block values
    a_all = out["a"].cpu().numpy().astype(np.float64)
    vmask = np.arange(spec.G)[None, :] < vl[:, None]
    ar = (a_all * vmask).sum(0) / np.maximum(vmask.sum(0), 1)
    assert np.max(np.abs(out["accept_rate"].cpu().numpy() - ar)) <= 1e-5
    ctx.close()


@pytest.mark.parametrize("R,dtype,act,expect", [
    (16, "bf16", "none", "tcgen05"),
    (15, "bf16", "none", "tcgen05"),
    (1, "bf16", "none", "tcgen05"),
    (64, "f32", "none", "simt"),
    (64, "bf16", "silu", "tcgen05"),
])
def test_auto_engine_choice(dsd, R, dtype, act, expect):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=R, V=1032, seed=36, dtype=dtype)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=dtype, act=act, engine="auto")
    ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1)
    assert ctx.sync_status() == 0
    assert ctx.last_engine() == expect
    ctx.close()


@pytest.mark.parametrize("temperature", [0.0, 1.0])
def test_cycle_host_matches_the_device_cycle(dsd, temperature):
    """dsd_cycle_host from host buffers gives the device cycle's results: with
    pinned P (read in place over the CPU-GPU link) and with pageable P
    (staged on the device)."""
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=33,
                        p_noise=1.0 if temperature else 0.5, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    dev = ctx.cycle(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["P"], x["sps"],
                    req_id=x["req_id"], temperature=temperature, seed=x["seed"])
    host = {k: x[k].cpu() for k in ("U", "conf", "prev_tok", "req_id", "P")}
    for pinned in (True, False):
        h = {k: (v.pin_memory() if pinned else v) for k, v in host.items()}
        if not pinned:
            h["U"] = h["U"].pin_memory()
        out = ctx.cycle_host(h["U"], x["E"], x["W"], h["conf"], h["prev_tok"], h["P"], x["sps"],
                             req_id_host=h["req_id"], temperature=temperature, seed=x["seed"])
        assert ctx.sync_status() == 0
        assert ctx.last_p_in_place() == pinned
        for k in ("tokens", "keep_len", "accept_len", "next_token"):
            assert torch.equal(out[k], dev[k].cpu()), (pinned, k)
    ctx.close()


@pytest.mark.parametrize("name,temperature", [("small", 0.0), ("small", 1.0), ("highconc", 0.0),
                                              ("greedy", 0.0)])
def test_cycle_call_matches_the_three_calls(dsd, name, temperature):
    """dsd_cycle computes the schedule inside the proposal's last launch, from
    the confidences; its outputs equal dsd_propose -> dsd_schedule ->
    dsd_verify on the same inputs, bit for bit, and the schedule equals the
    oracle's on the survivals (the whole batch)."""
    if name == "small":
        spec = synth.scaled(synth.CYCLE_SPECS["greedy"], temperature=temperature, seed=35,
                            p_noise=1.0 if temperature else 0.5, **SMALL)
    else:
        spec = synth.CYCLE_SPECS[name]
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype)
    kw = dict(req_id=x["req_id"], temperature=temperature, seed=x["seed"])
    one = ctx.cycle(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["P"], x["sps"], **kw)
    one = {k: v.clone() for k, v in one.items()}
    prop = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], **kw)
    sch = ctx.schedule(prop["survival"], x["sps"])
    ver = ctx.verify(x["P"], prop["tokens"], sch["keep_len"], U=x["U"], E=x["E"], W=x["W"],
                     prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                     logit_at_tok=prop["logit_at_tok"], **kw)
    assert ctx.sync_status() == 0
    three = {**prop, **sch, **ver}
    for k in ("tokens", "lse_q", "logit_at_tok", "survival", "keep_len", "theta_B", "accept_len",
              "next_token"):
        assert torch.equal(one[k], three[k]), k
    ref = O.schedule(one["survival"].cpu().numpy(), synth.to_numpy(x["sps"]))
    parity.compare_schedule(one["keep_len"].cpu().numpy(), one["theta_B"].cpu().numpy(), ref)
    ctx.close()


def test_cycle_rejects_bad_arguments_before_any_launch(dsd):
    # an argument error of the verification half is found before the
    # proposal launches anything
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], seed=37, **SMALL)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16")
    out = ctx.cycle_outputs(spec.R)
    n0 = ctx.launch_count()
    for P, acc in ((None, out["accept_len"]), (x["P"], None)):
        with pytest.raises(dsd.DsdError):
            dsd.dsd_cycle(ctx.handle, spec.R, x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                          x["req_id"], P, x["sps"], x["sps"].numel(), 0.0, 1, out["tokens"],
                          out["lse_q"], out["logit_at_tok"], out["survival"], out["keep_len"],
                          out["theta_B"], acc, out["next_token"], None, 0)
    assert ctx.launch_count() == n0
    assert ctx.sync_status() == 0
    ctx.close()
