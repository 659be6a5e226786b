"""dsd_confidence_head, dsd_threshold_keep and dsd_calibration against the
oracle, element by element, through the C ABI.

Tolerances, from the arithmetic: the head's logits are fp32 sums of at most
a few thousand exact bf16 products (relative rounding ~1e-6 of |s| <= ~5),
so conf = sigmoid(s) and the survival products agree to ~1e-6; the tests
allow 1e-4 absolute.  Threshold decisions compare the same fp32 values on
both sides, so keep lengths are bit-exact.  Calibration: both sides form the
survival as an fp64 product of the same fp32 inputs (identical bits), so
the bin counts are bit-exact and the fp64 sums agree to ~1e-12; outputs are
fp32 (1e-6 allowed).
"""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
TOL = 1e-4
CAL_TOL = 1e-6


@pytest.fixture(scope="module")
def dsd():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from semi_autoregressive_draft_gb300 import build as b

    b.build()
    import semi_autoregressive_draft_gb300 as m

    return m


def _head_case(dsd, R, G, H, V, r, dtype, seed):
    x = synth.confidence_inputs(R, G, H, V, r, seed=seed, dtype=dtype, device=DEV)
    ctx = dsd.Context(V, r, G, max(R, 1), dtype=dtype)
    out = ctx.confidence_head(x["h"], x["E"], x["w_c"], x["b_c"], x["prev_tok"], x["tokens"])
    assert ctx.sync_status() == 0
    ref = O.confidence_head(synth.to_numpy(x["h"]), synth.to_numpy(x["E"]),
                            synth.to_numpy(x["w_c"]), x["b_c"], synth.to_numpy(x["prev_tok"]),
                            synth.to_numpy(x["tokens"]))
    assert np.max(np.abs(out["conf"].cpu().numpy() - ref["conf"])) <= TOL
    assert np.max(np.abs(out["survival"].cpu().numpy() - ref["survival"])) <= TOL
    return ctx, x


# H = 328: 41 sixteen-byte chunks over a warp's 32 lanes (a ragged tail);
# rank 64 and 8; f32 and bf16; R = 19 and 1; gamma 7, 1 and 16.
@pytest.mark.parametrize("R,G,H,V,r,dtype", [(19, 7, 328, 2568, 64, "bf16"),
                                             (19, 7, 328, 2568, 64, "f32"),
                                             (1, 1, 8, 64, 8, "bf16"),
                                             (5, 16, 2560, 1032, 64, "bf16")])
def test_confidence_head_small(dsd, R, G, H, V, r, dtype):
    ctx, _ = _head_case(dsd, R, G, H, V, r, dtype, seed=40 + R + G)
    ctx.close()


def test_confidence_head_full_size(dsd):
    # the high-concurrency batch: R = 256, gamma = 7, H = 2560, V = 151936, rank 256
    ctx, _ = _head_case(dsd, 256, 7, 2560, 151936, 256, "bf16", seed=47)
    ctx.close()


def test_confidence_head_feeds_the_scheduler(dsd):
    # survival from the head is the scheduler's input: same allocation as the
    # oracle's schedule of the oracle's survival (outside survival ties)
    R, G, V, r = 32, 7, 2568, 64
    ctx, x = _head_case(dsd, R, G, 328, V, r, "bf16", seed=48)
    out = ctx.confidence_head(x["h"], x["E"], x["w_c"], x["b_c"], x["prev_tok"], x["tokens"])
    sps = torch.tensor(1.0 / (1e-3 + 2e-5 * np.maximum(0, np.arange(1, R * (G + 1) + 1) - 16)),
                       dtype=torch.float32, device=DEV)
    sch = ctx.schedule(out["survival"], sps)
    ref = O.schedule(out["survival"].cpu().numpy(), sps.cpu().numpy())
    assert np.array_equal(sch["keep_len"].cpu().numpy(), ref["keep_len"])
    ctx.close()


def test_confidence_head_errors(dsd):
    R, G, H, V, r = 4, 7, 64, 1032, 64
    x = synth.confidence_inputs(R, G, H, V, r, seed=49, device=DEV)
    ctx = dsd.Context(V, r, G, R, dtype="bf16")
    bad = x["tokens"].clone()
    bad[1, 3] = V
    ctx.confidence_head(x["h"], x["E"], x["w_c"], x["b_c"], x["prev_tok"], bad)
    assert ctx.sync_status() == -1
    h = x["h"].clone()
    h[2, 0, 5] = float("nan")
    ctx.confidence_head(h, x["E"], x["w_c"], x["b_c"], x["prev_tok"], x["tokens"])
    assert ctx.sync_status() == -6
    with pytest.raises(dsd.DsdError):       # H not a multiple of 8
        ctx.confidence_head(x["h"][:, :, :60].contiguous(), x["E"], x["w_c"][:60 + r].contiguous(),
                            x["b_c"], x["prev_tok"], x["tokens"])
    ctx.close()


def test_threshold_keep_matches_the_oracle(dsd):
    R, G = 300, 7
    c = synth.calibration_inputs(R, G, seed=50, device=DEV)["conf"]
    c[5, 2] = float("nan")
    c[6, :] = 0.7                             # ties with the threshold are kept
    ctx = dsd.Context(1032, 64, G, 8, dtype="bf16")
    for thr in (0.0, 0.5, 0.7, 0.9, 1.01):
        k = ctx.threshold_keep(c, thr)
        assert np.array_equal(k.cpu().numpy(), O.threshold_keep(c.cpu().numpy(), thr)), thr
    assert ctx.sync_status() == 0
    assert ctx.threshold_keep(c[:0], 0.5).numel() == 0
    ctx.close()


def _cal_compare(out, ref):
    b = out["bins"].cpu().numpy()
    assert np.array_equal(b[0].astype(np.int64), ref["count"])
    assert np.max(np.abs(b[1] - ref["mean_pred"])) <= CAL_TOL
    assert np.max(np.abs(b[2] - ref["mean_real"])) <= CAL_TOL
    pos = out["pos"].cpu().numpy()
    assert np.max(np.abs(pos[0] - ref["pos_pred"])) <= CAL_TOL
    assert np.max(np.abs(pos[1] - ref["pos_real"])) <= CAL_TOL
    m = out["metrics"].cpu().numpy()
    assert abs(m[0] - ref["ece"]) <= CAL_TOL
    assert abs(m[1] - ref["abs_error"]) <= CAL_TOL
    assert abs(m[2] - ref["cumprod_bias"]) <= CAL_TOL
    assert int(m[3]) == ref["n_tested"]


@pytest.mark.parametrize("M,n_bins", [(5000, 10), (70001, 64), (3, 1)])
def test_calibration_matches_the_oracle(dsd, M, n_bins):
    G = 7
    x = synth.calibration_inputs(M, G, seed=51 + n_bins, device=DEV)
    ctx = dsd.Context(1032, 64, G, 8, dtype="bf16")
    ref = O.calibration(x["conf"].cpu().numpy(), x["accept_len"].cpu().numpy(), n_bins)
    for _ in range(2):                        # the workspace sums reset between calls
        out = ctx.calibration(x["conf"], x["accept_len"], n_bins)
        assert ctx.sync_status() == 0
        _cal_compare(out, ref)
    ctx.close()


def test_calibration_page_example_and_edges(dsd):
    # the paper-reading page's example: 0.85 per step against a true 0.80
    G = 6
    L = []
    for k in range(G + 1):
        ge = 5 ** (G - k) * 4 ** k
        gt = 5 ** (G - k - 1) * 4 ** (k + 1) if k < G else 0
        L += [k] * (ge - gt)
    acc = torch.tensor(L, dtype=torch.int32, device=DEV)
    conf = torch.full((len(L), G), 0.85, dtype=torch.float32, device=DEV)
    ctx = dsd.Context(1032, 64, G, 8, dtype="bf16")
    out = ctx.calibration(conf, acc, 10)
    assert ctx.sync_status() == 0
    _cal_compare(out, O.calibration(conf.cpu().numpy(), L, 10))
    pos = out["pos"].cpu().numpy()
    assert abs(pos[0, G - 1] - 0.85 ** 6) < 1e-6 and abs(pos[1, G - 1] - 0.8 ** 6) < 1e-6
    # empty call writes zeros; an out-of-range accept length is reported
    e = ctx.calibration(conf[:0], acc[:0], 10)
    assert float(e["metrics"].abs().sum()) == 0.0 and float(e["bins"].abs().sum()) == 0.0
    bad = acc.clone()
    bad[0] = G + 1
    ctx.calibration(conf, bad, 10)
    assert ctx.sync_status() == -1
    ctx.close()


# ---------------------------------------------------------------------- AUROC
# Both sides form the survivals as the same fp64 products of the same fp32
# confidences and count pairs exactly (integers); only the final division is
# floating point, so the results agree to fp64 rounding.
AUC_TOL = 1e-12


@pytest.mark.parametrize("M,G,seed", [(1, 7, 60), (200, 7, 61), (5000, 7, 62), (40000, 7, 63),
                                      (37, 1, 64), (1500, 16, 65)])
def test_auroc_matches_the_oracle(dsd, M, G, seed):
    # n = M G from 7 (one tile) through 280,000 (a 2^19-key bitonic network)
    x = synth.calibration_inputs(M, G, seed=seed, device=DEV)
    ctx = dsd.Context(1024, 64, G, 4, dtype="f32")
    got = float(ctx.auroc(x["conf"], x["accept_len"]).cpu()[0])
    assert ctx.sync_status() == 0
    ref = O.auroc(x["conf"].cpu().numpy(), x["accept_len"].cpu().numpy())
    assert abs(got - ref) <= AUC_TOL, (got, ref)
    ctx.close()


def test_auroc_ties_edges_and_scratch(dsd):
    rng = np.random.default_rng(66)
    G = 5
    ctx = dsd.Context(1024, 64, G, 4, dtype="f32")
    # confidences from a few values: many equal survivals across requests
    conf = torch.as_tensor(rng.choice([0.5, 0.8, 1.0], size=(3000, G)).astype(np.float32),
                           device=DEV)
    L = torch.as_tensor(rng.integers(0, G + 1, size=3000).astype(np.int32), device=DEV)
    got = float(ctx.auroc(conf, L).cpu()[0])
    assert abs(got - O.auroc(conf.cpu().numpy(), L.cpu().numpy())) <= AUC_TOL
    # one class only: one half
    full = torch.full((50,), G, dtype=torch.int32, device=DEV)
    assert float(ctx.auroc(conf[:50], full).cpu()[0]) == 0.5
    # a caller-owned scratch reused across calls, then one that is too small
    need = dsd.dsd_auroc_scratch_bytes(3000, G)
    scratch = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = torch.empty(1, dtype=torch.float64, device=DEV)
    for _ in range(2):
        dsd.dsd_auroc(ctx.handle, 3000, conf, L, scratch, out)
        assert float(out.cpu()[0]) == got
    with pytest.raises(dsd.DsdError) as ei:
        dsd.dsd_auroc(ctx.handle, 3000, conf, L, scratch[: need - 256], out)
    assert ei.value.code == -4
    assert ctx.sync_status() == 0
    ctx.close()
