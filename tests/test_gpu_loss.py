"""dsd_loss_forward (two tcgen05 passes and an fp64 finalize) against the
oracle's loss_forward, element by element, through the C ABI.

Tolerances, from the arithmetic: the kernel's biased logits are fp32 sums of
exact bf16 products (relative rounding ~1e-7 of |l| <= ~30), its
exponentials are ex2.approx (relative error ~2^-22) and its per-range sums
are fp32 over at most a few thousand terms each, merged in fp64.  That
bounds |CE| and |L1| errors by a few 1e-5; the tests allow 1e-4 absolute.
"""

import numpy as np
import pytest
import torch

from oracle import dsd_oracle as O
from semi_autoregressive_draft_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
ROW_TOL = 1e-4       # l1, accept, ce, bce per row (absolute)
LOSS_RTOL = 2e-5     # the four batch losses (relative, + ROW_TOL absolute)


@pytest.fixture(scope="module")
def dsd():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from semi_autoregressive_draft_gb300 import build as b

    b.build()
    import semi_autoregressive_draft_gb300 as m

    return m


def host(x):
    return {k: synth.to_numpy(v) for k, v in x.items()}


def oracle_of(h, baf=True, blocks=None, **kw):
    sel = (lambda a: a) if blocks is None else (lambda a: a[blocks])
    return O.loss_forward(sel(h["U"]), h["E"], h["W"], sel(h["prev_tok"]), sel(h["P"]),
                          sel(h["target"]), sel(h["conf_logit"]), bias_at_first=baf, **kw)


def compare_rows(row, ref, rows=None):
    """row: kernel [4, n] (l1, accept, ce, bce); ref: oracle dict; rows: the
    kernel rows that ref covers (default all)."""
    names = ("l1", "accept", "ce", "bce")
    for i, nm in enumerate(names):
        k = row[i] if rows is None else row[i][rows]
        o = ref[nm].reshape(-1)
        err = np.max(np.abs(k.astype(np.float64) - o))
        assert err <= ROW_TOL, f"{nm}: max abs error {err}"


def compare_losses(losses, ref):
    for i, nm in enumerate(("ce_loss", "l1_loss", "conf_loss", "loss")):
        k, o = float(losses[i]), float(ref[nm])
        assert abs(k - o) <= ROW_TOL + LOSS_RTOL * abs(o), f"{nm}: {k} vs {o}"


def run(dsd, spec, baf=True, R_max=None, **kw):
    x = synth.loss_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, R_max or spec.B, dtype="bf16", bias_at_first=baf)
    out = ctx.loss_forward(x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"],
                           x["conf_logit"], **kw)
    st = ctx.sync_status()
    return ctx, x, out, st


# Shapes: one, two, three and eight M-tiles (the CTAs of one vocabulary
# range read W at about the same time); ranks 64..256 including an odd
# number of 64-wide K-chunks; vocabularies whose last tile is ragged in
# either column half; gamma 1, 4, 7, 16; both readings of position 0.
@pytest.mark.parametrize("B,G,V,r,baf", [
    (9, 7, 2568, 64, True),
    (30, 7, 2600, 256, True),
    (40, 7, 4104, 128, False),
    (37, 4, 1032, 256, True),
    (64, 16, 8200, 192, True),
    (1, 1, 1000, 64, True),
    (23, 7, 3000, 256, False),
])
def test_loss_small_shapes(dsd, B, G, V, r, baf):
    spec = synth.LossSpec(B=B, G=G, V=V, r=r, ew_std=0.2, seed=40 + B)
    ctx, x, out, st = run(dsd, spec, baf)
    assert st == 0
    ref = oracle_of(host(x), baf)
    compare_rows(out["row"].cpu().numpy(), ref)
    compare_losses(out["losses"].cpu().numpy(), ref)
    ctx.close()


def test_loss_maximum_rows(dsd):
    # R_max * gamma = 4096 rows: 32 M-tiles, the largest grid of the kernel
    spec = synth.LossSpec(B=512, G=8, V=2048, r=64, ew_std=0.2, seed=47)
    ctx, x, out, st = run(dsd, spec)
    assert st == 0
    ref = oracle_of(host(x))
    compare_rows(out["row"].cpu().numpy(), ref)
    compare_losses(out["losses"].cpu().numpy(), ref)
    ctx.close()


def test_loss_weights_and_decay_are_arguments(dsd):
    spec = synth.LossSpec(B=12, V=2056, r=128, ew_std=0.2, seed=48)
    kw = dict(ce_alpha=0.3, l1_alpha=0.25, conf_alpha=2.0, decay=1.5)
    ctx, x, out, st = run(dsd, spec, **kw)
    assert st == 0
    ref = oracle_of(host(x), **kw)
    compare_losses(out["losses"].cpu().numpy(), ref)
    ctx.close()


def test_loss_is_deterministic_and_launches_three_kernels(dsd):
    spec = synth.LossSpec(B=30, V=2600, r=256, ew_std=0.2, seed=49)
    ctx, x, out, st = run(dsd, spec)
    n0 = ctx.launch_count()
    again = ctx.loss_forward(x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"],
                             x["conf_logit"])
    assert ctx.sync_status() == 0
    assert ctx.launch_count() - n0 == 3
    assert torch.equal(out["row"], again["row"]) and torch.equal(out["losses"], again["losses"])
    ctx.close()


def test_loss_without_row_output_and_empty_batch(dsd):
    spec = synth.LossSpec(B=5, V=1032, r=64, ew_std=0.2, seed=50)
    ctx, x, out, st = run(dsd, spec, rows=False)
    assert st == 0 and out["row"] is None
    compare_losses(out["losses"].cpu().numpy(), oracle_of(host(x)))
    z = {k: v[:0] for k, v in x.items() if k not in ("E", "W")}
    e = ctx.loss_forward(z["U"], x["E"], x["W"], z["prev_tok"], z["P"], z["target"],
                         z["conf_logit"])
    assert ctx.sync_status() == 0
    assert torch.all(e["losses"] == 0)
    ctx.close()


def test_loss_bad_tokens_and_nonfinite_logits_are_reported(dsd):
    spec = synth.LossSpec(B=4, V=1032, r=64, ew_std=0.2, seed=51)
    x = synth.loss_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.B, dtype="bf16")
    args = lambda x: (x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"], x["conf_logit"])
    y = dict(x, target=x["target"].clone())
    y["target"][1, 3] = spec.V
    out = ctx.loss_forward(*args(y))
    assert ctx.sync_status() == -1
    assert torch.isnan(out["row"][2, 1 * spec.G + 3])
    y = dict(x, prev_tok=x["prev_tok"].clone())
    y["prev_tok"][0, 0] = -5
    ctx.loss_forward(*args(y))
    assert ctx.sync_status() == -1
    y = dict(x, U=x["U"].clone())
    y["U"][2, 6, 17] = float("nan")
    ctx.loss_forward(*args(y))
    assert ctx.sync_status() == -6
    assert ctx.sync_status() == 0
    ctx.close()


def test_loss_rejects_unsupported_configurations_before_any_launch(dsd):
    spec = synth.LossSpec(B=2, V=1032, r=64, seed=52)
    x = synth.loss_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.B, dtype="bf16", act="silu")
    n0 = ctx.launch_count()
    with pytest.raises(dsd.DsdError) as ei:
        ctx.loss_forward(x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"],
                         x["conf_logit"])
    assert ei.value.code == -9 and ctx.launch_count() == n0
    ctx.close()
    ctx = dsd.Context(spec.V, spec.r, spec.G, 1, dtype="bf16")
    with pytest.raises(dsd.DsdError) as ei:   # B > R_max
        ctx.loss_forward(x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"],
                         x["conf_logit"])
    assert ei.value.code == -4
    ctx.close()


def test_full_size_loss_sampled_blocks(dsd):
    """The bench's workload (512 blocks x 7 positions, V = 151936, rank 256,
    in the launch configuration the bench times): sampled blocks against the
    oracle; the batch losses against an fp64 reduction of all kernel rows."""
    spec = synth.LossSpec()
    ctx, x, out, st = run(dsd, spec)
    assert st == 0
    row = out["row"].cpu().numpy()
    blocks = np.array([0, 1, 137, 300, 511])
    h = {k: synth.to_numpy(v[blocks]) if k not in ("E", "W") else None for k, v in x.items()}
    h["E"], h["W"] = synth.to_numpy(x["E"]), synth.to_numpy(x["W"])
    ref = O.loss_forward(h["U"], h["E"], h["W"], h["prev_tok"], h["P"], h["target"],
                         h["conf_logit"])
    rows = (blocks[:, None] * spec.G + np.arange(spec.G)[None, :]).reshape(-1)
    compare_rows(row, ref, rows)
    # the batch losses from the kernel's own per-row values, in fp64
    G, B = spec.G, spec.B
    w = O.position_weights(G)
    r64 = row.astype(np.float64).reshape(4, B, G)
    ce_loss = float(np.sum(w * r64[2].mean(0)))
    l1_loss = float(np.sum(w * r64[0].mean(0)))
    # bce from the rounded accept values differs from the kernel's fp64 one
    # by at most |z| * 2^-24
    conf_loss = float(r64[3].mean())
    k = out["losses"].cpu().numpy().astype(np.float64)
    for got, want in zip(k, (ce_loss, l1_loss, conf_loss,
                             0.1 * ce_loss + 0.9 * l1_loss + conf_loss)):
        assert abs(got - want) <= 1e-5 * abs(want) + 1e-6
    ctx.close()
