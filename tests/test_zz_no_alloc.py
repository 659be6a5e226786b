"""dsd_propose_noalloc: the propose call for callers that cannot allocate
device memory (an engine that owns all GPU memory through its own pool, code
running under a stream capture that forbids allocation, loops that must not
pay an allocation's synchronisation).  It keeps its scratch in a fixed array
inside the library instead of a context workspace.

Checked through the C ABI against the context-based dsd_propose (CUDA-core
engine) with the same tolerances as the other parity tests, on two calls in
a row so that the scratch left behind by the first call cannot leak into the
second.  This file is collected last on purpose."""

import numpy as np
import pytest
import torch

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


def _outputs(R, G):
    return dict(tokens=torch.full((R, G), -7, dtype=torch.int32, device=DEV),
                lse_q=torch.full((R, G), float("nan"), device=DEV),
                logit_at_tok=torch.full((R, G), float("nan"), device=DEV),
                survival=torch.full((R, G), float("nan"), device=DEV))


def _noalloc(dsd, spec, x, out, prev_tok=None, expect_status=0):
    status = torch.full((1,), 99, dtype=torch.int32, device=DEV)
    dsd.dsd_propose_noalloc(spec.V, spec.r, spec.G, spec.dtype, "none", True, spec.R, x["U"],
                            x["E"], x["W"], x["conf"],
                            x["prev_tok"] if prev_tok is None else prev_tok, x["req_id"],
                            spec.temperature, x["seed"], out["tokens"], out["lse_q"],
                            out["logit_at_tok"], out["survival"], status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == expect_status
    return {k: v.cpu().numpy() for k, v in out.items()}


def _context_propose(dsd, spec, x):
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, engine="simt")
    ref = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"],
                      spec.temperature, x["seed"])
    assert ctx.sync_status() == 0
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    ctx.close()
    return ref


def _same(a, b):
    assert np.array_equal(a["tokens"], b["tokens"])
    assert np.max(np.abs(a["lse_q"] - b["lse_q"])) <= parity.LOGIT_TOL
    assert np.max(np.abs(a["logit_at_tok"] - b["logit_at_tok"])) <= parity.LOGIT_TOL
    assert np.array_equal(a["survival"], b["survival"])


@pytest.mark.parametrize("dtype,temperature,seed", [("bf16", 0.0, 41), ("bf16", 1.0, 42),
                                                    ("f32", 0.7, 43)])
def test_noalloc_matches_context_propose_twice(dsd, dtype, temperature, seed):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=19, V=2568, dtype=dtype, ew_std=0.3,
                        temperature=temperature, seed=seed)
    x = synth.cycle_inputs(spec, device=DEV)
    ref = _context_propose(dsd, spec, x)
    first = _noalloc(dsd, spec, x, _outputs(spec.R, spec.G))
    second = _noalloc(dsd, spec, x, _outputs(spec.R, spec.G))
    _same(first, ref)
    _same(second, ref)
    assert np.isfinite(first["lse_q"]).all()


def test_noalloc_second_call_with_other_inputs(dsd):
    # a different batch after a larger one: nothing of the first call remains
    big = synth.scaled(synth.CYCLE_SPECS["greedy"], R=40, V=2568, ew_std=0.3, seed=44)
    small = synth.scaled(synth.CYCLE_SPECS["greedy"], R=7, V=2568, ew_std=0.3, seed=45)
    xb = synth.cycle_inputs(big, device=DEV)
    xs = synth.cycle_inputs(small, device=DEV)
    _noalloc(dsd, big, xb, _outputs(big.R, big.G))
    got = _noalloc(dsd, small, xs, _outputs(small.R, small.G))
    _same(got, _context_propose(dsd, small, xs))


def test_noalloc_more_vocabulary_tiles_than_ctas(dsd):
    # 313 vocabulary tiles of 128: more tiles than CTAs per draft step, so
    # every CTA walks several tiles; the split must match the context call's
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=4, V=40000, ew_std=0.3, seed=47)
    x = synth.cycle_inputs(spec, device=DEV)
    ref = _context_propose(dsd, spec, x)
    _same(_noalloc(dsd, spec, x, _outputs(spec.R, spec.G)), ref)
    _same(_noalloc(dsd, spec, x, _outputs(spec.R, spec.G)), ref)


def test_noalloc_reports_device_status_then_recovers(dsd):
    # a prev_tok outside [0, V) is reported through the status output, and
    # the next call, with valid inputs, reports 0 and drafts the same tokens
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=6, V=2568, ew_std=0.3, seed=48)
    x = synth.cycle_inputs(spec, device=DEV)
    bad = x["prev_tok"].clone()
    bad[2] = spec.V + 5
    _noalloc(dsd, spec, x, _outputs(spec.R, spec.G), prev_tok=bad, expect_status=-1)
    _same(_noalloc(dsd, spec, x, _outputs(spec.R, spec.G)), _context_propose(dsd, spec, x))


def test_noalloc_rejects_sizes_beyond_its_scratch(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=147, V=1032, ew_std=0.3, seed=46)
    x = synth.cycle_inputs(spec, device=DEV)    # 147 * 7 = 1029 > 1024
    out = _outputs(spec.R, spec.G)
    with pytest.raises(dsd.DsdError) as ei:
        dsd.dsd_propose_noalloc(spec.V, spec.r, spec.G, "bf16", "none", True, spec.R, x["U"],
                                x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1,
                                out["tokens"], out["lse_q"], out["logit_at_tok"],
                                out["survival"], status=None)
    assert ei.value.code == -4
    torch.cuda.synchronize()
    assert int(out["tokens"][0, 0]) == -7         # nothing was launched
