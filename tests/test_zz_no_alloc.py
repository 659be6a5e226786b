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


def _noalloc(dsd, spec, x, out):
    dsd.dsd_propose_noalloc(spec.V, spec.r, spec.G, spec.dtype, "none", True, spec.R, x["U"],
                            x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"],
                            spec.temperature, x["seed"], out["tokens"], out["lse_q"],
                            out["logit_at_tok"], out["survival"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


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
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=dtype, engine="simt")
    ref = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"],
                      temperature, x["seed"])
    assert ctx.sync_status() == 0
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    ctx.close()
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
    ctx = dsd.Context(small.V, small.r, small.G, small.R, dtype="bf16", engine="simt")
    ref = ctx.propose(xs["U"], xs["E"], xs["W"], xs["conf"], xs["prev_tok"], xs["req_id"], 0.0,
                      xs["seed"])
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    ctx.close()
    _same(got, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(dsd):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=147, V=1032, ew_std=0.3, seed=46)
    x = synth.cycle_inputs(spec, device=DEV)    # 147 * 7 = 1029 > 1024
    out = _outputs(spec.R, spec.G)
    with pytest.raises(dsd.DsdError) as ei:
        dsd.dsd_propose_noalloc(spec.V, spec.r, spec.G, "bf16", "none", True, spec.R, x["U"],
                                x["E"], x["W"], x["conf"], x["prev_tok"], x["req_id"], 0.0, 1,
                                out["tokens"], out["lse_q"], out["logit_at_tok"],
                                out["survival"])
    assert ei.value.code == -4
    torch.cuda.synchronize()
    assert int(out["tokens"][0, 0]) == -7         # nothing was launched
