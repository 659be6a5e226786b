"""Failure path of the bounded device waits, made to run out on purpose
without faulting or hanging the GPU: a self-test kernel waits on mbarriers
that nothing completes (no copy or tensor-core work in flight).  The wait
must give up, the context must report DSD_ERR_TIMEOUT through
dsd_sync_status, and the same context must then run a normal draft-verify
cycle with status 0 and oracle-matching results.

The pages' only failure handling is the scheduler's fallback under overload
("DSpark 论文精读" section 6); the rule tested here, that every device wait
ends in a status rather than a hang, is the library's own."""

import numpy as np
import pytest
import torch

from semi_autoregressive_draft_gb300 import synth
from tests import parity
from tests.test_gpu_parity import check_cycle, dsd  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def _cycle_on(ctx, spec, x):
    T = spec.temperature
    prop = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"], req_id=x["req_id"],
                       temperature=T, seed=x["seed"])
    sch = ctx.schedule(prop["survival"], x["sps"])
    ver = ctx.verify(x["P"], prop["tokens"], sch["keep_len"], U=x["U"], E=x["E"], W=x["W"],
                     prev_tok=x["prev_tok"], lse_q=prop["lse_q"],
                     logit_at_tok=prop["logit_at_tok"], req_id=x["req_id"], temperature=T,
                     seed=x["seed"])
    st = ctx.sync_status()
    k = {n: t.cpu().numpy() for n, t in {**prop, **sch, **ver}.items()}
    k["keep_used"] = k["keep_len"]
    return st, k


@pytest.mark.parametrize("engine,temperature", [("auto", 0.0), ("simt", 1.0)])
def test_wait_that_never_completes_times_out_and_context_recovers(dsd, engine, temperature):
    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=19, V=2568, ew_std=0.3,
                        temperature=temperature, seed=61)
    x = synth.cycle_inputs(spec, device=DEV)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine=engine)
    # a first cycle, so the timeout lands on a context that has already run
    st, before = _cycle_on(ctx, spec, x)
    assert st == 0
    roles = torch.full((3,), -1, dtype=torch.int32, device=DEV)
    dsd.dsd_wait_selftest(ctx.handle, 4096, roles)
    assert ctx.sync_status() == -7                 # DSD_ERR_TIMEOUT, read and cleared
    assert roles.tolist() == [0, 0, 2]             # neither phase completed; both waiters left
    assert ctx.sync_status() == 0
    st, after = _cycle_on(ctx, spec, x)
    assert st == 0
    check_cycle(spec, x, after)
    for name in ("tokens", "keep_len", "accept_len", "next_token"):
        assert np.array_equal(after[name], before[name]), name
    assert np.max(np.abs(after["lse_q"] - before["lse_q"])) <= parity.LOGIT_TOL
    ctx.close()


def test_wait_selftest_rejects_bad_limits_before_any_launch(dsd):
    ctx = dsd.Context(2568, 64, 7, 4, dtype="bf16")
    n0 = ctx.launch_count()
    for bad in (0, (1 << 20) + 1):
        with pytest.raises(dsd.DsdError) as ei:
            dsd.dsd_wait_selftest(ctx.handle, bad)
        assert ei.value.code == -1
    assert ctx.launch_count() == n0
    assert ctx.sync_status() == 0
    ctx.close()
