"""Host-side logic of bench.py: the replica aggregation used when it runs
under torchrun (world size 2, gloo, on CPU) and the JSON helpers."""

import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = bench.dist_info()
    assert (r, lr, w) == (rank, rank, world)
    bench.barrier(world)
    step_ms = 10.0 + 5.0 * rank           # rank 1 is the slow one
    m = bench.max_over_ranks(step_ms, world, torch.device("cpu"))
    out[rank] = m
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1] == 15.0
    # whole-job value of two replicas = 2 cycles per max step time
    assert 2 * 1e3 / out[0] == pytest.approx(133.333, rel=1e-4)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_algorithmic_bytes_of_the_high_concurrency_workload():
    spec = bench.cycle_spec("highconc")
    # one draft step: U rows of one position + all of W + E rows + argmax keys
    step = bench.propose_step_bytes(spec)
    assert step == 256 * 151936 * 2 + 151936 * 256 * 2 + 256 * 256 * 2 + 256 * 8
    # the phase: seven steps + confidences, previous tokens, four outputs
    b = bench.propose_alg_bytes(spec)
    assert b == 7 * step + 256 * 7 * 4 + 256 * 4 + 4 * 256 * 7 * 4
    assert 1.08e9 < b < 1.10e9
    # W once per phase: U 256*7*151936*2 + W 151936*256*2 + E rows + small I/O
    w1 = bench.propose_w_once_bytes(spec)
    assert w1 == 256 * 7 * 151936 * 2 + 151936 * 256 * 2 + 256 * 7 * 256 * 2 + 256 * 7 * 4 \
        + 256 * 4 + 4 * 256 * 7 * 4
    assert 620e6 < w1 < 630e6


def test_traffic_lookup_is_null_when_source_changed(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"simt_bias_kernel": {"greedy": {
        "source_hash": "0" * 16, "dram_bytes": 123}}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_for("simt_bias_kernel", "greedy") is None
    f.write_text(json.dumps({"simt_bias_kernel": {"greedy": {
        "source_hash": bench.source_hash("simt_bias_kernel"), "dram_bytes": 123}}}))
    assert bench.traffic_for("simt_bias_kernel", "greedy") == 123


def test_tensor_report_of_the_high_concurrency_workload():
    spec = bench.cycle_spec("highconc")
    rep = bench.tensor_report(spec, 1e-3, "tcgen05")
    # 2 R r V flops per draft step, seven steps: 139.4 GFLOP per phase
    assert rep["flops_per_phase"] == 2.0 * 256 * 256 * 151936 * 7
    assert abs(rep["achieved_tflops"] - rep["flops_per_phase"] / 1e-3 / 1e12) < 1e-9
    assert rep["frac"] == rep["achieved_tflops"] / rep["peak_tflops"]


def test_oracle_pool_times_whole_cycles_and_matches_the_oracle():
    # the CPU baseline's worker pool (spawned processes, single-threaded BLAS)
    # runs the same oracle cycle as a direct call: same committed tokens
    import numpy as np

    from oracle import dsd_oracle as O
    from semi_autoregressive_draft_gb300 import synth

    spec = synth.scaled(synth.CYCLE_SPECS["greedy"], R=5, V=1032, ew_std=0.3, seed=3)
    x = synth.cycle_inputs(spec, device="cpu")
    h = {k: synth.to_numpy(v) for k, v in x.items() if isinstance(v, torch.Tensor)}
    ref = O.cycle(h["U"], h["E"], h["W"], h["conf"], h["prev_tok"], h["P"], h["sps"],
                  req_id=h["req_id"].astype(np.int64), temperature=0.0, seed=x["seed"])
    want = int((ref["verify"]["accept_len"] + 1).sum())
    with bench.OraclePool(spec, x, workers=2) as pool:
        wall, tokens, busy = pool.cycle()
        assert tokens == want
        assert wall > 0 and busy > 0
        est, st_wall = pool.single_thread(2)
        assert est > 0 and st_wall > 0
    line = bench.oracle_baseline(spec, x, n_cycles=1, n_single=2)
    assert line["kind"] == "oracle" and line["cores"] >= 1 and line["value"] > 0
    assert line["single_thread"]["cores"] == 1
    assert "measured, not extrapolated" in line["sample"]
