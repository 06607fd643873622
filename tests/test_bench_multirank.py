"""bench.py's multi-rank logic on CPU: two gloo ranks, max-over-ranks timing and the
whole-job rate (each rank an independent replica, so the rate sums over ranks)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    local_ms = 100.0 + 50.0 * rank  # rank 1 is the slower one
    mx = bench.max_over_ranks(local_ms)
    rate = bench.whole_job_rate(2.0e12, 10, ws, mx)
    out[rank] = (ws, r, local, mx, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][:3] == (2, 0, 0) and res[1][:3] == (2, 1, 1)
    for rank in (0, 1):
        assert res[rank][3] == 150.0
        assert abs(res[rank][4] - 2.0e12 * 10 * 2 / 0.150) < 1e-3 * res[rank][4]


def _rank_with_dead_peer(rank, world, port, out):
    import datetime
    import sys
    import time
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    if rank == 1:
        os._exit(0)  # the peer dies between steps, with nothing of its own in flight
    t0 = time.time()
    try:
        bench.max_over_ranks(1.0)
        out[rank] = ("returned", time.time() - t0)
    except Exception as e:  # the collective reports the missing peer instead of waiting forever
        out[rank] = (type(e).__name__, time.time() - t0)


def test_a_dead_peer_is_reported_not_waited_for():
    """Failure detection on the host: one of two gloo ranks exits after joining the group;
    the survivor's max-over-ranks reduction raises within the group's timeout instead of
    hanging (no GPU is involved)."""
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_with_dead_peer, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert 0 in res and 1 not in res
    kind, elapsed = res[0]
    assert kind != "returned", "the reduction returned without its peer"
    assert elapsed < 60.0


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(1.0, 4, 1, 2.0) == 2000.0


def test_peak_fractions():
    """A figure equal to a peak reads 100 % of it; the nominal dense bf16 rates are the
    datasheet figures halved for 2:4 sparsity: 2250 (HGX B300) and 2500 (GB300 NVL72)."""
    import json
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    burst, _, kind = bench.peaks()
    f = bench.peak_fractions(burst)
    assert f[f"of_{kind}_burst"] == 100.0
    assert f["of_nominal_dense_bf16_hgx_b300"] == round(100 * burst / 2250.0, 2)
    assert f["of_nominal_dense_bf16_gb300_nvl72"] == round(100 * burst / 2500.0, 2)
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            sus = json.load(fh).get("bf16_tflops_sustained")
        if sus:
            assert bench.peak_fractions(sus)["of_measured_sustained"] == 100.0


def test_results_file_gets_one_record_per_run(tmp_path, capsys):
    """--results appends each run's JSON line to a JSON-lines file, as printed."""
    import json
    import sys
    import types
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    path = tmp_path / "runs.jsonl"
    args = types.SimpleNamespace(results=str(path))
    bench.emit(args, {"metric": "m", "value": 1.0})
    bench.emit(args, {"metric": "m", "value": 2.0})
    printed = [json.loads(x) for x in capsys.readouterr().out.strip().splitlines()]
    stored = [json.loads(x) for x in path.read_text().strip().splitlines()]
    assert printed == stored == [{"metric": "m", "value": 1.0}, {"metric": "m", "value": 2.0}]
    bench.emit(types.SimpleNamespace(results=None), {"value": 3.0})  # stdout only
    assert len(path.read_text().strip().splitlines()) == 2
