"""Host logic of bench.py: clock parsing, workload arithmetic, and the multi-rank
bookkeeping (barrier, max over ranks, whole-job aggregate) on two gloo ranks."""
import os
import socket
import types

import pytest
import torch.multiprocessing as mp

import bench


def test_workload_arithmetic_matches_pages():
    # "mojo-baro", round v2: bf16 weights 100.7 MB, q8 with a 4-byte scale slot 56.6 MB,
    # byte ratio 0.563 (round v1)
    rows = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "decode_bytes.txt")) as f:
        for line in f:
            p = line.split()
            if p and not p[0].startswith("#") and p[0] != "ratio":
                rows[p[2]] = (int(p[0]), int(p[1]), int(p[3]), float(p[4]))
            elif p and p[0] == "ratio":
                ratio = float(p[1])
    K, N, _, mb = rows["bf16"]
    assert round(bench.decode_weight_bytes(K, N, "bf16") / 1e6, 1) == mb
    K, N, sb, mb = rows["q8"]
    q8 = bench.decode_weight_bytes(K, N, "q8", scale_bytes=sb)
    assert round(q8 / 1e6, 1) == mb
    # printed to three places (0.5625 is printed as 0.563)
    assert abs(q8 / bench.decode_weight_bytes(K, N, "bf16") - ratio) <= 5e-4 + 1e-12
    assert bench.gemm_flops(4096, 4096, 4096) == 2 * 4096 ** 3


def test_parse_clock_csv():
    text = ("0, 1965, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1800, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "0, 300, 2070, 150.0, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active\n"
            "garbage line\n")
    s = bench.parse_clock_csv(text)
    assert s["sm_mhz"] == (1965 + 1800) / 2
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3 and s["samples_under_load"] == 2
    assert bench.parse_clock_csv("")["samples"] == 0


def test_parse_clock_csv_with_utilisation_and_temperature():
    # with the utilisation column, "under load" is utilisation >= 50 %, whatever the clock
    text = ("0, 2070, 2070, 185.0, 0x0, Not Active, Not Active, Not Active, Not Active, 41, 0\n"
            "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active, 52, 100\n"
            "0, 1920, 2070, 1398.0, 0x4, Not Active, Not Active, Not Active, Active, 58, 99\n"
            "0, 2070, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active, [N/A], 75\n")
    s = bench.parse_clock_csv(text)
    assert s["samples"] == 4 and s["samples_under_load"] == 3
    assert s["sm_mhz"] == 2070 and s["sm_mhz_min_under_load"] == 1920
    assert s["power_w_max"] == 1398.0 and s["power_w_median_under_load"] == (950.0 + 1398.0) / 2
    assert s["temp_c_max"] == 58 and s["reasons"] == ["sw_power_cap"]


def test_oracle_sample_plan_bounds():
    plan = bench.oracle_sample_plan(60e9)
    assert [n for n, _ in plan] == bench.SWEEP
    for n, rows in plan:
        assert 1 <= rows <= n
    assert sum(2.0 * r * n * n for n, r in plan) <= 66e9


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    w, r = bench.dist_init("gloo")
    bench.barrier()
    mx = bench.max_over_ranks(1.5 + r)  # rank r "took" 1.5 + r seconds
    val = bench.aggregate_value(100.0, 10, w, mx)
    q.put((r, w, mx, val))
    dist.destroy_process_group()


def test_two_rank_bookkeeping_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, mx, val in out:
        assert w == 2
        assert mx == 2.5                  # the slowest rank's time
        assert val == 100.0 * 10 * 2 / 2.5  # units of all ranks / slowest time


def test_record_traffic_and_staleness(tmp_path, monkeypatch):
    # an ncu --csv log of one launch -> bytes per launch, tied to the kernel family's sources
    csv_path = tmp_path / "t.csv"
    csv_path.write_text(
        "==PROF== Connected to process 1\n"
        '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
        '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
        '"0","1","p","h","gemv_q8_dp2a_kernel","1","7","(128, 1, 1)","(1216, 1, 1)","0","10.3","s",'
        '"dram__bytes_read.sum","Mbyte","53.51"\n'
        '"0","1","p","h","gemv_q8_dp2a_kernel","1","7","(128, 1, 1)","(1216, 1, 1)","0","10.3","s",'
        '"dram__bytes_write.sum","Kbyte","49.15"\n')
    monkeypatch.setattr(bench, "TRAFFIC", str(tmp_path / "traffic.json"))
    bench.record_traffic(types.SimpleNamespace(ncu_csv=str(csv_path), key="gemv_q8"))
    assert bench.load_traffic("gemv_q8") == 53510000 + 49150
    # a record taken on other sources is not used
    assert bench.traffic_note("gemv_q8") is None
    monkeypatch.setattr(bench, "kernel_source_digest", lambda kind="gemm": "0" * 16)
    assert bench.load_traffic("gemv_q8") is None
    note = bench.traffic_note("gemv_q8")
    assert "53559150 bytes" in note and "0" * 16 in note
    assert bench.traffic_note("gemm_4096") == "no ncu record for this launch"


def test_tuned_configurations_freeze_into_a_loadable_table(tmp_path):
    import shape_driven_tile_gb300 as sdt
    p = tmp_path / "tuned.txt"
    out = bench.write_tune_table(str(p), [
        (4096, 4096, 4096, {"tile": "2cta_256x256", "stagger": 0, "raster": 1, "stages": 6}),
        (16, 16384, 4096, {"tile": "64x64"}),            # gemm_f16 cannot run this shape: left out
        (1024, 1024, 1024, {"tile": "64x64", "stagger": -1, "raster": 0, "stages": 0})], "a test")
    assert out["entries"] == 2
    sdt.load_tune_table(str(p))
    try:
        assert sdt.lib().sdt_tune_table_size() == 2
        assert sdt.tile_info(sdt.tune_table_lookup(4096, 4096, 4096))["name"] == "2cta_256x256"
        assert sdt.tune_table_lookup(16, 16384, 4096) == -1
    finally:
        sdt.clear_tune_table()


def test_sweep_resume_file(tmp_path):
    # an interrupted sweep keeps its finished shapes; a torn last line is ignored
    path = tmp_path / "sweep.jsonl"
    bench.append_resume(str(path), {"shape": [256, 256, 256], "pick": "64x64", "best": "64x64", "slowdown": 0.0,
                                    "us": {"64x64": 8.0}})
    bench.append_resume(str(path), {"shape": [512, 512, 512], "pick": "64x64", "best": "64x64", "slowdown": 0.0,
                                    "us": {"64x64": 9.0}})
    with open(path, "a") as f:
        f.write('{"shape": [768, 768, 7')
    rows = bench.load_resume(str(path), [(256, 256, 256), (768, 768, 768)])
    assert [r["shape"] for r in rows] == [[256, 256, 256]]
    assert bench.load_resume(str(tmp_path / "missing.jsonl"), [(256, 256, 256)]) == []
    assert bench.load_resume(None, [(256, 256, 256)]) == []


@pytest.mark.parametrize("steps", [1, 9, 10, 11, 19, 20, 25, 2000])
@pytest.mark.parametrize("graphed", [True, False])
def test_step_schedule_covers_every_step_once(steps, graphed):
    plan = bench.step_schedule(steps, 10, 8, graphed=graphed)
    seen = [i for kind, first, count in plan for i in range(first, first + count)]
    assert seen == list(range(steps))
    inst = [first for kind, first, _ in plan if kind == "instrumented"]
    assert inst == (list(range(9, steps, 10)) or [steps - 1])
    for kind, first, count in plan:
        if kind == "graph":
            # nine steps replayed right before an instrumented one
            assert graphed and count == 9 and first % 10 == 0 and first + 9 in inst
    if graphed and steps >= 10:
        # every instrumented step is queued behind a graph replay
        kinds = [k for k, _, _ in plan]
        assert all(kinds[j - 1] == "graph" for j, k in enumerate(kinds) if k == "instrumented")
    if not graphed:
        assert all(kind != "graph" for kind, _, _ in plan)
    # graphs are keyed by their first step's decode buffer: at most four distinct keys
    assert len({first % 8 for kind, first, _ in plan if kind == "graph"}) <= 4


def test_reference_arm_prints_the_contract_line():
    # the reference arm is the oracle timed on the host cores: it runs here, without a GPU
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    for key in ("metric", "value", "unit", "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
                "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_cpu_baseline_leg_reports_all_threads_and_one(monkeypatch):
    # small sweep sizes stand in for the real ones: the leg's bookkeeping, not its scale
    import torch

    import bench
    from shape_driven_tile_gb300 import inputs

    monkeypatch.setattr(bench, "SWEEP", [64, 128])
    monkeypatch.setattr(bench, "DEC_K", 64)
    monkeypatch.setattr(bench, "DEC_N", 32)
    host = {n: (inputs.uniform((n, n), seed=3 * n), inputs.uniform((n, n), seed=3 * n + 1)) for n in (64, 128)}
    x = inputs.uniform((64,), seed=5, dtype=torch.bfloat16)
    W = inputs.uniform((32, 64), seed=6, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(32, 64, seed=7)
    host["dec_bf16"] = (x, W)
    host["dec_q8"] = (x, q, s)
    import oracle

    before = oracle.max_threads()
    base, gate = bench.cpu_baseline_leg(host, None, budget_flops=1e6, check=False)
    assert gate is None
    assert base["kind"] == "oracle" and base["cores"] == before and base["value"] > 0
    one = base["one_thread"]
    assert one["value"] > 0 and one["sample"].startswith("128^3: 32 rows")
    # the one-thread figure leaves the oracle's thread count as it was: a second leg (the
    # benchmark runs a calibration leg first) still uses every thread
    assert oracle.max_threads() == before
    assert bench.cpu_baseline_leg(host, None, budget_flops=1e6, check=False)[0]["cores"] == before


def test_packed_staging_buffer_views():
    # the end-to-end leg's staging buffers: 256-byte aligned views that alias one buffer
    import torch

    import bench

    specs = [("a", (3, 5), torch.float16), ("b", (7,), torch.float32), ("c", (2, 2, 2), torch.int8)]
    buf, v = bench._packed(specs, lambda n: torch.zeros(n, dtype=torch.uint8))
    assert buf.numel() == 768
    offs = {k: t.data_ptr() - buf.data_ptr() for k, t in v.items()}
    assert offs == {"a": 0, "b": 256, "c": 512}
    assert all(tuple(v[k].shape) == shape and v[k].dtype == dt for k, shape, dt in specs)
    v["b"].fill_(2.0)
    assert torch.equal(buf[256:284].view(torch.float32), torch.full((7,), 2.0))
