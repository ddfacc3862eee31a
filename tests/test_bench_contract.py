"""bench.py's reference arm (the CPU oracle, timed on a bounded sample) prints the
contract's JSON line on a machine without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["value"] > 0 and j["unit"] == "steps/s" and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["cpu_model"]
    up = j["cpu_baseline"]["upkeep"]          # the CPU analogue of the pages' upkeep comparison
    assert up["naive_ms_per_step"] > up["write_time_ms_per_step"] > 0
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # one block step timed: 1/60 of a full step, extrapolated x60, and said so
    assert j["block_steps_timed"] == 1 and abs(j["steps"] - 1 / 60) < 1e-12
    assert j["extrapolated"] is True and j["extrapolation_factor"] == 60
    assert abs(j["ms_per_step"] - 60 * j["cpu_baseline"]["block_step_ms"][0]) < 1e-6
    assert j["cpu_baseline"]["whole"]["tiny_100_steps_ms"] > 0
    assert j["config"]["workload"].startswith("steady denoise step")


def test_other_ranks_of_the_reference_arm_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_workload_figures_and_the_3d_workload():
    """The algorithmic figures the bench divides by, and the 3-D workload is one
    the library accepts (whole frames per write and per ring)."""
    sys.path.insert(0, ROOT)
    import bench
    from kv_cache_gb300 import kvring as kv
    w = dict(bench.WORKLOAD)
    # the pages' workload: every attention call reads 5,788 slots of which 757 are
    # new, 240 calls per step (60 blocks x 4 passes), positions reset every 42
    # steps (ai.info, "Characters funziona in tempo reale su quattro H100", section
    # "La gestione della cache spostata al momento della scrittura")
    assert (w["R"], w["T"], w["L"] * w["passes"], w["reset_every"]) == (5788, 757, 240, 42)
    write_bytes, attend_flop, rebase_bytes = bench.algorithmic(w)
    assert write_bytes == 757 * 16 * 128 * 6                # bf16 K, V in + e4m3 K, V out
    assert attend_flop == 4 * 757 * 5788 * 128 * 16          # Q K^T and P V, 2 FLOP per MAC
    assert rebase_bytes == 2 * 60 * 16 * 5788 * 128          # e4m3 K read + written
    c = dict(w)
    c.update(bench.ROPE_3D)
    S, W, pt, ph = c["rope_3d"]
    assert c["T"] % S == 0 and c["R"] % S == 0 and S % W == 0
    assert pt + 2 * ph == c["d"] // 2                        # width band as wide as the height band
    assert bench.rebase_row_bytes(c) == 48                   # 22 time pairs = 44 bytes -> three 16-byte pieces
    assert bench.rebase_row_bytes(w) == 128
    ring = kv.KVRing(1, c["H"], c["d"], c["R"], c["T"], max_position=c["R"] + 42 * c["T"], host_only=True,
                     rope_3d=c["rope_3d"])
    ring.close()


def test_gpu_arm_line_has_every_contract_key(monkeypatch, capsys):
    """The GPU arm's JSON line, assembled from a stand-in for the timed run (no GPU
    here): every key of the contract, with the roofline and CPU-baseline objects."""
    sys.path.insert(0, ROOT)
    import bench
    K = 42
    fake = dict(ms=15.4 * K, w_ms=[0.0166] * 60, w_b2b_ms=0.008, w_floor_ms=0.003, rb_more=[0.274, 0.275, 0.274, 0.276, 0.274], a_ms=[0.0631] * 240, r_ms=[], rb_ms=0.275, launches=25201,
                clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4},
                e2e_ms=16.1 * 12, e2e_steps=12, h2d=1116241920, d2h=1488322560, resets_timed=1)
    monkeypatch.setattr(bench, "run_gpu", lambda args, cfg, rank, world: fake)
    monkeypatch.setattr(bench, "oracle_sample", lambda cfg: {"block_s": 6.6, "step_s": 397.0, "cores": 16,
                                                             "cpu_model": "host", "sample": "one block"})
    monkeypatch.setattr(bench, "oracle_whole_configs", lambda: {
        "tiny_100_steps_ms": 900.0, "single_layer_write_attend_ms": 1500.0, "tiny_workload": "tiny",
        "single_layer_workload": "one layer"})
    monkeypatch.setattr(bench, "run_whole_configs_gpu", lambda: {"tiny_100_steps_ms": 4.0,
                                                                 "single_layer_write_attend_ms": 0.08})
    monkeypatch.setattr(bench, "oracle_upkeep_sample", lambda cfg: {"naive_ms_per_step": 6.8e5,
                                                                    "write_time_ms_per_step": 2.0e4, "ratio": 34.0,
                                                                    "sample": "one block"})
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main()
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "gpu_launches", "roofline",
                "cpu_baseline", "clocks"):
        assert key in j, key
    assert j["n_gpus"] == 1 and j["steps"] == K and abs(j["ms_per_step"] - 15.4) < 1e-9
    assert abs(j["value"] - 1e3 / 15.4) < 1e-6 and j["unit"] == "steps/s" and j["scaling"] == "weak"
    assert j["config"]["workload"].startswith("steady denoise step") and "l2" in j["config"]
    assert abs(j["e2e"]["value"] - 1e3 / 16.1) < 1e-6
    assert j["e2e"]["h2d_bytes_per_step"] > 0 and j["e2e"]["d2h_bytes_per_step"] > 0
    rf = j["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s"
    assert abs(rf["achieved"] - 4 * 757 * 5788 * 128 * 16 / 63.1e-6 / 1e12) < 1e-6
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-12
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 16 and cb["upkeep"]["ratio"] == 34.0
    # configurations 1 and 2 timed whole on both sides
    assert cb["whole"]["tiny_100_steps_ms"] == {"cpu_ms": 900.0, "gpu_ms": 4.0, "workload": "tiny"}
    assert cb["whole"]["single_layer_write_attend_ms"]["gpu_ms"] == 0.08
    assert j["resets_in_timed_steps"] == 1
    assert j["clocks"]["sm_mhz"] == 2070.0


def test_rebase_stress_line_counts_only_the_bytes_a_reset_moves(monkeypatch, capsys):
    """--rebase-stress (1-D and 3-D): the roofline's algorithmic bytes are the K
    bytes a reset reads and writes -- whole rows in 1-D, the time-band pieces in 3-D."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "run_rebase_stress", lambda args, cfg: [0.25] * 10)
    for extra, R, row in (([], 5788, 128), (["--rope-3d"], 5797, 48)):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--rebase-stress"] + extra)
        bench.main()
        j = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][0])
        nbytes = 2.0 * 60 * 16 * R * row
        assert j["value"] == 0.25 and j["higher_is_better"] is False
        assert abs(j["roofline"]["achieved"] - nbytes / 0.25e-3 / 1e9) < 1e-6
        assert ("3-D" in j["config"]["workload"]) == bool(extra)


def test_session_line_reports_step_times_and_drift(monkeypatch, capsys):
    """--session (the unsharded-width session): per-step median and p99, the
    breakdown, and the drift checkpoints with the rule that judges them."""
    sys.path.insert(0, ROOT)
    import bench
    drift = [{"step": s, "block": b, "bookkeeping_exact": True, "k_identical": 1.0, "v_identical": 1.0,
              "k_max_steps": 0.0, "attn_max_abs": 4e-3 if s == 1 else 5e-3, "attn_mean_rel": 1e-4}
             for s in (1, 41, 42, 43, 500, 999) for b in (0, 59)]
    fake = dict(step_ms=[20.0] * 980 + [25.0] * 20, drift=drift, clocks={"sm_mhz": 2070.0, "reasons": []},
                w_ms=[0.04] * 60, a_ms=[0.08] * 240, rb_ms=1.0)
    monkeypatch.setattr(bench, "run_session", lambda args, cfg: fake)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--session"])
    bench.main()
    j = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][0])
    assert j["unit"] == "ms/step" and j["higher_is_better"] is False and j["steps"] == 1000
    assert j["step_ms"]["median"] == 20.0 and j["step_ms"]["p99"] == 25.0
    assert abs(j["value"] - (980 * 20 + 20 * 25) / 1000) < 1e-9
    assert j["config"]["heads"] == 64 and j["config"]["attention_calls_per_step"] == 240
    assert j["no_drift"] is True and len(j["drift"]) == 12
    assert abs(j["breakdown"]["rebase_gbs"] - 2 * 60 * 64 * 5788 * 128 / 1e-3 / 1e9) < 1e-6
    fake["drift"][-1]["k_identical"] = 0.99
    bench.main()
    j = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][0])
    assert j["no_drift"] is False
