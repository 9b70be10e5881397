"""The benchmark's byte model and its roofline bookkeeping, on CPU.

The roofline fraction divides the algorithmic bytes of a step by its time:
the whole K cache, every distinct (sequence, KV head, key) V row any head of
a group drew (a row read once serves all heads of its group, Eq. 4 with GQA),
q and the fp32 output.  These tests recount those bytes from the tensors'
shapes and a made-up draw table, independently of bench.py's formulas."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _ragged_inputs():
    wl = synth.Workload("model_ragged", 3, 8, 2, 64, 700, "bf16", 16, "stratified", ragged=(100, 700),
                        S_rule="max64_nk_div128")
    return synth.generate(wl, 2)


def test_unique_rows_counts_each_group_row_once():
    inp = _ragged_inputs()
    B, H, _ = inp.q.shape
    G = H // inp.wl.n_kv_heads
    S = inp.S_max
    rng = np.random.default_rng(0)
    idx = np.full((B, H, S), -1, np.int32)
    want = 0
    for b in range(B):
        S_b = inp.S_of(b)
        nk = int(inp.nk_per_seq[b])
        for k in range(inp.wl.n_kv_heads):
            rows = set()
            for g in range(G):
                draws = np.sort(rng.integers(0, nk, S_b))
                idx[b, k * G + g, :S_b] = draws
                rows.update(draws.tolist())
            want += len(rows)
    assert bench.count_unique_rows(inp, idx) == want


def test_step_bytes_from_shapes():
    inp = _ragged_inputs()
    B, H, d = inp.q.shape
    rows_total = int(inp.nk_per_seq.sum())
    unique = 123
    k_bytes = rows_total * inp.wl.n_kv_heads * d * 2          # bf16 keys of every sequence
    want = k_bytes + unique * d * 2 + B * H * d * 2 + B * H * d * 4
    assert bench.step_bytes(inp, unique) == want
    assert bench.dense_bytes(inp) == 2 * k_bytes + B * H * d * 2 + B * H * d * 4


def test_llama32k_byte_budget():
    """The Llama-3.1-8B layer at 32K: 67,108,864 bytes of K; the byte model
    adds 256 bytes per distinct drawn row, q (8 KiB) and out (16 KiB)."""
    inp = synth.generate(synth.llama32k(32768, 256, "systematic"), 0)
    assert bench.step_bytes(inp, 0) == 67108864 + 8192 + 16384
    assert bench.step_bytes(inp, 3782) - bench.step_bytes(inp, 0) == 3782 * 256


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    """A recorded ncu traffic figure is used only for the workload it was
    taken on and while the kernel sources hash to the recorded value."""
    import json
    rec = {"workload": "w", "dram_bytes_per_launch": 5, "source_hash": bench.source_hash(bench.KERNEL_SOURCES)}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w") == 5
    assert bench.recorded_traffic("other") is None
    rec["source_hash"] = "0" * 16
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic("w") is None


def _run_bench(args, **env):
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                       text=True, timeout=600, env=dict(os.environ, **env))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle as the reference arm) prints
    one JSON line with the GPU arm's metric, unit and config keys, its own
    cpu_baseline and a zero-byte e2e; ranks other than 0 exit quietly."""
    out = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    assert len(out) == 1
    line = out[0]
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["value"] > 0 and line["higher_is_better"] is False and line["steps"] == 3 and line["warmup"] == 3
    assert line["config"]["workload"] == synth.tiny("systematic").name
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                      RANK="1", WORLD_SIZE="2", LOCAL_RANK="1") == []
