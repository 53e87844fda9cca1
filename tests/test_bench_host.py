"""Host logic of bench.py that needs no GPU: the source digest that keys the
committed DRAM-traffic records to the code they were measured on."""
import json
import os

import bench

CSRC = os.path.join(bench.ROOT, "paged_kv_cache_261_gb300", "csrc")


def test_code_only_drops_comments_and_keeps_literals():
    src = 'int a = 1; // one\n/* two\n lines */ const char *s = "x // y /* z */";\nchar c = \'/\';  int b;'
    assert bench.code_only(src) == 'int a = 1; const char *s = "x // y /* z */"; char c = \'/\'; int b;'
    assert bench.code_only('s = "q\\" // in"; // out') == 's = "q\\" // in";'
    assert bench.code_only("x;// it's\ny;") == "x; y;"


def test_prose_edits_keep_the_digest_and_code_edits_change_it():
    with open(os.path.join(CSRC, "decode_tc.cu"), encoding="utf-8") as f:
        text = f.read()
    base = bench.code_only(text)
    reworded = "// a new first line of prose\n" + text.replace("\n\n", "\n\n/* note */\n", 3)
    assert bench.code_only(reworded) == base
    changed = text.replace("constexpr int kStages = 3;", "constexpr int kStages = 4;")
    assert changed != text and bench.code_only(changed) != base


def test_every_traffic_record_names_a_kernel_family():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for wl, ent in rec.items():
        assert ent["dram_bytes_per_launch"] > 0
        assert len(ent["source_digest"]) == 16
        assert bench.traffic_family(wl) in bench._KERNEL_SOURCES


def test_reference_arm_prints_the_contract_line(capsys):
    import argparse
    args = argparse.Namespace(workload="llama8b_decode", steps=2, warmup=1, gpus=1)
    bench.run_reference(args, budget_total_s=0.5)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True and line["steps"] == 2
    assert line["config"]["workload"] == "llama8b_decode" and line["config"]["sampled_seqs"] >= 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main()
    assert capsys.readouterr().out == ""


def test_clock_samples_summary():
    lines = ["2070, 2070, 812.3, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
             "2055, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
             "1980, 2070, 1401.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
             "[N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n",
             "garbage line\n"]
    got = bench.ClockSampler.summarise(lines)
    assert got == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 4}
    hot = bench.ClockSampler.summarise(["1500, 2070, 1400, 0x48, Active, Active, Not Active, Not Active\n"])
    assert hot["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.ClockSampler.summarise(["only, three, fields\n"]) is None


def test_algorithmic_bytes_by_hand_on_the_tiny_batch():
    import workloads
    w = workloads.tiny_fp32()                       # contexts 5, 17, 33, 64; H = Hk = 4; D 64; bs 4; fp32
    ab = w.algorithmic_bytes()
    assert ab["kv"] == (5 + 17 + 33 + 64) * 4 * 64 * 2 * 4          # K and V once: 243,712 B
    assert ab["qo"] == 2 * 4 * 4 * 64 * 4                           # q in, out back
    assert ab["meta"] == 4 * (2 + 5 + 9 + 16) + 4 * 4               # table entries used, lengths
    assert ab["decode"] == ab["kv"] + ab["qo"] + ab["meta"]
    assert ab["write"] == 2 * 4 * 4 * 64 * (4 + 4) + 4 * 4          # one token per sequence, K and V
    # an 8-bit cache counts one byte per cached element, the queries keep theirs
    ab8 = w.algorithmic_bytes(cache_elem_bytes=1)
    assert ab8["kv"] * 4 == ab["kv"] and ab8["qo"] == ab["qo"]


def test_decode_bytes_of_the_8b_shaped_batch():
    import workloads
    w = workloads.llama8b_decode()
    ab = w.algorithmic_bytes()
    expect_kv = int(w.context_lens.astype("int64").sum()) * 8 * 128 * 2 * 2
    assert ab["kv"] == expect_kv and 0.5e9 < ab["decode"] < 0.7e9   # about 0.6 GB a step


def test_prefill_flops_by_brute_force():
    import numpy as np
    import workloads
    pw = workloads.make_prefill("flops", 5, np.array([0, 3, 40], np.int32), np.array([4, 1, 7], np.int32),
                                8, 2, 64, 16, "bf16")
    visible = 0
    for prior, n in [(0, 4), (3, 1), (40, 7)]:
        for i in range(n):                          # query row i sits at position prior + i
            visible += prior + i + 1                # and sees every key up to itself
    assert pw.flops() == 4 * 64 * 8 * visible

