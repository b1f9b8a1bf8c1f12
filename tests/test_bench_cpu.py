"""The bench on CPU: its algorithmic byte counts (the roofline numerators) and
the JSON line of its reference arm.

A decode frame at batch 1 streams every weight it needs once: the 36 Slow AR
layers, the 4,096 semantic rows of the tied head (the constrained argmax needs
no other row), and 9 Fast AR passes over the 4 Fast layers plus one codebook
head slice each ("s2pro-native", Where it stands: nine greedy passes per frame;
the per-frame parameter figure there is pinned in the oracle tests).  KV adds
2 x layers x kv heads x head dim elements per context token per sequence.
"""
import bench
from s2_inputs import S2, param_counts


def test_frame_weight_bytes_stream_each_weight_once():
    total, w = bench.bytes_per_frame(S2, 0, 1)
    assert total == w == 14_742_978_560
    c = param_counts(S2)
    d, C = S2.d, S2.codebook_size
    assert c["layer"] == S2.d * (S2.q_dim + 2 * S2.kv_dim) + S2.q_dim * S2.d + 3 * S2.ffn * S2.d
    assert w == 2 * (36 * c["layer"] + C * d + 9 * (4 * c["layer"] + C * d))
    # the full tied head instead of the semantic slice would add 151,936 rows
    full_head = 2 * (c["tok_emb"] - C * d)
    assert full_head == 2 * 151_936 * d


def test_kv_term_per_context_token():
    _, w = bench.bytes_per_frame(S2, 0, 1)
    per_tok_bf16 = 36 * 2 * 8 * 128 * 2
    assert per_tok_bf16 == 147_456 == bench.kv_bytes_per_token(S2)
    for kv_bytes, per_tok in ((2, per_tok_bf16), (4, 2 * per_tok_bf16)):
        t, w2 = bench.bytes_per_frame(S2, 100.5, 3, kv_bytes=kv_bytes)
        assert w2 == w
        # each sequence reads its context and writes one new token
        assert t - w == (3 * 100.5 + 3) * per_tok


def test_shared_radix_prefix_is_read_once_per_step():
    """32 sequences over one 896-token shared prefix (56 pages) read those
    pages once per step, plus their own 194 private context tokens each."""
    t, w = bench.bytes_per_frame(S2, 1090, 32, shared_prefix=896)
    assert t - w == (896 + 32 * (1090 - 896) + 32) * 147_456
    t_unshared, _ = bench.bytes_per_frame(S2, 1090, 32)
    assert t_unshared - t == 31 * 896 * 147_456


def test_decode_call_bytes_match_the_scope_table():
    """Call totals of the four full-size workloads (n - 1 slow steps, n heads
    and Fast AR loops, bf16 KV, the shared prefix once): 877.9, 2,974.3,
    4,728.8 and 48,985 GB for the batch-1, voice-clone, batch-32 and
    batch-128 workloads."""
    from s2_inputs import make_workload
    want = {1: 877.9, 2: 2974.3, 3: 4728.8, 4: 48985.2}
    for i, gb in want.items():
        wl = make_workload(i)
        T = max(p.T for p in wl.prompts)
        t, w = bench.decode_call_bytes(S2, T, wl.n_frames, wl.batch, wl.shared_prefix // 16 * 16)
        assert abs(t / 1e9 - gb) < 0.06, (i, t / 1e9)
    # batch 1, 41-token prompt: the KV is 4,189 token reads and writes
    t, w = bench.decode_call_bytes(S2, 41, 60, 1)
    assert t - w == 4189 * 147_456
    assert w == 59 * 2 * 36 * 100_925_440 + 60 * (14_742_978_560 - 2 * 36 * 100_925_440)


def test_batch_shares_the_weight_stream():
    # 32 sequences read the weights once per frame, not 32 times
    t1, w = bench.bytes_per_frame(S2, 0, 1)
    t32, w32 = bench.bytes_per_frame(S2, 0, 32)
    assert t1 == t32 == w == w32


def test_reference_arm_prints_the_contract_line(tmp_path):
    """``bench.py --impl reference`` (the oracle on the host cores) on the tiny
    workload: one JSON line with the metric, the reference marker, the
    cpu_baseline description and an e2e entry that moves no bytes."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, S2_WEIGHTS_DIR=str(tmp_path))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "0", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, env=env, timeout=600, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == "frames/s" and d["unit"] == "frames/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny_b1_t16_f4"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "frames/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_vocoder_plan_counts():
    """The vocoder's launch list and algorithmic work: 4 + 7 per block
    launches; per frame ~2.1 GFLOP, dominated by the k=7 convolutions, with
    the transposed convolutions at 2 * s * c_out * c_in * 2 per input row."""
    import bench
    from s2_inputs.vocoder import DAC_S2, DAC_MINI
    for cfg in (DAC_S2, DAC_MINI):
        plan = bench.dac_plan(cfg, 1, 1)
        assert len(plan) == 4 + 7 * len(cfg.rates)
    plan = bench.dac_plan(DAC_S2, 2, 3)
    fl = sum(p[1] for p in plan) / 6
    assert 2.0e9 < fl < 2.3e9, fl
    d = dict((p[0], p) for p in plan)
    # block 0: 6 input rows -> 48 output rows, 1536 -> 768 channels, 2 taps reach each output
    assert d["block.0.up"][1] == 2 * 48 * 768 * 1536 * 2
    assert d["block.4.res.2.conv1"][1] == 2 * 6 * 2048 * 48 * 48 * 7
    assert d["block.4.res.2.conv2"][2] == 6 * 2048 * 48 * 4 * 3 + 2 * 48 * 48


def test_vocoder_summary_is_json_and_finds_the_dominant_launch():
    import json
    import numpy as np
    import bench
    from s2_inputs.vocoder import DAC_S2
    plan = bench.dac_plan(DAC_S2, 2, 3)
    per = np.full(len(plan), 0.01, np.float32)
    per[10] = 0.5
    rec = bench.vocoder_summary(DAC_S2, 2, 3, np.float32(1.0), np.int64(39), per,
                                {"bf16_tflops": 1928.0, "hbm_gbs": 6780.4})
    json.dumps(rec)
    assert rec["roofline"]["kernel"].endswith(f"({plan[10][0]})")
    assert abs(rec["roofline"]["us_per_launch"] - 500) < 1e-3
    assert 0 < rec["frac_of_roofline"] < 1


def test_frame_trace_summary_on_a_synthetic_timeline(tmp_path):
    """bench.py --frame-trace: per launch kind the medians of step (last exit
    after the previous launch's last exit), wait (median pass of the wait after
    that exit), prologue, body and tail, from the per-CTA stamps (ns) the
    library writes; rows far from a launch's entries (an earlier graph's
    leftovers in the slot) are dropped."""
    lines = ["launch 0 gemv A", "launch 1 attn B", "launch 2 gemv A"]
    t = 1_000_000_000
    # launch 0: two CTAs
    lines += [f"0 0 {t} {t + 500} {t + 1500} {t + 9000}", f"0 1 {t + 100} {t + 600} {t + 1600} {t + 10000}"]
    # launch 1: one CTA entering before launch 0 ended, passing its wait 1 us after
    lines += [f"1 0 {t + 8000} {t + 11000} {t + 12000} {t + 15000}"]
    # launch 2: two CTAs plus a stale row from long ago
    lines += [f"2 0 {t + 14000} {t + 16000} {t + 17000} {t + 20000}",
              f"2 1 {t + 14500} {t + 16000} {t + 18000} {t + 22000}",
              f"2 2 {t - 500_000_000} {t - 499_999_000} {t - 499_998_000} {t - 499_997_000}"]
    f = tmp_path / "trace.txt"
    f.write_text("\n".join(lines) + "\n")
    s = bench.frame_trace_summary(str(f))
    assert s["launches"] == 3
    assert s["span_us"] == 22.0                       # 1.000000000 s .. + 22 us, stale row dropped
    a, b = s["by_kind"]["gemv A"], s["by_kind"]["attn B"]
    assert a["launches"] == 2 and b["launches"] == 1
    assert b["step"] == 5.0 and b["wait"] == 1.0      # exits 10 us -> 15 us; wait passed at 11 us
    assert b["prologue"] == 1.0 and b["body"] == 3.0 and b["tail"] == 0.0
    # gemv A: launch 0 has no predecessor (no step / wait); launch 2's step 7 us, wait 1 us
    assert a["step"] == 7.0 and a["wait"] == 1.0
    assert a["prologue"] == 1.25 and a["tail"] == 0.75   # medians over both launches
