"""The bench's own arithmetic and timing order, on the host: the algorithmic
flops and bytes behind every roofline fraction, the interleaving of timings,
and the comment-insensitive source hash that gates the recorded DRAM traffic."""
from __future__ import annotations

import pytest

import bench


def test_flops_per_row_and_per_chain():
    # GPT-3 MLP shard: 4 H F flops per row = 302 MFLOP; 618 GFLOP at M = 2048
    assert bench.chain_flops("gelu", 1, 12288, 6144) == pytest.approx(302.0e6, rel=1e-3)
    assert bench.chain_flops("gelu", 2048, 12288, 6144) == pytest.approx(618.5e9, rel=1e-3)
    # LLaMA SwiGLU shard: gate, up and down projections, 135 MFLOP per row
    assert bench.chain_flops("swiglu", 1, 8192, 2752) == pytest.approx(135.3e6, rel=1e-3)
    # stress chain: 4 M 8192^2
    assert bench.chain_flops("gelu", 1536, 8192, 8192) == 4.0 * 1536 * 8192 ** 2


def test_attention_flops_count_the_causal_half():
    M, H, F = 7, 12288, 1536
    proj = 2.0 * M * H * 3 * F + 2.0 * M * F * H
    # Q K^T and P V: 2 * head_dim flops per (query, key <= query) pair and head, twice
    pairs = sum(i + 1 for i in range(M))
    assert bench.chain_flops("attn", M, H, F) == pytest.approx(proj + 2 * 2 * pairs * F)


def test_weight_bytes_of_the_workloads():
    # weights once: GPT-3 302 MB, LLaMA 135 MB, attention 151 MB, stress 268 MB
    w = lambda kind, H, F: bench.chain_bytes(kind, 0, H, F)  # noqa: E731
    assert w("gelu", 12288, 6144) == pytest.approx(302e6, rel=1e-3)
    assert w("swiglu", 8192, 2752) == pytest.approx(135.3e6, rel=1e-3)
    assert w("attn", 12288, 1536) == pytest.approx(151e6, rel=1e-2)
    assert w("gelu", 8192, 8192) == pytest.approx(268.5e6, rel=1e-3)
    # per row: X read and Y written (2 H), the intermediate written and read (2 F)
    assert bench.chain_bytes("gelu", 1, 12288, 6144) - w("gelu", 12288, 6144) == 2 * (2 * 12288 + 2 * 6144)
    assert bench.chain_bytes("attn", 1, 12288, 1536) - w("attn", 12288, 1536) == 2 * (2 * 12288 + 8 * 1536)
    with pytest.raises(ValueError):
        bench.chain_bytes("conv", 1, 8, 8)


def test_interleaved_rounds_put_every_fn_in_every_place(monkeypatch):
    order = []
    monkeypatch.setattr(bench, "simple_time", lambda fn, repeats=1: (order.append(fn()), 1.0)[1])
    fns = {c: (lambda c=c: c) for c in "abcd"}
    med = bench.interleaved_times(fns, rounds=4)
    assert med == {c: 1.0 for c in "abcd"}
    rounds = [order[i:i + 4] for i in range(0, 16, 4)]
    assert rounds == [list("abcd"), list("bcda"), list("cdab"), list("dabc")]
    for pos in range(4):
        assert sorted(r[pos] for r in rounds) == list("abcd")


@pytest.mark.parametrize("src,want", [
    ("int a; // note\nint b;", "int a; int b;"),
    ("int a; /* one\n two */ int b;", "int a; int b;"),
    ('const char* s = "// not a comment";', 'const char* s = "// not a comment";'),
    ("char c = '/'; char d = '*'; // x", "char c = '/'; char d = '*';"),
    ('const char* e = "a\\"/*b";  int x;', 'const char* e = "a\\"/*b"; int x;'),
])
def test_strip_comments(src, want):
    assert bench.strip_comments(src) == want


def test_kernel_sha_follows_device_code_and_ring_configurations(tmp_path, monkeypatch):
    d = tmp_path / "consumer_gemm_chain_gb300" / "csrc"
    d.mkdir(parents=True)
    (d / "cs_kernel.cuh").write_text("int x = 1;\n")
    (d / "cs_ptx.cuh").write_text("int y = 1;\n")
    (d / "cs_chain.cu").write_text("constexpr int NS_A = 6, SB_A = 32768;\nint host = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    a = bench.kernel_sha()
    # comments, and host code other than the ring configurations, do not count
    (d / "cs_kernel.cuh").write_text("// a comment\nint   x = 1; /* another */\n")
    (d / "cs_chain.cu").write_text("constexpr int NS_A = 6, SB_A = 32768; // ring\nint host = 2;\n")
    assert bench.kernel_sha() == a
    # device code and ring depths do
    (d / "cs_ptx.cuh").write_text("int y = 2;\n")
    assert bench.kernel_sha() != a
    (d / "cs_ptx.cuh").write_text("int y = 1;\n")
    assert bench.kernel_sha() == a
    (d / "cs_chain.cu").write_text("constexpr int NS_A = 7, SB_A = 32768;\nint host = 2;\n")
    assert bench.kernel_sha() != a


def test_schedule_sha_follows_the_plans_tiles():
    import consumer_gemm_chain_gb300 as cs
    cs.cs_tune_clear()
    d = cs.cs_chain_desc_init(kind="gelu", M=2048, H=12288, F=6144, weight_layout="nk")
    a = bench.schedule_sha(cs, d, 152)
    assert bench.schedule_sha(cs, d, 152) == a
    d.tile_m, d.tile_n = 256, 256
    assert bench.schedule_sha(cs, d, 152) != a


def test_chunk_ready_from_a_timeline():
    decode = lambda u: (u >> 30, (u >> 14) & 0xFFF, u & 0x3FFF, (u >> 26) & 0xF)  # noqa: E731
    enc = lambda s, m, n: (s << 30) | (m << 14) | n  # noqa: E731
    # 2 tile rows of 512 (M = 1024): producers claimed from 100 ns, done at 140; row 0's
    # consumers done at 160, row 1's at 200
    recs = [[enc(0, m, n), 0, 100 + n, 0, 0, 0, 0, 140] for m in (0, 1) for n in (0, 1)]
    recs += [[enc(1, 0, n), 0, 140, 0, 0, 0, 0, 150 + 10 * n] for n in (0, 1)]
    recs += [[enc(1, 1, n), 0, 160, 0, 0, 0, 0, 190 + 10 * n] for n in (0, 1)]
    recs += [[enc(1, 1, 2), 0, 0, 0, 0, 0, 0, 0]]  # a record of a unit never reached
    r = bench.chunk_ready(recs, 1, 512, 1024, 4, decode)
    # chunks of 256 rows: the first two lie in tile row 0 (ready at 60), the others in row 1 (100)
    assert r["chunk_ready_frac"] == [0.6, 0.6, 1.0, 1.0]
    assert r["overlap_window_frac"] == pytest.approx(0.2)
    assert r["kernel_span_us"] == pytest.approx(0.1)


@pytest.mark.parametrize("steps", [1, 3, 200, 201, 2000, 4000])
def test_launch_samples_spread_over_the_timed_region(steps):
    slot = bench.sampled_calls(steps)
    assert sorted(slot.values()) == list(range(len(slot)))
    assert 0 in slot and len(slot) <= 201
    assert max(slot) >= steps - max(1, steps // 200)  # the last calls are sampled too


def _rec(sm, claim, first, acc, done, unit=0):
    # timestamps are ns of the global timer; 0 means "not reached", so offset them
    return [unit, sm, 1000 + claim, 1000 + claim, 1000 + first, 1000 + acc, 1000 + acc, 1000 + done]


def test_sm_busy_stats_on_a_hand_made_timeline():
    # SM 0 runs two units back to back over [0, 10]; SM 1 one unit over [0, 4];
    # SM 2 gets no unit: it counts against the whole-launch busy fraction and
    # is reported as unused, while the tail (from SM 1's end at 4) is measured
    # over the two SMs that ran units.
    recs = [_rec(0, 0, 0, 5, 6), _rec(0, 4, 5, 10, 10), _rec(1, 0, 0, 4, 4)]
    st = bench.sm_busy_stats(recs, 3)
    assert st["span_us"] == pytest.approx(10 / 1e3)
    assert st["busy_frac"] == pytest.approx(14 / 30) and st["busy_frac_used_sms"] == pytest.approx(14 / 20)
    assert st["sms_used"] == 2 and st["sms_unused"] == 1
    assert st["tail_us"] == pytest.approx(6 / 1e3) and st["tail_busy_frac"] == pytest.approx(6 / 12)
    st = bench.sm_busy_stats(recs, 2)
    assert st["busy_frac"] == pytest.approx(14 / 20)
    assert st["tail_us"] == pytest.approx(6 / 1e3)
    assert st["tail_busy_frac"] == pytest.approx(6 / 12)
    assert st["tail_idle_sm_us"] == pytest.approx(6 / 1e3)


def test_union_of_overlapping_intervals():
    assert bench._union_len([(0, 5), (3, 8), (10, 12)]) == 10
    assert bench._union_len([(0, 5), (3, 8), (10, 12)], 4, 11) == 5


def test_stream_k_remainder_is_the_last_wave_of_the_last_stage():
    q = {"stages": 2, "split_k": [1, 1, 1], "sched_units": [96, 96, 0], "workers": 36}
    assert bench.stream_k_remainder(q) == (96 + 96) % 36  # 12 tiles after five whole waves
    assert bench.stream_k_remainder(dict(q, sched_units=[90, 90, 0])) == 0  # whole waves
    assert bench.stream_k_remainder(dict(q, split_k=[1, 3, 1])) == 0  # a split last stage takes no tail
    assert bench.stream_k_remainder(dict(q, sched_units=[70, 10, 0], workers=40)) == 0  # remainder > last stage


@pytest.mark.parametrize("steps", [1, 5, 199, 200, 201, 250, 399, 400, 401, 2000, 3875])
def test_sampled_calls_never_exceed_the_limit_and_spread_evenly(steps):
    s = bench.sampled_calls(steps)
    assert 1 <= len(s) <= 200
    assert sorted(s.values()) == list(range(len(s)))
    idx = sorted(s)
    assert idx[0] == 0 and all(i < steps for i in idx)
    gaps = {b - a for a, b in zip(idx, idx[1:])}
    assert len(gaps) <= 1  # one stride


def test_kernel_label_follows_the_configuration_rules():
    """The instantiation named in the bench line follows the library's rules:
    8- and 32-row activation tiles up to 8 and 32 rows on single SMs, the 48 KB
    stages for 256-wide single-SM tiles, pairs and 4-CTA clusters."""
    import bench

    def q(tile_m, tile_n, stages=2):
        return {"tile_m": tile_m, "tile_n": [tile_n] * stages + [128] * (3 - stages), "stages": stages}

    assert bench.kernel_label("gelu", 1, q(128, 128)) == "cs_chain_kernel<11,17408,1,0,1,8>"
    assert bench.kernel_label("swiglu", 8, q(128, 256)) == "cs_chain_kernel<5,33792,1,0,1,8>"
    assert bench.kernel_label("gelu", 9, q(128, 128)) == "cs_chain_kernel<9,20480,1,0,1,32>"
    assert bench.kernel_label("swiglu", 32, q(128, 128)) == "cs_chain_kernel<5,36864,1,0,1,32>"
    assert bench.kernel_label("gelu", 33, q(128, 128)) == "cs_chain_kernel<6,32768,1>"
    assert bench.kernel_label("gelu", 64, q(128, 256)) == "cs_chain_kernel<4,49152,1>"
    assert bench.kernel_label("gelu", 256, q(256, 256)) == "cs_chain_kernel<6,32768,2>"
    assert bench.kernel_label("gelu", 2048, q(512, 256)).startswith("cs_chain_kernel<6,32768,2,0,4>")
    assert bench.kernel_label("attn", 16, q(128, 128, 3)).startswith("cs_chain_kernel<6,32768,1,1>")
