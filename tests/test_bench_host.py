"""Host-side logic of bench.py (CPU only): workload selection for profiling
captures and the DRAM-traffic lookup from a committed ncu summary."""
import bench
import workloads as wl


def test_select_groups_and_fraction():
    w = bench.select_groups(wl.llama3_405b_layer(), [1, 3])
    assert [(g.m, g.n) for g in w.groups] == [(16384, 1024), (53248, 16384)]
    assert w.name == "llama3-405b-layer[1,3]"
    w = bench.select_groups(wl.square(4096), None, 1.0 / 16)
    assert w.groups[0].rank(w.fraction) == 256
    assert bench.select_groups(wl.gpt_small(), None) == wl.gpt_small()


def test_profiled_traffic_reads_summary_and_checks_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic_demo.txt").write_text(
        "# ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum ...\n"
        "csrc_sha256 abc123\n"
        "launch 0 dion_update_tc read_bytes 100 write_bytes 50\n"
        "launch 1 dion_update_tc read_bytes 300 write_bytes 150\n"
        "launch 2 other_kernel read_bytes 7 write_bytes 7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "csrc_digest", lambda: "abc123")
    v, src = bench.profiled_traffic("demo", "dion_update_tc")
    assert v == 300.0 and "2 launches" in src
    assert bench.profiled_traffic("demo", "missing")[0] is None
    assert bench.profiled_traffic("nothere", "dion_update_tc")[0] is None
    monkeypatch.setattr(bench, "csrc_digest", lambda: "0" * 64)   # sources changed since the capture
    v, why = bench.profiled_traffic("demo", "dion_update_tc")
    assert v is None and "changed" in why


def test_csrc_digest_covers_the_sources():
    d = bench.csrc_digest()
    assert len(d) == 64 and d == bench.csrc_digest()


def test_streaming_kernel_bound_follows_the_larger_floor():
    """At rank 1024 the update's 4 m n r flops outweigh its 14 m n bytes (so
    its floor is the tensor one); at rank 256 the bytes set it."""
    peaks = dict(hbm_gbs=6790.7, bf16_tflops=1919.3)
    for w, want in ((wl.llama3_405b_layer(), "tensor"), (wl.llama3_8b(), "hbm")):
        state = [{"g": g, "r": g.rank(w.fraction)} for g in w.groups if g.rank(w.fraction) >= 256]
        b, c = bench.kernel_cost("dion_update_tc", w, state)
        f = bench.kernel_flops("dion_update_tc", w, state)
        assert b == "hbm" and c > 0 and f > 0
        got, cost = bench.mixed_bound(b, c, f, **peaks)
        assert got == want and cost == (f if want == "tensor" else c)
    assert bench.mixed_bound("alu", 1.0, 1e30, **peaks) == ("alu", 1.0)


def test_l2_flush_only_for_workloads_near_the_l2_size():
    assert bench.input_footprint(wl.square(1024)) == 8 * 1024 * 1024 * 8
    assert bench.needs_l2_flush(wl.square(1024)) and bench.needs_l2_flush(wl.square(2048))
    for w in (wl.square(4096), wl.gpt_small(), wl.llama3_8b(), wl.llama3_405b_layer()):
        assert not bench.needs_l2_flush(w)


def test_qr_product_cost_counts_every_launch_of_a_step():
    """Two Grams per step (both CholeskyQR passes); two applies through the
    GEMM at rank <= 248, one above (the blocked path applies the first pass)."""
    one = lambda g, r: g.batch * 6 * 2.0 * g.m * r * r
    w = wl.gpt_small()
    st = [{"g": g, "r": g.rank(w.fraction)} for g in w.groups]
    assert bench.kernel_cost("qr_gram_tc", w, st)[1] == sum(2 * one(x["g"], x["r"]) for x in st)
    assert bench.kernel_cost("qr_apply_tc", w, st)[1] == sum(2 * one(x["g"], x["r"]) for x in st)
    w = wl.square(16384)
    st = [{"g": g, "r": g.rank(w.fraction)} for g in w.groups]
    assert st[0]["r"] == 4096
    assert bench.kernel_cost("qr_gram_tc", w, st)[1] == 2 * one(st[0]["g"], 4096)
    assert bench.kernel_cost("qr_apply_tc", w, st)[1] == one(st[0]["g"], 4096)
