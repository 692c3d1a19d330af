"""Host-side pieces of bench.py (no GPU): the kernel-source hash that keys the DRAM-traffic record,
the record's scaling to the layers a run launches, and the timeline summary's arithmetic on a
synthetic stamp array."""
import numpy as np

import bench


def test_code_only_drops_comments_and_layout_but_keeps_strings():
    a = "int a;  // one\n/* two\n lines */ int b = \"// kept\";\n"
    b = "int a; int b = \"// kept\";"
    assert bench.code_only(a) == bench.code_only(b) == 'int a; int b = "// kept";'
    assert bench.code_only("x = 1;") != bench.code_only("x = 2;")
    assert bench.code_only("c = '/';  // q") == "c = '/';"


def test_kernel_source_hash_is_stable():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()


def test_timeline_summary_on_synthetic_stamps():
    C, L, P = 4, 10, 64
    t = np.zeros((C, L, P), np.uint64)
    ghz = 2.0
    for c in range(C):
        for l in range(L):
            top = 1_000_000 + l * 20_000 + c * 100          # cycles: 10 us per layer at 2 GHz
            t[c, l, 5] = top
            t[c, l, 56] = top // 2                          # globaltimer ns
            t[c, l, 8] = top + 4_000                        # first stage 2 us after the top
            t[c, l, 57] = (top + 18_000) // 2               # arrival 9 us after the top
            t[c, l, 59] = (1_000_000 + (l + 1) * 20_000 + 3 * 100 + 18_000) // 2 + 500
            for i in range(12):
                t[c, l, 16 + i] = top + 4_000 + 1_000 * i
                t[c, l, 28 + i] = top + 2_000 + 500 * i
                t[c, l, 40 + i] = top + 3_000 + 1_000 * i
    s = bench.timeline_summary(t)
    assert abs(s["sm_ghz_median"] - ghz) < 1e-6
    assert abs(s["layer_us"]["median"] - 10.0) < 1e-6
    assert abs(s["points_after_consumer_layer_top"]["consumers: first stage landed"]["median_us"]
               - 2.0) < 1e-6
    assert [st["stage"] for st in s["stages"]] == list(range(12))
    assert abs(s["stages"][3]["full_us"] - 3.5) < 1e-6 and abs(s["stages"][3]["issued_us"] - 1.75) < 1e-6


def test_profiled_traffic_scales_by_layers(tmp_path, monkeypatch):
    """A record of bytes per launch of its own layer count gives a run of other layers the same
    bytes per layer; a record on other sources, or of another kernel or workload, gives none."""
    (tmp_path / "profiles").mkdir()
    src = bench.kernel_source_hash()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"kernel=cols_kernel workload=w layers=48 src={src} dram_bytes_per_launch=4800\n"
        f"kernel=cols_kernel workload=old layers=48 src=0000000000000000 dram_bytes_per_launch=1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: src)
    assert bench.profiled_traffic("cols_kernel", "w", 48) == 4800
    assert bench.profiled_traffic("cols_kernel", "w", 6) == 600
    assert bench.profiled_traffic("cols_kernel", "old", 48) is None
    assert bench.profiled_traffic("fused_kernel", "w", 48) is None
