"""bench.py's DRAM-traffic bookkeeping on the host: a traffic line from an ncu
summary is reported only for its kernel and workload key and only while the
sources that decide the GEMMs' traffic still hash to the value it was
captured from."""
import bench


def _profiles(tmp_path, lines):
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "k.md").write_text("summary text\n\n" + "\n".join(lines) + "\n")
    return str(tmp_path)


def test_traffic_line_matches_kernel_workload_and_source(tmp_path, monkeypatch):
    h = "0123456789ab"
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    root = _profiles(tmp_path, [f"traffic tc_bwd_dz small 210150912 src={h}",
                                f"traffic tc_dh_kept small-untiled 209008128 src={h}",
                                "traffic tc_bwd_dh audio40 1870576181 src=000000000000"])
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.recorded_traffic("tc_bwd_dz", "small") == 210150912
    assert bench.recorded_traffic("tc_dh_kept", "small-untiled") == 209008128
    assert bench.recorded_traffic("tc_bwd_dz", "small-untiled") is None
    assert bench.recorded_traffic("tc_bwd_dh", "small") is None
    # captured from other kernel sources: not reported
    assert bench.recorded_traffic("tc_bwd_dh", "audio40") is None


def test_source_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    src = tmp_path / "asr_tiled_tanh_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k_tc.cu").write_text("int f() { return 1; }  // a comment\n")
    (src / "ptx.cuh").write_text("/* header */\n#define X 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (src / "k_tc.cu").write_text("int  f()\n{ return 1; }  // another comment\n")
    assert bench.kernel_source_hash() == h0
    (src / "k_tc.cu").write_text("int f() { return 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_source_hash_covers_the_gemm_sources_only(tmp_path, monkeypatch):
    # k_tc.cu, the headers it includes (transitively) and api.cu decide the
    # GEMMs' traffic; another translation unit does not
    src = tmp_path / "asr_tiled_tanh_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k_tc.cu").write_text('#include "tc.h"\nint f() { return 1; }\n')
    (src / "tc.h").write_text('#include "common.cuh"\n')
    (src / "common.cuh").write_text("constexpr int TT = 32;\n")
    (src / "api.cu").write_text("int plan() { return 0; }\n")
    (src / "k_lattice.cu").write_text("int walk() { return 0; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (src / "k_lattice.cu").write_text("int walk() { return 1; }\n")
    assert bench.kernel_source_hash() == h0
    (src / "common.cuh").write_text("constexpr int TT = 16;\n")
    h1 = bench.kernel_source_hash()
    assert h1 != h0
    (src / "api.cu").write_text("int plan() { return 1; }\n")
    assert bench.kernel_source_hash() != h1

