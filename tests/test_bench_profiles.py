"""bench.py's reader of the ncu counters recorded under profiles/: a
profile's per-launch values count only while the kernel's sources are the
ones it was captured from (a hash that ignores comments and blank space)."""
import bench


def _write(tmp_path, monkeypatch, kernel, body):
    (tmp_path / "profiles").mkdir(exist_ok=True)
    (tmp_path / "profiles" / f"{kernel}_case.md").write_text(body)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def _sources(tmp_path, kernel, text):
    d = tmp_path / "kv_cache_quantization_hc_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    for name in bench.KERNEL_SOURCES[kernel]:
        (d / name).write_text(text + name)


def test_values_need_the_current_hash(tmp_path, monkeypatch):
    _sources(tmp_path, "k_crc32", "int f(int x) { return x + 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("k_crc32")
    body = f"capture: one launch\nsource_sha256: {h}\nalu_warp_instructions_per_launch: 1234\n"
    _write(tmp_path, monkeypatch, "k_crc32", body)
    v = bench.profiled_values("k_crc32", "case", ("alu_warp_instructions_per_launch",))
    assert v["alu_warp_instructions_per_launch"] == 1234 and v["capture"] == "one launch"
    _write(tmp_path, monkeypatch, "k_crc32", body.replace(h, "0" * 16))
    assert bench.profiled_values("k_crc32", "case", ("alu_warp_instructions_per_launch",)) is None
    _write(tmp_path, monkeypatch, "k_crc32", f"source_sha256: {h}\n")      # value missing
    assert bench.profiled_values("k_crc32", "case", ("alu_warp_instructions_per_launch",)) is None


def test_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _sources(tmp_path, "k_fetch", "int f(int x) { return x + 1; }\n")
    h0 = bench.kernel_source_hash("k_fetch")
    _sources(tmp_path, "k_fetch", "// a note\nint f(int x) {  /* why */ return x + 1; }\n\n")
    assert bench.kernel_source_hash("k_fetch") == h0
    _sources(tmp_path, "k_fetch", "int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash("k_fetch") != h0


def test_crc_alu_roofline(monkeypatch):
    """The CRC's roofline against the integer ALU: recorded ALU-pipe warp
    instructions x 32 over the live time, against SMs x 64 lanes x 2070 MHz;
    only for the launch the count was recorded on."""
    from types import SimpleNamespace
    monkeypatch.setattr(bench, "profiled_values", lambda k, w, keys: {
        "alu_warp_instructions_per_launch": 350_000_000, "units_per_launch": 36 * 2048,
        "capture": "c", "source": "s"})
    r = bench.crc_alu_roofline(SimpleNamespace(L=36, nb=2048, wire_name="fp8"), 0.7e-3, 152)
    assert r["bound"] == "alu" and abs(r["peak"] - 152 * 64 * 2.07e9 / 1e12) < 1e-9
    assert abs(r["achieved"] - 350e6 * 32 / 0.7e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert bench.crc_alu_roofline(SimpleNamespace(L=4, nb=2048, wire_name="fp8"), 0.7e-3, 152) is None
    assert bench.crc_alu_roofline(SimpleNamespace(L=36, nb=2048, wire_name="int4"), 0.7e-3, 152) is None
