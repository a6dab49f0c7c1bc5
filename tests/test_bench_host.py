"""Host-side pieces of bench.py that need no GPU.

The roofline's `traffic` figure is valid only for the kernel code it was
captured from: bench.py hashes that code (comments left out) and reports the
figure only while the hash matches the recorded one.
"""

import bench


def test_code_only_drops_comments_and_blank_lines():
    src = ("// header\n"
           "int a = 1;  // trailing\n"
           "\n"
           "/* block\n   comment */ int b = 2;\n"
           "   \n"
           "int c = a /* inline */ + b;\n")
    assert bench._code_only(src) == "int a = 1;\n int b = 2;\nint c = a  + b;"


def test_code_only_keeps_every_code_change():
    base = "int a = 1;\nint b = a + 2;\n"
    assert bench._code_only(base) != bench._code_only(base.replace("a + 2", "a + 3"))
    assert bench._code_only(base) == bench._code_only(base.replace("a + 2;", "a + 2;  // sum"))


def test_traffic_is_reported_only_for_the_recorded_code(monkeypatch):
    recorded = bench.TRAFFIC["sources_sha256"]
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: recorded)
    assert bench.recorded_traffic() == bench.TRAFFIC["bytes_per_launch"] > 0
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda: "0" * 64)
    assert bench.recorded_traffic() is None
