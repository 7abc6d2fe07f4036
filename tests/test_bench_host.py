"""Host-side logic of bench.py that needs no GPU: the roofline traffic comes
from a committed ncu summary only while the kernel sources it lists are
unchanged."""
import os

import bench


def _summary(tmp_path, name, traffic, block, sources):
    lines = [f"    traffic_bytes_per_launch = {traffic}", f"    block_size_m = {block}"]
    lines += [f"    source {n} code sha256 = {d}" for n, d in sources]
    (tmp_path / name).write_text("# summary\n\n" + "\n".join(lines) + "\n")


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    (csrc / "k.cu").write_text("kernel v1 // a comment\n")
    digest = bench.code_digest(str(csrc / "k.cu"))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    _summary(tmp_path, "s.md", 123456, 16, [("k.cu", digest)])
    assert bench.profiled_traffic("s.md", 16) == 123456
    assert bench.profiled_traffic("s.md", 128) is None          # another block size
    assert bench.profiled_traffic("missing.md", 16) is None
    (csrc / "k.cu").write_text("kernel  v1 /* another\n comment */\n")  # comments only
    assert bench.profiled_traffic("s.md", 16) == 123456
    (csrc / "k.cu").write_text("kernel v2\n")                     # the kernel changed
    assert bench.profiled_traffic("s.md", 16) is None
    _summary(tmp_path, "t.md", 5, 16, [("gone.cu", digest)])     # a listed source is missing
    assert bench.profiled_traffic("t.md", 16) is None


def test_committed_summaries_parse():
    """Every committed summary that carries a traffic line names its sources."""
    for name in os.listdir(bench.PROFILES):
        text = open(os.path.join(bench.PROFILES, name)).read()
        if "traffic_bytes_per_launch" in text:
            assert "code sha256 =" in text and "block_size_m =" in text, name
