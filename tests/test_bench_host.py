"""bench.py host logic that needs no GPU: a committed ncu traffic record is reported only while
the kernel sources it names still hash to the recorded value."""
import glob
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CSRC = os.path.join(ROOT, "mixture_experts_routed_logits_gb300", "csrc")


def _hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def test_traffic_record_used_only_while_the_sources_match(tmp_path, monkeypatch):
    rec = tmp_path / "summary.md"
    monkeypatch.setattr(glob, "glob", lambda pattern: [str(rec)])
    files = ["gemv.cu", "common.cuh"]
    line = "traffic-record: kernel=k1 workload=w1 bytes=123456 files=" + ",".join(files)
    rec.write_text("text\n" + line + " src_sha256=" + _hash(files) + "\n")
    assert bench.captured_traffic("k1", "w1") == 123456
    assert bench.captured_traffic("k1", "other") is None
    assert bench.captured_traffic("k2", "w1") is None
    rec.write_text(line + " src_sha256=" + "0" * 64 + "\n")            # the sources changed since
    assert bench.captured_traffic("k1", "w1") is None
    rec.write_text(line.replace("common.cuh", "no_such_file.cu") + " src_sha256=00\n")
    assert bench.captured_traffic("k1", "w1") is None

