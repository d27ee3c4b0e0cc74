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


def test_both_bench_arms_name_the_same_workload():
    from mixture_experts_routed_logits_gb300 import synth
    names = {bench.workload_name(synth.CONFIGS[c], t) for c, t in [(2, 8)] + bench.PER_CONFIG}
    assert len(names) == 1 + len(bench.PER_CONFIG)
    assert bench.workload_name(synth.CONFIGS[2], 8) == "gptoss_decode_T8_H2880_E32_k4_mxfp4"
    assert bench.workload_name(synth.CONFIGS[3], 512) == "gptoss_prefill_T512_H2880_E32_k4_mxfp4_skew"
    src = open(bench.__file__).read()
    # the reference arm labels its line with the same function as the measured arm
    assert src.count("workload_name(c, T)") == 1 and "workload_name(cfg, T)" in src


def test_dtype_label_names_the_path_arithmetic():
    from mixture_experts_routed_logits_gb300 import synth
    assert "e2m1" in bench.dtype_label(synth.CONFIGS[2], False)
    assert "mma.sync" in bench.dtype_label(synth.CONFIGS[2], False)
    assert "tcgen05" in bench.dtype_label(synth.CONFIGS[5], True)
    assert "int4" in bench.dtype_label(synth.CONFIGS[4], False)
