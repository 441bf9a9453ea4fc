"""Host-side pieces of the benchmark that need no GPU: the kernel-source digest
that ties a committed DRAM capture to the kernel code, the traffic lookup and
the L2 note."""
import json

import numpy as np

import bench
import synth


def test_digest_ignores_comments_and_spacing():
    a = "int f(int x) {  // add one\n  return x + 1; /* done */\n}\n"
    b = "int f(int x) {\n\n    return x + 1;\n}  // trailing\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._strip_comments(a) == bench._strip_comments(b)
    assert bench._strip_comments(a) != bench._strip_comments(c)
    # comment markers inside string literals are code
    assert bench._strip_comments('s = "a//b /* c */";') == 's = "a//b /* c */";'
    assert bench._strip_comments('s = "q\\"//x"; // y') == 's = "q\\"//x";'


def test_traffic_record_used_only_for_the_same_kernel_code(tmp_path, monkeypatch):
    digest = bench.kernel_source_digest()
    (tmp_path / "profiles").mkdir()
    rec = {"kernel_source_sha256": digest, "dram_bytes_per_launch": {"w": 1234}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: digest)
    assert bench.load_traffic("w") == 1234
    assert bench.load_traffic("other") is None
    rec["kernel_source_sha256"] = "0" * 64
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w") is None


def test_l2_note_states_whether_inputs_fit():
    big = synth.Problem("big", np.zeros((1, 32, 128), np.uint8), np.zeros((1 << 20, 128), np.uint8),
                        np.zeros((1 << 20, 4), np.uint8), np.zeros((1, 32), np.float32),
                        np.zeros(1, np.int32), np.ones(1, np.int32), 512)
    small = synth.Problem("small", np.zeros((1, 32, 128), np.uint8), np.zeros((4096, 128), np.uint8),
                          np.zeros((4096, 4), np.uint8), np.zeros((1, 32), np.float32),
                          np.zeros(1, np.int32), np.ones(1, np.int32), 512)
    assert bench.l2_note(big).startswith("inputs exceed L2")
    assert "fits in L2" in bench.l2_note(small)
