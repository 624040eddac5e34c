"""Host-side pieces of bench.py (no GPU): the code digest that keeps a
recorded ncu traffic figure tied to the kernel's code."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_digest_ignores_comments_and_space_but_not_code(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text("// header\nint f(int x) {\n  return x + 1;  // add one\n}\n")
    b.write_text("/* another\n   header */ int f(int x) { return x + 1; }\n")
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b))
    assert bench.code_digest(str(a)) != bench.code_digest(str(c))


def test_traffic_record_is_read_only_for_matching_code():
    # the committed record names its code digest; it is returned only when
    # the current source has that digest, else the bench reports null
    rec = os.path.join(ROOT, "profiles", "gemv_seq_traffic.txt")
    text = open(rec).read()
    digest = bench.code_digest(os.path.join(ROOT, "q4_weight_matmul_gb300", "csrc", "gemv_seq.cu"))
    got = bench.profile_traffic("gemv_seq", "gemv_seq.cu")
    assert (got is not None) == (f"source_sha256_16: {digest}" in text)
    assert bench.profile_traffic("no_such_kernel", "gemv_seq.cu") is None
