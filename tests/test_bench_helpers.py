"""Host-side helpers of bench.py that decide what the bench line reports (no GPU).

The `traffic` figure of the bench line comes from profiles/traffic.json only while the code digest of
the kernel sources equals the one the DRAM counters were taken on.  That digest must ignore comments and
layout, and change with any code token, a string literal's content included.
"""
import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


SRC = '''// header comment
#include "a.h"   /* trailing */
constexpr int kA = 512 + 16;  // a constant
__device__ void f() {
  asm volatile("cp.async.bulk.commit_group; // not a comment" ::: "memory");
  const char c = '/';   /* a block
                           comment over lines */
  int x = 1 /* inline */ + 2;
}
'''


def test_comments_and_layout_are_ignored():
    b = _bench()
    s = b.strip_comments(SRC)
    assert "header comment" not in s and "trailing" not in s and "inline" not in s and "block" not in s
    reflowed = SRC.replace("constexpr int kA = 512 + 16;", "constexpr int kA =\n    512 + 16;")
    recommented = SRC.replace("// a constant", "// another remark").replace("/* inline */", "")
    assert b.strip_comments(reflowed) == s
    assert b.strip_comments(recommented) == s


def test_code_and_literals_count():
    b = _bench()
    s = b.strip_comments(SRC)
    # a "//" inside a string literal is code, and so is the character literal '/'
    assert '"cp.async.bulk.commit_group; // not a comment"' in s
    assert "'/'" in s
    for old, new in [("512 + 16", "512 + 32"), ("commit_group;", "commit_group ;"), ("x = 1", "x = 3"),
                     ("not a comment", "not a remark")]:
        assert b.strip_comments(SRC.replace(old, new)) != s, f"changing {old!r} went unnoticed"


def test_traffic_lookup_follows_the_code_digest(tmp_path, monkeypatch):
    b = _bench()
    files = ["flce_fwd.cu", "flce_bwd.cu", "sm100.cuh"]
    digest = b.kernel_source_digest(files)
    assert len(digest) == 16
    # an entry under another digest is not reported; one under this digest is
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(
        '{"long": {"k": {"dram_bytes_per_launch": 7, "source_digest": "%s"}, '
        '"old": {"dram_bytes_per_launch": 9, "source_digest": "0000000000000000"}}}' % digest)
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    assert b.dram_traffic("k", "long", digest) == 7
    assert b.dram_traffic("old", "long", digest) is None
    assert b.dram_traffic("missing", "long", digest) is None
