"""Host logic of the bench's profile bookkeeping (CPU only).

The bench reads a per-launch DRAM traffic figure from the committed ncu
summaries under profiles/, and trusts it only while the profiled kernel's code
is unchanged: each summary records a hash of the kernel sources with comments
and blank lines removed.  These tests check that hash input and the parsing of
the summaries' traffic lines.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_profile_hash_ignores_comments_only():
    """The profile summaries' kernel-source hash covers code, not comments: the
    stripped text keeps every code line and drops comment-only and blank lines."""
    import bench
    code = bench.kernel_code("ptx.cuh")
    assert "mbar_init" in code and "cp.async.bulk" in code
    for line in code.splitlines():
        assert line.strip() and not line.lstrip().startswith("//")
    raw = open(os.path.join(ROOT, "q5_lm_head_gb300", "csrc", "ptx.cuh")).read()
    assert len(code) < len(raw)


def test_profile_fields_per_workload_lines(tmp_path):
    """A summary that covers several workloads carries one traffic line per
    workload; each workload reads its own, a plain line serves any workload,
    and a workload the summary does not name reads None."""
    import bench
    multi = tmp_path / "multi.md"
    multi.write_text("# title\nkernel-source: 0123abcd  (hash)\n"
                     "traffic_bytes_per_launch[attn_q]: 111\ntraffic_bytes_per_launch[attn_k]: 222\n")
    assert bench._profile_fields(str(multi), "attn_q") == ("0123abcd", 111)
    assert bench._profile_fields(str(multi), "attn_k") == ("0123abcd", 222)
    assert bench._profile_fields(str(multi), "tiny") == ("0123abcd", None)
    plain = tmp_path / "plain.md"
    plain.write_text("kernel-source: feed\ntraffic_bytes_per_launch: 333\n")
    assert bench._profile_fields(str(plain), "anything") == ("feed", 333)
    assert bench._profiled_traffic("gemm_tc", "no_such_workload") is None
