"""Host-side helpers of the benchmark (CPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def test_kernel_hash_ignores_comments_only():
    """The bench keys its ncu traffic figure by the kernel sources' code: a
    comment or blank-space edit keeps the key, a code edit changes it, and
    string literals (inline PTX) count as code."""
    import bench

    src = 'asm("mov.b32 %0, %1; // not a comment");  // a comment\nint x = 1; /* block */\n'
    same = 'asm("mov.b32 %0, %1; // not a comment");\n\n   int x = 1;\n'
    assert bench.strip_comments(src) == bench.strip_comments(same)
    assert bench.strip_comments(src) != bench.strip_comments(src.replace("x = 1", "x = 2"))
    assert "// not a comment" in bench.strip_comments(src)
