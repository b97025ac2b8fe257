"""The suite's size is pinned: a test that disappears (a renamed file, a broken parametrization,
an import error swallowed by a skip) changes the collected count and fails here. Adding tests
means raising the pin."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINNED = 177


def test_collected_count_is_pinned():
    r = subprocess.run([sys.executable, "-m", "pytest", "--collect-only", "-q", "-p", "no:cacheprovider", "tests"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    m = re.search(r"(\d+) tests? collected", r.stdout)
    assert m, r.stdout[-2000:] + r.stderr[-2000:]
    assert int(m.group(1)) == PINNED, f"collected {m.group(1)} tests, pinned {PINNED}"
