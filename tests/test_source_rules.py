"""Source rules for the CUDA kernels that need no GPU to check: every spin-wait
loop is bounded by the global timer, and no kernel traps on purpose."""
import glob
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_draft_round_gb300", "csrc")


def _sources():
    files = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")))
    assert files
    return [(os.path.basename(f), open(f, encoding="utf-8").read().splitlines()) for f in files]


def test_every_spin_wait_is_bounded_by_the_timer():
    spin = re.compile(r"while\s*\(\s*(true|1|!\s*mbar_try_wait\()")
    loops, unbounded = 0, []
    for name, lines in _sources():
        for i, line in enumerate(lines):
            if spin.search(line):
                loops += 1
                window = "\n".join(lines[i:i + 8])
                if "globaltimer()" not in window:
                    unbounded.append("%s:%d" % (name, i + 1))
    assert loops > 0
    assert unbounded == []


def test_no_kernel_traps():
    hits = ["%s:%d" % (name, i + 1) for name, lines in _sources() for i, line in enumerate(lines)
            if re.search(r"__trap\s*\(|\btrap;|\bbrkpt\b", line)]
    assert hits == []
