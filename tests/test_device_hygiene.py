"""Device-code rules, checked on the sources (CPU).

Every mbarrier wait in the kernels is bounded: the only place that polls an
mbarrier is the bounded wait of `fa_device_common.cuh`, which gives up after
the kernel's cycle limit, records a timeout and returns false. No kernel
traps or asserts on the device: failures come back as status codes.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_87_gb300", "csrc")


def _sources():
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            text = open(os.path.join(CSRC, f)).read()
            # drop comments so that prose does not count
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            yield f, text


def test_no_trap_or_device_assert():
    for f, text in _sources():
        assert "__trap" not in text, f
        assert "trap;" not in text, f
        assert not re.search(r"(?<![\w_])assert\s*\(", text), f"{f}: device assert"


def test_mbarrier_polled_only_by_the_bounded_wait():
    callers = {f for f, text in _sources() if re.search(r"\bmbar_try_wait\s*\(", text)}
    assert callers == {"sm103_ptx.cuh", "fa_device_common.cuh"}, callers
    common = dict(_sources())["fa_device_common.cuh"]
    # the one polling loop compares the elapsed clock against the wait limit
    loops = re.findall(r"while \(true\) \{(.*?)\n  \}", common, flags=re.S)
    assert len(loops) == 1
    assert "mbar_try_wait" in loops[0] and "clock64()" in loops[0] and "wait_limit" in loops[0]
    assert "record_timeout" in loops[0]


def test_no_other_unbounded_loops():
    for f, text in _sources():
        n = len(re.findall(r"while \(true\)|for \(;;\)", text))
        assert n == (1 if f == "fa_device_common.cuh" else 0), f
