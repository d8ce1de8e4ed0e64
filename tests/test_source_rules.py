"""Static checks of the CUDA sources: no construct that stops a GPU on
purpose, every mbarrier wait bounded, one target architecture."""
import re
from pathlib import Path

CSRC = Path(__file__).resolve().parents[1] / "spec_verification_gb300" / "csrc"
SOURCES = sorted(list(CSRC.glob("*.cu")) + list(CSRC.glob("*.cuh")))


def _code(path):
    text = path.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def test_no_trap_or_device_assert():
    assert SOURCES
    for f in SOURCES:
        code = _code(f)
        assert "__trap" not in code, f
        assert not re.search(r"\btrap\s*;", code), f          # inline PTX trap
        assert not re.search(r"\bassert\s*\(", code), f        # device assert
        assert "__brkpt" not in code, f


def test_every_mbarrier_wait_is_bounded():
    # the only polling loop on an mbarrier is the helper with an iteration limit
    waits = [(f, m.start()) for f in SOURCES for m in re.finditer(r"mbarrier\.try_wait", _code(f))]
    assert len(waits) == 1, waits
    f, at = waits[0]
    code = _code(f)
    helper = code[code.rfind("__device__", 0, at):at]
    assert re.search(r"for\s*\(\s*int\s+i\s*=\s*0\s*;\s*i\s*<\s*kSpinLimit", helper), "unbounded wait"
    assert re.search(r"constexpr int kSpinLimit = 1 << \d+;", code)
    for g in SOURCES:
        assert not re.search(r"while\s*\(\s*(true|1)\s*\)", _code(g)), g
        assert not re.search(r"for\s*\(\s*;\s*;\s*\)", _code(g)), g


def test_single_target_architecture():
    from spec_verification_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-gencode" not in build.flags()[2:]
