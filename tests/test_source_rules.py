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
    # the only polling loop on an mbarrier is the helper with an iteration
    # limit; its callers pass the plan's limit (default 2^22, never 0, carried
    # in the ring context) or the drain limit
    waits = [(f, m.start()) for f in SOURCES for m in re.finditer(r"mbarrier\.try_wait", _code(f))]
    assert waits
    f, at = waits[0]
    code = _code(f)
    start = code.rfind("__device__", 0, at)
    end = code.find("__device__", at)
    assert all(g == f and start < a < end for g, a in waits), waits   # all inside one helper
    helper = code[start:at]
    assert re.search(r"bool mbar_wait\([^)]*uint32_t limit, uint32_t hint_ns\)", helper), "the wait takes a limit"
    assert re.search(r"for\s*\(\s*uint32_t\s+i\s*=\s*0\s*;\s*i\s*<\s*limit", helper), "unbounded wait"
    calls = re.findall(r"mbar_wait\(([^;]*)\);", code)
    calls = [c for c in calls if "uint32_t limit" not in c and "uint32_t hint_ns" not in c]
    assert calls
    for c in calls:
        assert re.search(r"(R\.spin_limit, R\.spin_hint_ns|kDrainSpin, 0u)\)?$", c.strip()), c
    assert re.search(r"R\.spin_limit = P\.spin_limit;", code)
    assert re.search(r"constexpr uint32_t kDrainSpin = 1u << \d+;", code)
    api = (CSRC / "ss_api.cu").read_text()
    assert re.search(r"constexpr uint32_t kDefaultSpin = 1u << \d+;", api)
    assert re.search(r"spin_limit = polls == 0 \? kDefaultSpin : polls;", api)
    for g in SOURCES:
        assert not re.search(r"while\s*\(\s*(true|1)\s*\)", _code(g)), g
        assert not re.search(r"for\s*\([^;]*;\s*;", _code(g)), g


def test_single_target_architecture():
    from spec_verification_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-gencode" not in build.flags()[2:]
