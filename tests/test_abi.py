"""CPU-side checks of the C ABI: the library builds, loads and exports every
function include/ss.h declares; the Python binding's struct layouts match the
header's field lists; the oracle is never reachable from the product package."""
import ast
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "ss.h"


def header_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(ss_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from spec_verification_gb300 import build
    path = build.build()
    return ctypes.CDLL(str(path))


def test_library_exports_every_header_function(lib):
    names = header_functions()
    assert {"ss_sample", "ss_verify", "ss_plan_create", "ss_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    from spec_verification_gb300 import native
    assert set(native.EXPORTS) == set(names)


def test_struct_layouts_match_header():
    from spec_verification_gb300 import native
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)

    def fields(struct):
        body = re.search(r"typedef struct \{([^{}]*)\}\s*" + struct + ";", text, flags=re.S).group(1)
        out = []
        for decl in body.split(";"):
            toks = [t for t in decl.replace("*", " ").replace(",", " ").split() if t != "const"]
            if not toks:
                continue
            out += toks[1:]
        return out

    assert fields("ss_batch") == [f for f, _ in native.Batch._fields_]
    assert fields("ss_out") == [f for f, _ in native.Out._fields_]
    assert fields("ss_row_params") == list(native.ROW_DTYPE.names)
    assert fields("ss_bias_entry") == list(native.BIAS_DTYPE.names)


def test_flag_values_agree():
    from spec_verification_gb300 import native
    from spec_verification_gb300 import workloads as W
    text = HEADER.read_text()
    for name, val in [("SS_GREEDY", W.GREEDY), ("SS_MASK", W.MASK), ("SS_PENALTY", W.PENALTY),
                      ("SS_BIAS", W.BIAS), ("SS_TOPK", W.TOPK), ("SS_TOPP", W.TOPP), ("SS_MINP", W.MINP),
                      ("SS_BOUNDED_P", W.BOUNDED_P), ("SS_EXACT", W.EXACT)]:
        m = re.search(name + r" = 1u << (\d+)", text)
        assert m and (1 << int(m.group(1))) == val, name
    m = re.search(r"SS_ST_CAPACITY = 1u << (\d+)", text)
    assert m and (1 << int(m.group(1))) == native.ST_CAPACITY


def test_plan_create_without_gpu_reports_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from spec_verification_gb300 import native
    with pytest.raises(native.SSError):
        native.Plan(1000, 4)


def test_product_package_never_imports_oracle():
    pkg = ROOT / "spec_verification_gb300"
    for f in pkg.rglob("*.py"):
        tree = ast.parse(f.read_text())
        for node in ast.walk(tree):
            if isinstance(node, ast.Import):
                assert not any(a.name.split(".")[0] == "oracle" for a in node.names), f
            if isinstance(node, ast.ImportFrom):
                assert (node.module or "").split(".")[0] != "oracle", f
    for f in (pkg / "csrc").glob("*"):
        assert not re.search(r"\bsso_|oracle/|liboracle", f.read_text()), f


def test_host_side_misuse_returns_negative_codes(lib):
    """Arguments the host can check are refused before any device query or
    launch, with the header's negative status codes."""
    import ctypes as C
    from spec_verification_gb300 import native
    L = native.library()
    ERR_ARG, ERR_UNSUPPORTED = -1, -3
    p = C.c_void_p(12345)

    def create(V=1000, rows=4, positions=8, ldt=0, qdt=0, tile=0):
        p.value = 12345
        return L.ss_plan_create(C.byref(p), V, rows, positions, ldt, qdt, tile, 0)

    for kw, code in [({"V": 0}, ERR_UNSUPPORTED), ({"V": (1 << 20) + 1}, ERR_UNSUPPORTED),
                     ({"rows": 0}, ERR_ARG), ({"positions": 3}, ERR_ARG),
                     ({"positions": (1 << 24) + 1}, ERR_ARG), ({"ldt": 7}, ERR_ARG),
                     ({"qdt": -1}, ERR_ARG), ({"tile": 4096}, ERR_UNSUPPORTED)]:
        assert create(**kw) == code, kw
        assert p.value is None, kw          # *plan is NULL on failure
        assert L.ss_last_error()             # and the reason is recorded
    assert L.ss_plan_create(None, 1000, 4, 8, 0, 0, 0, 0) == ERR_ARG
    # calls without params, out or plan
    out = native.Out()
    batch = native.Batch()
    assert L.ss_sample(None, None, None, None, None, None, C.byref(out)) == ERR_ARG
    assert L.ss_sample(None, C.byref(batch), None, None, None, None, None) == ERR_ARG
    assert L.ss_sample(None, C.byref(batch), None, None, None, None, C.byref(out)) == ERR_ARG
    assert L.ss_verify(None, None, None, C.byref(batch), None, C.byref(out)) == ERR_ARG
    assert L.ss_sample_noalloc(None, C.byref(batch), None, None, None, None, C.byref(out)) == ERR_ARG
    assert L.ss_plan_enable_exact(None, 1) == ERR_ARG
    # plan queries on NULL
    assert L.ss_workspace_bytes(None) == 0 and L.ss_plan_tile(None) == 0
    assert L.ss_plan_num_tiles(None) == 0 and L.ss_plan_stage1_ctas(None) == 0
    L.ss_plan_destroy(None)
    for code, text in [(0, b"ok"), (-1, b"invalid argument"), (-2, b"misaligned row"),
                       (-3, b"unsupported size"), (-4, b"workspace too small"), (-5, b"CUDA error"),
                       (42, b"unknown status")]:
        assert L.ss_status_str(code) == text
