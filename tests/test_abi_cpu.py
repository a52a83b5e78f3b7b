"""CPU checks of the C ABI: the library builds, loads, exports every entry
point declared in include/dcoco.h, and rejects bad arguments before any CUDA
call (so these run without a GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_correction_slot_gb300 as dc
    return dc


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(dcoco_[a-z_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(dc):
    names = declared_functions()
    assert {"dcoco_create", "dcoco_correct", "dcoco_topk", "dcoco_destroy"} <= names
    lib = C.CDLL(dc.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared but not exported"
    # the Python binding exposes the same names
    for n in names:
        assert callable(getattr(dc, n)), n


def test_version_and_status_strings(dc):
    assert dc.dcoco_version() >= 100
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert dc.dcoco_status_string(s) != "unknown status"
    assert dc.dcoco_status_string(-99) == "unknown status"


@pytest.mark.parametrize("kw,status", [
    (dict(topk=12), -2), (dict(topk=64), -2), (dict(rank=64), -2), (dict(mlp_hidden=512), -2),
    (dict(variant=2), -2), (dict(slots=2), -2), (dict(slots=40), -2), (dict(path_rule=3), -2), (dict(path_rule=2, beam_width=0), -2),
    (dict(path_rule=2, beam_width=5), -2), (dict(path_rule=2, beam_topm=17), -2),
    (dict(hidden=4000), -1), (dict(hidden=0), -1), (dict(vocab=8), -1),
    (dict(max_batch=0), -1), (dict(ln_eps=0.0), -1), (dict(vocab=1 << 21), -1),
])
def test_create_rejects_bad_config_without_cuda(dc, kw, status):
    args = dict(vocab=151936, hidden=4096)
    args.update(kw)
    with pytest.raises(dc.DcocoError) as e:
        dc.dcoco_create(**args)
    assert e.value.status == status


def test_null_arguments_rejected(dc):
    lib = C.CDLL(dc.LIB_PATH)
    lib.dcoco_create.argtypes = [C.c_void_p, C.c_void_p]
    assert lib.dcoco_create(None, None) == -1
    assert lib.dcoco_get_device_status(None) == -1
    lib.dcoco_correct.argtypes = [C.c_void_p] * 2 + [C.c_int] + [C.c_void_p] * 3
    assert lib.dcoco_correct(None, None, 1, None, None, None) == -1
    lib.dcoco_topk.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_int64, C.c_void_p, C.c_void_p,
                               C.c_void_p]
    assert lib.dcoco_topk(None, 1, None, 0, None, None, None) == -1
    lib.dcoco_selftest_wait_timeout.argtypes = [C.c_void_p, C.c_longlong, C.c_void_p]
    assert lib.dcoco_selftest_wait_timeout(None, 1_000_000, None) == -1
    lib.dcoco_destroy.argtypes = [C.c_void_p]
    lib.dcoco_destroy(None)  # NULL is allowed
    lib.dcoco_weights_destroy.argtypes = [C.c_void_p]
    lib.dcoco_weights_destroy(None)


def test_library_never_loads_the_oracle(dc):
    """The product path has no route to the CPU oracle."""
    pkg = os.path.join(ROOT, "draft_correction_slot_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in re.sub(r"#.*|//.*", "", src).replace("oracle's", ""), fn


def test_host_range_predicate(dc):
    """dcoco_correct_host reads host logits in place only when the page-locked
    range the driver reports holds the whole extent the top-K reads."""
    f = dc.dcoco_host_range_covers
    base, size = 0x10000, 0x8000
    assert f(base, size, base, size)                 # the whole range
    assert f(base, size, base + 0x100, size - 0x100)  # ends exactly at the range end
    assert not f(base, size, base + 0x100, size - 0xFF)  # one byte past the end
    assert not f(base, size, base - 16, 32)          # starts before the range
    assert not f(base, size, base + size, 16)        # starts at the end
    assert f(base, size, base + size, 0)             # empty extent at the end
    assert not f(base, 0, base, 0)                   # no range
    assert not f(0, 2**64 - 1, 2**63, 2**63 + 1)     # no wrap-around
