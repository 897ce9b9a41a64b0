"""The C-ABI library: it loads, exports every declared entry point, and
rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import quantized_moe_expert_gb300 as ds4

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ds4moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("ds4moe_create", "ds4moe_route", "ds4moe_forward", "ds4moe_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(ds4.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ds4moe.h but not exported"
        assert name in ds4.SIGNATURES, f"{name} has no binding"


def test_binding_constants_match_the_header():
    import re
    text = open(HEADER).read()

    def macro(name):
        return int(re.search(r"#define\s+" + name + r"\s+(0x[0-9A-Fa-f]+|\d+)u?", text).group(1), 0)
    assert macro("DS4MOE_MAGIC") == ds4.DS4MOE_MAGIC
    assert macro("DS4MOE_VERSION") == ds4.DS4MOE_VERSION
    assert macro("DS4MOE_AUTO_DECODE_MAX_T") == ds4.AUTO_DECODE_MAX_T
    assert macro("DS4MOE_AUTO_BATCH_MAX_T") == ds4.AUTO_BATCH_MAX_T
    assert macro("DS4MOE_BATCH_MAX_T") == ds4.BATCH_MAX_T
    assert macro("DS4MOE_AUTO_MX4_PREFILL_MIN_T") == ds4.AUTO_MX4_PREFILL_MIN_T
    assert macro("DS4MOE_AUTO_VQ_PREFILL_MIN_T") == ds4.AUTO_VQ_PREFILL_MIN_T
    paths = dict(re.findall(r"(DS4MOE_PATH_\w+)\s*=\s*(\d+)", text))
    assert {k: int(v) for k, v in paths.items()} == {
        "DS4MOE_PATH_AUTO": ds4.PATH_AUTO, "DS4MOE_PATH_DECODE": ds4.PATH_DECODE,
        "DS4MOE_PATH_PREFILL": ds4.PATH_PREFILL, "DS4MOE_PATH_BATCH": ds4.PATH_BATCH}
    assert macro("DS4MOE_FLAG_MXFP4") == ds4.FLAG_MXFP4
    # the weights struct the binding passes has the header's fields in order
    body = re.search(r"typedef struct \{([^}]*)\} ds4moe_weights;", text).group(1)
    fields = re.findall(r"\*\s*(\w+);", body)
    assert fields == [f[0] for f in ds4.Weights._fields_]


def test_strerror_names_every_code():
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert ds4.ds4moe_strerror(code) not in ("", "unknown ds4moe error")
    assert ds4.ds4moe_strerror(-99) == "unknown ds4moe error"


def test_create_rejects_bad_descriptions_on_the_host():
    w = ds4.Weights()
    h = ctypes.c_void_p()
    good = dict(hidden=512, inter=256, n_experts=32, top_k=6, shared_inter=256, max_tokens=8)
    bad = [dict(good, hidden=500), dict(good, inter=100), dict(good, n_experts=0), dict(good, top_k=9),
           dict(good, top_k=33), dict(good, shared_inter=32), dict(good, max_tokens=0),
           dict(good, n_experts=2000), dict(good, flags=2)]
    for b in bad:
        d = ds4.make_desc(**b)
        assert ds4._lib.ds4moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == ds4.DS4MOE_EINVAL
    d = ds4.make_desc(**good)
    d.magic = 0
    assert ds4._lib.ds4moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == ds4.DS4MOE_EINVAL
    d = ds4.make_desc(**good)
    for v in (ds4.DS4MOE_VERSION - 1, ds4.DS4MOE_VERSION + 1):
        d.version = v
        assert ds4._lib.ds4moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == ds4.DS4MOE_EINVAL
    # good description, NULL weight pointers
    d = ds4.make_desc(**good)
    assert ds4._lib.ds4moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h)) == ds4.DS4MOE_EINVAL


def test_null_handle_is_rejected():
    assert ds4._lib.ds4moe_forward(None, None, 0, None) == ds4.DS4MOE_EINVAL
    assert ds4._lib.ds4moe_status(None) == ds4.DS4MOE_EINVAL
    assert ds4._lib.ds4moe_destroy(None) == ds4.DS4MOE_OK
