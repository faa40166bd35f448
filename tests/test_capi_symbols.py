"""librimuru.so loads without a GPU and exports every entry point include/rimuru.h declares."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "rimuru.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rimuru_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_named_entry_points():
    names = declared_functions()
    for required in ("rimuru_pool_create", "rimuru_view_create", "rimuru_expert_map",
                     "rimuru_moe_forward"):
        assert required in names


def test_library_exports_every_declared_symbol():
    from paged_moe_shared_gb300 import rimuru as R
    lib = ctypes.CDLL(R.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []
    assert sorted(R.EXPORTS) == declared_functions()


def test_status_strings():
    from paged_moe_shared_gb300 import rimuru as R
    assert R.rimuru_status_string(0) == "RIMURU_OK"
    assert R.rimuru_status_string(-4) == "RIMURU_ERR_UNMAPPED"
    assert R.rimuru_kernel_name(R.K_GEMM1) == "moe_gemm1_swiglu"
    assert R.rimuru_kernel_name(R.K_COUNT) is None
    assert R.rimuru_kernel_name(99) is None


def test_kernel_slot_numbers_match_the_header():
    """The binding's K_* constants are the header's RIMURU_K_* enumerators."""
    from paged_moe_shared_gb300 import rimuru as R
    text = open(os.path.join(ROOT, "include", "rimuru.h")).read()
    slots = dict((m, int(v)) for m, v in re.findall(r"RIMURU_K_([A-Z0-9_]+)\s*=\s*(\d+)", text))
    assert slots == {name: getattr(R, "K_" + name) for name in slots}
    assert slots["COUNT"] == max(v for k, v in slots.items() if k != "COUNT") + 1


def test_selftest_rejects_bad_limits_before_touching_a_device():
    import pytest
    from paged_moe_shared_gb300 import rimuru as R
    for bad in (0, 3_000_000):
        with pytest.raises(R.RimuruError) as e:
            R.rimuru_selftest_bounded_wait(bad)
        assert e.value.status == R.ERR_ARG


def header_struct_members(name):
    """(type, member) pairs of `typedef struct <name> { ... } <name>;` in the header."""
    text = open(os.path.join(ROOT, "include", "rimuru.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef struct " + name + r"\s*\{(.*?)\}\s*" + name + r"\s*;", text, re.S)
    assert body, name
    return re.findall(r"\b(u?int(?:32|64)_t)\s+([a-z_0-9]+)\s*;", body.group(1))


def test_binding_structs_match_the_header():
    """The ctypes structures of the binding list the header's members in order, with the
    same integer widths and signedness."""
    import ctypes
    from paged_moe_shared_gb300 import rimuru as R
    ctype = {"uint64_t": ctypes.c_uint64, "int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32,
             "uint32_t": ctypes.c_uint32}
    for cname, cls in (("rimuru_level_stats", R.LevelStats), ("rimuru_ws_layout", R.WsLayout),
                       ("rimuru_offload_counters", R.OffloadCounters)):
        members = header_struct_members(cname)
        assert [(n, ctype[t]) for t, n in members] == list(cls._fields_), cname


def header_prototypes():
    """name -> (return type, [parameter types]) for every function the header declares."""
    text = open(os.path.join(ROOT, "include", "rimuru.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for ret, name, params in re.findall(r"([A-Za-z_][A-Za-z_0-9 ]*?\**)\s*\b(rimuru_[a-z0-9_]+)\s*\(([^)]*)\)\s*;",
                                        text):
        types = []
        for p in params.split(","):
            p = p.strip()
            if p in ("", "void"):
                continue
            types.append(re.sub(r"\s*\b[a-z_0-9]+$", "", p) if not p.endswith("*") else p)
        protos[name] = (ret.strip(), types)
    return protos


def test_binding_signatures_match_the_header():
    """Every entry point's argument and result types in the binding agree with its C
    prototype: pointers and handles as pointers, and integers of the same width and sign."""
    import ctypes
    from paged_moe_shared_gb300 import rimuru as R
    ints = {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64,
            "uint64_t": ctypes.c_uint64, "uint32_t": ctypes.c_uint32, "double": ctypes.c_double}

    def agrees(ctype_str, ct):
        c = ctype_str.replace("const ", "").strip()
        if c.endswith("*") or c.endswith("_t") and c.startswith("rimuru_"):
            return ct in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(ct, "_type_") and \
                issubclass(ct, ctypes._Pointer)
        return ct is ints[c]

    protos = header_prototypes()
    assert len(protos) == len(R.EXPORTS)
    for name, (ret, params) in protos.items():
        fn = getattr(R.lib, name)
        assert len(fn.argtypes) == len(params), (name, params, fn.argtypes)
        for c, ct in zip(params, fn.argtypes):
            assert agrees(c, ct), (name, c, ct)
        assert agrees(ret, fn.restype), (name, ret, fn.restype)
