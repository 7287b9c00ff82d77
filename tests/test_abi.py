"""The C ABI library loads and exports every symbol include/ice.h declares, and
rejects bad arguments on the host (no GPU work is launched by these calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    txt = open(os.path.join(ROOT, "include", "ice.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ice_[a-z_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    from semantic_paged_kv_head_gb300 import build
    build.build_lib()
    from semantic_paged_kv_head_gb300 import ice
    return ice


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert {"ice_build", "ice_insert", "ice_select", "ice_sparse_attn"} <= set(names)
    raw = lib.raw_library()
    for n in names:
        assert hasattr(raw, n), n
    assert sorted(lib.EXPORTS) == names


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.status_string(code) != "unknown status"
    assert lib.status_string(-99) == "unknown status"


def test_host_side_argument_errors(lib):
    raw = lib.raw_library()
    out = ctypes.c_void_p()
    # no parameters / no output handle
    assert raw.ice_build(None, None, None, 0, None, ctypes.byref(out)) == lib.ICE_ERR_INVALID_ARG
    p = lib.ice_params(d=128, n_kv_heads=8, n_q_heads=32, n_layers=1, batch=1, page_size=16,
                       n_proj=8, n_composite=2, n_cand=0, dtype=lib.ICE_BF16, max_tokens=100, seed=0)
    assert raw.ice_build(ctypes.byref(p), None, None, 0, None, None) == lib.ICE_ERR_INVALID_ARG
    bad = [("d", 64, lib.ICE_ERR_UNSUPPORTED), ("n_proj", 4, lib.ICE_ERR_UNSUPPORTED),
           ("page_size", 0, lib.ICE_ERR_INVALID_ARG), ("page_size", 65, lib.ICE_ERR_INVALID_ARG),
           ("n_composite", 3, lib.ICE_ERR_INVALID_ARG), ("n_q_heads", 30, lib.ICE_ERR_INVALID_ARG),
           ("n_q_heads", 24, lib.ICE_ERR_UNSUPPORTED), ("dtype", 7, lib.ICE_ERR_INVALID_ARG),
           ("n_cand", -1, lib.ICE_ERR_INVALID_ARG), ("max_tokens", -1, lib.ICE_ERR_INVALID_ARG),
           ("kv_location", 2, lib.ICE_ERR_INVALID_ARG)]
    for field, val, code in bad:
        q = lib.ice_params.from_buffer_copy(p)
        setattr(q, field, val)
        assert raw.ice_build(ctypes.byref(q), None, None, 0, None, ctypes.byref(out)) == code, field
    # n_tokens beyond the capacity, or keys missing for n > 0
    assert raw.ice_build(ctypes.byref(p), None, None, 101, None, ctypes.byref(out)) == lib.ICE_ERR_INVALID_ARG
    assert raw.ice_build(ctypes.byref(p), None, None, 10, None, ctypes.byref(out)) == lib.ICE_ERR_INVALID_ARG
    # misaligned key pointer
    assert raw.ice_build(ctypes.byref(p), 8, 16, 10, None, ctypes.byref(out)) == lib.ICE_ERR_INVALID_ARG
    # calls on a NULL handle
    assert raw.ice_insert(None, 16, 16, None) == lib.ICE_ERR_INVALID_ARG
    assert raw.ice_select(None, 16, 256, 16, 16, None, None) == lib.ICE_ERR_INVALID_ARG
    assert raw.ice_sparse_attn(None, 16, 16, 16, 16, 16, None) == lib.ICE_ERR_INVALID_ARG
    assert raw.ice_get_error(None, None) == lib.ICE_ERR_INVALID_ARG
    info = lib.ice_info()
    assert raw.ice_get_info(None, ctypes.byref(info)) == lib.ICE_ERR_INVALID_ARG
    raw.ice_destroy(None)  # a no-op


def test_struct_layouts_match_the_header(lib, tmp_path):
    """The ctypes mirrors of ice_params and ice_info have the header's field
    offsets and sizes (compiled with the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    structs = {"ice_params": lib.ice_params, "ice_info": lib.ice_info}
    lines = ['#include <stdio.h>', '#include "ice.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{name} {fname} %zu\\n", offsetof({name}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        name, field, val = line.split()
        got[(name, field)] = int(val)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert got[(name, fname)] == getattr(cls, fname).offset, (name, fname)
