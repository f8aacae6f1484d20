"""The C ABI without a GPU: the library builds, loads, exports every entry
point include/mhc_boundary.h declares, its structs have the same layout as
the binding's, and host-side checks answer without touching a device."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mhc_boundary.h")


@pytest.fixture(scope="session")
def capi():
    from mhc_residual_boundary_gb300 import build
    build.build()
    from mhc_residual_boundary_gb300 import capi as c
    c.lib()
    return c


def declared_functions():
    import glob
    text = "\n".join(open(h).read() for h in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mhc_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(capi):
    names = declared_functions()
    assert {"mhc_boundary_create", "mhc_boundary_run", "mhc_boundary_finalize_moe",
            "mhc_boundary_join", "mhc_boundary_destroy", "mhc_mxfp8_scale_bytes",
            "mhc_status_string", "mhc_last_error"} <= set(names)
    lib = capi.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (mhc_\w+)", out))
    assert set(names) <= exported


def test_struct_layouts_match_the_header(capi, tmp_path):
    checks = {
        "mhc_boundary_config_t": capi.mhc_boundary_config_t,
        "mhc_run_args_t": capi.mhc_run_args_t,
        "mhc_moe_args_t": capi.mhc_moe_args_t,
        "mhc_consume_args_t": capi.mhc_consume_args_t,
        "mhc_profile_t": capi.mhc_profile_t,
    }
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "mhc_boundary.h"', "int main(void) {"]
    for cname, ctype in checks.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in ctype._fields_:
            lines.append(f'printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for line in filter(None, got):
        cname, field, value = line.split()
        ctype = checks[cname]
        expect = ctypes.sizeof(ctype) if field == "size" else getattr(ctype, field).offset
        assert int(value) == expect, line


def test_scale_bytes_and_status_strings(capi, oracle_lib):
    for m, h in ((1, 128), (127, 256), (128, 6144), (4096, 6144), (300, 512), (5, 5120)):
        assert capi.mhc_mxfp8_scale_bytes(m, h) == oracle_lib.mxfp8_scale_bytes(m, h)
    assert capi.mhc_mxfp8_scale_bytes(0, 128) == 0
    assert capi.mhc_mxfp8_scale_bytes(4, 100) == 0
    for s in range(7):
        assert capi.mhc_status_string(s)
    assert capi.mhc_status_string(99) == "unknown status"


@pytest.mark.parametrize("field,value,status", [
    ("hc_mult", 3, "MHC_ERR_UNSUPPORTED"), ("hidden", 12, "MHC_ERR_INVALID_ARG"),
    ("hidden", 32768, "MHC_ERR_UNSUPPORTED"), ("tp", 0, "MHC_ERR_INVALID_ARG"),
    ("max_num_tokens", 0, "MHC_ERR_INVALID_ARG"), ("sinkhorn_repeat", 0, "MHC_ERR_INVALID_ARG"),
    ("top_k", 65, "MHC_ERR_INVALID_ARG"), ("flags", 1 << 7, "MHC_ERR_INVALID_ARG"),
])
def test_create_rejects_bad_config(capi, field, value, status):
    cfg = capi.mhc_boundary_config_t(6144, 4, 4, 256, 20, 8, 1e-6, 1e-6, 2.0, 1e-6, 0)
    setattr(cfg, field, value)
    with pytest.raises(capi.MhcError, match=status):
        capi.mhc_boundary_create(cfg, 0)
    assert capi.mhc_last_error(None)


def test_mxfp8_needs_hidden_multiple_of_128(capi):
    cfg = capi.mhc_boundary_config_t(5000, 4, 4, 16, 20, 0, 1e-6, 1e-6, 2.0, 1e-6, capi.MHC_FLAG_MXFP8)
    with pytest.raises(capi.MhcError, match="INVALID_ARG"):
        capi.mhc_boundary_create(cfg, 0)


def test_null_handle_calls_fail_cleanly(capi):
    lib = capi.lib()
    assert lib.mhc_boundary_run(None, None, None) == 1
    assert lib.mhc_boundary_join(None, None) == 1
    assert lib.mhc_boundary_destroy(None) == 0
    assert lib.mhc_boundary_launches_per_call(None) == 0


def test_flag_values_match_the_header(capi):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    declared = {name: 1 << int(bit) for name, bit in re.findall(r"\b(MHC_FLAG_[A-Z0-9_]+)\s*=\s*1u\s*<<\s*(\d+)", text)}
    assert declared, "no flags found in the header"
    bound = {name: getattr(capi, name) for name in dir(capi) if name.startswith("MHC_FLAG_")}
    assert declared == bound


def _static_args(capi, m=4):
    # fake, 16-byte aligned device addresses: every case below is refused by
    # the host-side checks, before the first CUDA call, so none is dereferenced
    a = capi.mhc_run_args_t()
    a.m = m
    for i, f in enumerate(("partials", "residual", "post", "comb", "hc_fn", "scale", "base", "norm_weight",
                           "residual_out", "layer_input", "post_out", "comb_out")):
        setattr(a, f, 0x10000 * (i + 1))
    return a


def _static(capi, cfg, a):
    import ctypes
    err = ctypes.create_string_buffer(512)
    status = capi.lib().mhc_boundary_run_static(ctypes.byref(cfg), ctypes.byref(a), None, err, len(err))
    return capi.STATUS[status], err.value.decode()


@pytest.mark.parametrize("case,status,text", [
    ("hidden", "MHC_ERR_INVALID_ARG", "hidden must be a positive multiple of 8"),
    ("owner_flag", "MHC_ERR_UNSUPPORTED", "only MHC_FLAG_MXFP8"),
    ("m0", "MHC_ERR_CAPACITY", "outside [1, 865]"),
    ("m_big", "MHC_ERR_CAPACITY", "outside [1, 865]"),
    ("null", "MHC_ERR_INVALID_ARG", "partials is NULL"),
    ("misaligned", "MHC_ERR_INVALID_ARG", "residual is not 16-byte aligned"),
    ("two_weights", "MHC_ERR_INVALID_ARG", "exactly one of hc_fn and hc_fn_bf16"),
    ("mx_half", "MHC_ERR_INVALID_ARG", "mxfp8_values and mxfp8_scales go together"),
    ("mx_no_flag", "MHC_ERR_UNSUPPORTED", "MXFP8 outputs need MHC_FLAG_MXFP8"),
])
def test_static_entry_refuses_before_any_launch(capi, case, status, text):
    cfg = capi.mhc_boundary_config_t(6144, 4, 4, 0, 20, 0, 1e-6, 1e-6, 2.0, 1e-6, 0)
    a = _static_args(capi)
    if case == "hidden":
        cfg.hidden = 6140
    elif case == "owner_flag":
        cfg.flags = capi.MHC_FLAG_OWNER_REDUCE
    elif case == "m0":
        a.m = 0
    elif case == "m_big":
        a.m = 866      # the 8 MiB scratch holds 865 tokens at H = 6144
    elif case == "null":
        a.partials = None
    elif case == "misaligned":
        a.residual += 8
    elif case == "two_weights":
        a.hc_fn_bf16 = 0x900000
    elif case == "mx_half":
        a.mxfp8_values = 0x900000
    elif case == "mx_no_flag":
        a.mxfp8_values, a.mxfp8_scales = 0x900000, 0xA00000
    got_status, got_text = _static(capi, cfg, a)
    assert got_status == status and text in got_text, (got_status, got_text)


def test_missing_library_fails_loudly(tmp_path):
    # a fresh interpreter whose binding points at a library that was never
    # built: the first use raises, and nothing falls back to a CPU path
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from mhc_residual_boundary_gb300 import capi\n"
        "capi.LIB_PATH = %r\n"
        "try:\n"
        "    capi.mhc_mxfp8_scale_bytes(128, 256)\n"
        "except ImportError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('no error')\n" % (ROOT, str(tmp_path / "libmhc_boundary.so")))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.startswith("raised:") and "no fallback" in out.stdout
