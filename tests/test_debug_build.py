"""The debug build (libmattn_debug.so, -DMATTN_DEBUG): every kernel checks
the indices of its global loads and stores outside the tensor-map copies,
records one out of range and skips the access, without trapping.

On the CPU: the debug library builds, exports the calls of both headers
(the release library none of the debug ones), and its record struct matches
the header. On the GPU: the check refuses an index planted past a buffer and
records it exactly (attn_debug_selftest, which touches nothing out of
range), and the whole GPU suite, run again on the debug library, leaves the
record empty after every test (tests/conftest.py checks it)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEBUG_HEADER = os.path.join(ROOT, "include", "mattn_debug.h")


def _functions(header):
    with open(header) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text,
                          flags=re.M)) - {"if", "while", "sizeof"}


def _exported(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True).stdout
    return {line.split()[-1] for line in out.splitlines() if " T " in line}


@pytest.fixture(scope="module")
def debug_lib():
    from masked_attention_gb300 import _build
    _build.build()
    return _build.build(debug=True)


def test_debug_library_exports_both_headers(debug_lib):
    from masked_attention_gb300 import _build
    debug_fns = _functions(DEBUG_HEADER)
    assert debug_fns == {"attn_debug_record", "attn_debug_site_name", "attn_debug_selftest"}
    release_fns = _functions(os.path.join(ROOT, "include", "mattn.h"))
    assert release_fns | debug_fns <= _exported(debug_lib)
    assert not debug_fns & _exported(_build.LIB_PATH)


def test_debug_info_layout_matches_c(debug_lib, tmp_path):
    import masked_attention_gb300 as M
    fields = [f for f, _ in M.attn_debug_info._fields_]
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{DEBUG_HEADER}"',
             'int main(void){', 'printf("size %zu\\n", sizeof(attn_debug_info));']
    lines += [f'printf("{f} %zu\\n", offsetof(attn_debug_info, {f}));' for f in fields]
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                       text=True, check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(M.attn_debug_info)
    for f in fields:
        assert int(got[f]) == getattr(M.attn_debug_info, f).offset, f


def _debug_env():
    env = dict(os.environ)
    env["MATTN_DEBUG"] = "1"
    return env


@pytest.mark.gpu
def test_debug_check_refuses_and_records_a_planted_index(debug_lib):
    code = ("import masked_attention_gb300 as M; M.debug_selftest(); "
            "r = M.debug_record(); assert r['count'] == 0, r; print('selftest ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_debug_env(),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "selftest ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
@pytest.mark.skipif(os.environ.get("MATTN_DEBUG", "0") not in ("", "0"),
                    reason="already running on the debug build")
def test_gpu_suite_leaves_debug_record_clean(debug_lib):
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-q", "-x",
           "-p", "no:cacheprovider", "--deselect", "tests/test_debug_build.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=_debug_env(), capture_output=True, text=True,
                       timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    print(tail)
    assert r.returncode == 0, tail
