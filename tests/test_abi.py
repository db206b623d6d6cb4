"""The C ABI without a GPU: the library loads, exports every function the
header declares, agrees with the header on constants and struct layout, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mattn.h")


@pytest.fixture(scope="module")
def M():
    from masked_attention_gb300 import _build
    _build.build()
    import masked_attention_gb300 as M
    M.lib()
    return M


def header_text():
    with open(HEADER) as f:
        return f.read()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", header_text(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                 text, flags=re.M)) - {"if", "while", "sizeof"})


def test_exports_every_declared_function(M):
    names = declared_functions()
    assert {"attn_fwd", "attn_bwd", "build_block_mask", "attn_block_mask_bytes",
            "attn_bwd_workspace_bytes", "attn_check_status", "attn_status_str"} <= set(names)
    L = M.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", M.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_constants_match_header(M):
    text = header_text()
    for name, value in (("ATTN_MASK_CAUSAL", M.MASK_CAUSAL), ("ATTN_MASK_WINDOW", M.MASK_WINDOW),
                        ("ATTN_MASK_DOCUMENT", M.MASK_DOCUMENT), ("ATTN_MASK_PREFIX", M.MASK_PREFIX),
                        ("ATTN_SCORE_ALIBI", M.SCORE_ALIBI), ("ATTN_SCORE_SOFTCAP", M.SCORE_SOFTCAP)):
        m = re.search(name + r"\s*=\s*1u\s*<<\s*(\d+)", text)
        assert m and (1 << int(m.group(1))) == value, name
    for name, value in (("ATTN_OK", 0), ("ATTN_ERR_INVALID_ARG", 1), ("ATTN_ERR_UNSUPPORTED", 2),
                        ("ATTN_ERR_MISALIGNED", 3), ("ATTN_ERR_WORKSPACE_TOO_SMALL", 4),
                        ("ATTN_ERR_CUDA", 5), ("ATTN_ERR_TIMEOUT", 6)):
        m = re.search(name + r"\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == value, name


def test_struct_layout_matches_c(M, tmp_path):
    """Compile a C program against the header and compare sizeof/offsetof
    with the ctypes mirrors."""
    fields = {"attn_params": [f for f, _ in M.attn_params._fields_],
              "attn_block_mask": [f for f, _ in M.attn_block_mask._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', 'int main(void){']
    for s, fs in fields.items():
        lines.append(f'printf("{s} %zu\\n", sizeof({s}));')
        for f in fs:
            lines.append(f'printf("{s}.{f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True,
                                                       text=True, check=True).stdout.splitlines())
    for s, cls in (("attn_params", M.attn_params), ("attn_block_mask", M.attn_block_mask)):
        assert int(got[s]) == ctypes.sizeof(cls), s
        for f in fields[s]:
            assert int(got[f"{s}.{f}"]) == getattr(cls, f).offset, f"{s}.{f}"


def test_last_cuda_error_starts_clean(M):
    """No CUDA call has failed on this thread: the name is cudaSuccess."""
    assert M.attn_last_cuda_error() == "cudaSuccess"


def test_status_strings(M):
    for code in range(7):
        assert M.attn_status_str(code)
    assert M.attn_status_str(6) == "device-side wait timed out"


def call_fwd(M, variant=0, D=64, Hq=2, Hkv=2, Sq=128, Skv=128, dtype=0, ptr=0x10000, **kw):
    p = M._params(dtype, kw.get("scale", 0.0), kw.get("window", 0), kw.get("softcap", 0.0), None,
                  kw.get("doc_id"), kw.get("prefix_len"), None, None, 0)
    q = kw.get("q", ptr)
    return M.lib().attn_fwd(q, ptr, ptr, ptr, ptr, 1, Hq, Hkv, Sq, Skv, D, variant,
                            ctypes.byref(p), None)


def test_argument_errors_return_before_launch(M):
    assert call_fwd(M, D=96) == M.ATTN_ERR_UNSUPPORTED
    assert call_fwd(M, Hq=3, Hkv=2) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, variant=1 << 5) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, variant=M.MASK_WINDOW, window=0) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, variant=M.SCORE_SOFTCAP, softcap=0.0) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, variant=M.MASK_DOCUMENT) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, variant=M.MASK_PREFIX) == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, q=0x10008) == M.ATTN_ERR_MISALIGNED
    # the backward takes any length and position offsets, but not a paged cache
    p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0, q_offset=128)
    p.page_table, p.page_size, p.pages_per_seq, p.num_pages = 0x30000, 64, 8, 8
    st = M.lib().attn_bwd(*([0x10000] * 10), 1 << 20, 1, 2, 2, 200, 328, 64, M.MASK_CAUSAL,
                          ctypes.byref(p), None)
    assert st == M.ATTN_ERR_UNSUPPORTED
    # the relative-position bias needs its table, in the backward too
    assert call_fwd(M, variant=M.SCORE_RELBIAS) == M.ATTN_ERR_INVALID_ARG
    p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0)
    st = M.lib().attn_bwd(*([0x10000] * 10), 1 << 20, 1, 2, 2, 128, 128, 64,
                          M.MASK_CAUSAL | M.SCORE_RELBIAS, ctypes.byref(p), None)
    assert st == M.ATTN_ERR_INVALID_ARG
    assert call_fwd(M, dtype=7) == M.ATTN_ERR_UNSUPPORTED
    assert call_fwd(M, scale=float("nan")) == M.ATTN_ERR_INVALID_ARG


def test_offset_and_merge_argument_errors(M):
    """Shards of a longer sequence: negative or overflowing offsets are
    invalid; offsets with the relative-position table, and in the backward,
    are not supported. The merge checks its arguments before any launch."""
    L = M.lib()

    def fwd(variant=0, **kw):
        p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0, rel_bias=kw.get("rb"),
                      q_offset=kw.get("qo", 0), kv_offset=kw.get("ko", 0))
        return L.attn_fwd(*([0x10000] * 5), 1, 2, 2, 128, 128, 64, variant, ctypes.byref(p), None)

    assert fwd(qo=-1) == M.ATTN_ERR_INVALID_ARG
    assert fwd(ko=-5) == M.ATTN_ERR_INVALID_ARG
    assert fwd(qo=2**31 - 100) == M.ATTN_ERR_INVALID_ARG
    assert fwd(M.SCORE_RELBIAS, rb=0x20000, qo=128) == M.ATTN_ERR_UNSUPPORTED
    # document ids: a row length shorter than the absolute positions used
    p = M._params(0, 0.0, 0, 0.0, None, 0x50000, None, None, None, 0, q_offset=64)
    p.doc_len = 150   # needs q_offset + Sq = 192
    st = L.attn_fwd(*([0x10000] * 5), 1, 2, 2, 128, 128, 64, M.MASK_DOCUMENT, ctypes.byref(p),
                    None)
    assert st == M.ATTN_ERR_INVALID_ARG
    # the backward takes offsets, not with the relative-position bias
    p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0, rel_bias=0x20000,
                  kv_offset=128)
    st = L.attn_bwd(*([0x10000] * 10), 1 << 20, 1, 2, 2, 128, 128, 64,
                    M.MASK_CAUSAL | M.SCORE_RELBIAS, ctypes.byref(p), None)
    assert st == M.ATTN_ERR_UNSUPPORTED
    # a block mask built for other offsets does not describe the call
    bm = M.attn_block_mask()
    bm.B, bm.Sq, bm.Skv, bm.nq, bm.nkv, bm.variant = 1, 128, 128, 1, 1, M.MASK_CAUSAL
    bm.full_cnt = bm.part_cnt = bm.full_idx = bm.part_idx = bm.order = 0x30000
    bm.q_offset = 128
    p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0)
    p.block_mask = ctypes.pointer(bm)
    st = L.attn_fwd(*([0x10000] * 5), 1, 2, 2, 128, 128, 64, M.MASK_CAUSAL, ctypes.byref(p), None)
    assert st == M.ATTN_ERR_INVALID_ARG

    def comb(o_parts=0x100000, lse_parts=0x200000, n=2, rows=64, D=128, dtype=0, o=0x300000,
             lse=0x400000):
        return L.attn_combine(o_parts, lse_parts, n, rows, D, dtype, o, lse, None)

    assert comb(n=0) == M.ATTN_ERR_INVALID_ARG
    assert comb(rows=-1) == M.ATTN_ERR_INVALID_ARG
    assert comb(D=96) == M.ATTN_ERR_UNSUPPORTED
    assert comb(dtype=7) == M.ATTN_ERR_UNSUPPORTED
    assert comb(rows=0) == M.ATTN_OK            # nothing to do, nothing launched
    assert comb(o_parts=0) == M.ATTN_ERR_INVALID_ARG
    assert comb(o=0x300008) == M.ATTN_ERR_MISALIGNED
    assert comb(lse=0x400002) == M.ATTN_ERR_MISALIGNED
    # the output may not overlap the parts
    assert comb(o=0x100000 + 256) == M.ATTN_ERR_INVALID_ARG
    assert comb(lse=0x200000 + 64) == M.ATTN_ERR_INVALID_ARG


def test_block_mask_buffer_checks(M):
    L = M.lib()
    p = M._params(0, 0.0, 0, 0.0, None, None, None, None, None, 0)
    out = M.attn_block_mask()
    need = M.attn_block_mask_bytes(2, 1000, 700)
    nq, nkv = 8, 6
    expect = sum(((4 * n + 255) // 256) * 256 for n in (2 * nq, 2 * nq, 2 * nq * nkv,
                                                         2 * nq * nkv, 2 * nq))
    assert need == expect
    assert M.attn_block_mask_bytes(2, 1000, 700, True) > need
    st = L.build_block_mask(M.MASK_CAUSAL, ctypes.byref(p), 2, 1000, 700, 0x100000, need - 1, 0,
                            ctypes.byref(out), None)
    assert st == M.ATTN_ERR_WORKSPACE_TOO_SMALL
    st = L.build_block_mask(M.MASK_CAUSAL, ctypes.byref(p), 2, 1000, 700, 0x100010, need, 0,
                            ctypes.byref(out), None)
    assert st == M.ATTN_ERR_MISALIGNED
    assert M.attn_bwd_workspace_bytes(8, 16, 4096) == 4 * 8 * 16 * 4096
    # the fp16 path: the row terms, a 256-byte range record, then fp16 copies
    # of q, k, v, dO, each 256-byte aligned
    a256 = lambda x: (x + 255) // 256 * 256
    for B, Hq, Hkv, Sq, Skv, D in ((8, 16, 16, 4096, 4096, 128), (2, 32, 8, 640, 384, 64)):
        rows = a256(4 * B * Hq * Sq)
        q = a256(2 * B * Hq * Sq * D)
        k = a256(2 * B * Hkv * Skv * D)
        assert M.attn_bwd_workspace_bytes_f16(B, Hq, Hkv, Sq, Skv, D) == rows + 256 + 2 * q + 2 * k
    assert M.attn_bwd_workspace_bytes_f16(-1, 1, 1, 1, 1, 64) == 0


def test_combine_binding_refuses_strided_views(M):
    """The Python binding passes raw addresses, so a strided view would be
    written as if contiguous: it is refused before the library is called."""
    import torch
    parts = torch.zeros(2, 4, 8, 64)
    lparts = torch.zeros(2, 4, 8)
    o, lse = torch.zeros(4, 16, 64), torch.zeros(4, 16)
    with pytest.raises(ValueError):
        M.attn_combine(parts, lparts, o[:, :8], lse[:, :8])
    with pytest.raises(ValueError):
        M.attn_combine(parts, lparts, torch.zeros(4, 9, 64), torch.zeros(4, 9))
