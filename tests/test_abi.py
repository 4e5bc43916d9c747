"""C ABI checks that need no GPU: the library loads, exports every function
include/gdpa.h declares, and rejects bad arguments on the host before any
CUDA call (no kernel is launched in this file)."""
import ctypes
import os
import re
import subprocess

import pytest

from jagged_attention_recsys_02_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdpa.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdpa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_and_binding_agree():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(gdpa_[a-z_0-9]+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert lib.gdpa_status_string(code).decode() == name
    assert lib.gdpa_status_string(99).decode() == "GDPA_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    f = lib.gdpa_fwd_workspace_size
    b = lib.gdpa_bwd_workspace_size
    assert f(4, 2, 64, 105, 105) >= 256 + 8 * 2 * (105 // 256 + 4)
    assert f(32, 4, 128, 10**6, 10**6) > f(32, 4, 128, 10**5, 10**6)
    # backward: work list + fp32 dQ accumulator + D
    assert b(4, 2, 64, 105, 105) >= 105 * 2 * 64 * 4 + 105 * 2 * 4
    assert f(-1, 2, 64, 1, 1) == 0 and b(2, 0, 64, 1, 1) == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(lib, **kw):
    a = dict(q=FAKE, qo=FAKE, k=FAKE, v=FAKE, ko=FAKE, B=2, H=2, d=64, Tq=10, Tkv=10, bias=None,
             act=0, causal=0, scale=0.125, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 20,
             stream=None)
    a.update(kw)
    return lib.gdpa_fwd(a["q"], a["qo"], a["k"], a["v"], a["ko"], a["B"], a["H"], a["d"], a["Tq"],
                        a["Tkv"], a["bias"], a["act"], a["causal"], a["scale"], a["out"],
                        a["lse"], a["ws"], a["ws_bytes"], a["stream"])


def _bwd(lib, **kw):
    a = dict(q=FAKE, qo=FAKE, k=FAKE, v=FAKE, ko=FAKE, B=2, H=2, d=64, Tq=10, Tkv=10, bias=None,
             act=0, causal=0, scale=0.125, out=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             ws=FAKE, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.gdpa_bwd(a["q"], a["qo"], a["k"], a["v"], a["ko"], a["B"], a["H"], a["d"], a["Tq"],
                        a["Tkv"], a["bias"], a["act"], a["causal"], a["scale"], a["out"],
                        a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["ws"], a["ws_bytes"],
                        a["stream"])


@pytest.mark.parametrize("call", [_fwd, _bwd])
def test_host_rejections(lib, call):
    assert call(lib, d=96) == UNSUPPORTED
    assert call(lib, d=256) == UNSUPPORTED
    assert call(lib, H=300) == UNSUPPORTED
    assert call(lib, H=0) == INVALID
    assert call(lib, B=-1) == INVALID
    assert call(lib, Tq=-5) == INVALID
    assert call(lib, act=7) == INVALID
    assert call(lib, causal=2) == INVALID
    assert call(lib, qo=None) == INVALID
    assert call(lib, ko=None) == INVALID
    assert call(lib, q=None) == INVALID
    assert call(lib, k=FAKE + 8) == INVALID         # not 16-byte aligned
    assert call(lib, ws=None) == WORKSPACE
    assert call(lib, ws_bytes=16) == WORKSPACE
    bad_bias = binding.gdpa_bias(binding.BIAS_RELPOS, None, 16)
    assert call(lib, bias=ctypes.byref(bad_bias)) == INVALID
    bad_rel = binding.gdpa_bias(binding.BIAS_RELPOS, FAKE, 0)
    assert call(lib, bias=ctypes.byref(bad_rel)) == INVALID
    odd_kind = binding.gdpa_bias(7, FAKE, 4)
    assert call(lib, bias=ctypes.byref(odd_kind)) == INVALID


def test_fwd_specific_rejections(lib):
    assert _fwd(lib, out=None) == INVALID
    assert _fwd(lib, lse=None) == INVALID             # softmax needs lse
    assert _fwd(lib, out=FAKE + 4) == INVALID


def test_bwd_specific_rejections(lib):
    assert _bwd(lib, do=None) == INVALID
    assert _bwd(lib, dk=None) == INVALID
    assert _bwd(lib, lse=None) == INVALID             # softmax needs lse
    assert _bwd(lib, dq=FAKE + 2) == INVALID


def test_empty_problem_is_a_no_op(lib):
    # B = 0 or Tq = 0: nothing to do, returns before touching the device
    assert _fwd(lib, B=0, Tq=0, Tkv=0) == OK
    assert _fwd(lib, Tq=0) == OK
    assert _bwd(lib, B=0, Tq=0, Tkv=0) == OK


def test_window_entry_points_reject_on_host(lib):
    """gdpa_fwd_window / gdpa_bwd_window: a negative window is an argument
    error; the other checks are those of gdpa_fwd / gdpa_bwd."""
    def fwd_w(window, **kw):
        a = dict(q=FAKE, qo=FAKE, k=FAKE, v=FAKE, ko=FAKE, d=64, ws=FAKE)
        a.update(kw)
        return lib.gdpa_fwd_window(a["q"], a["qo"], a["k"], a["v"], a["ko"], 2, 2, a["d"], 10, 10,
                                   None, 0, 1, window, 0.125, FAKE, FAKE, a["ws"], 1 << 20, None)

    def bwd_w(window, **kw):
        a = dict(d=64, bias=None, act=0, dbias=None)
        a.update(kw)
        return lib.gdpa_bwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, a["d"], 10, 10, a["bias"],
                                   a["act"], 1, window, 0.125, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   a["dbias"], FAKE, 1 << 20, None)

    for call in (fwd_w, bwd_w):
        assert call(-1) == INVALID
        assert call(5, d=96) == UNSUPPORTED
    assert fwd_w(5, q=None) == INVALID
    assert fwd_w(5, ws=None) == WORKSPACE
    # a bias-table gradient needs a relative-position table and 4-byte alignment
    table = ctypes.byref(binding.gdpa_bias(binding.BIAS_RELPOS, FAKE, 8))
    assert bwd_w(0, dbias=FAKE) == INVALID
    assert bwd_w(0, dbias=FAKE + 2, bias=table) == INVALID
    assert bwd_w(0, dbias=FAKE + 2, bias=table, act=1) == INVALID
    mx = lib.gdpa_fwd_mxfp8_window(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 10,
                                   10, None, 0, 1, -3, 0.125, FAKE, FAKE, FAKE, 1 << 20, None)
    assert mx == INVALID


def _bwd_mx(lib, window=None, **kw):
    a = dict(q=FAKE, qo=FAKE, k=FAKE, v=FAKE, ko=FAKE, B=2, H=2, d=128, Tq=10, Tkv=10, bias=None,
             act=0, causal=0, scale=0.125, out=FAKE, lse=FAKE, do=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    head = (a["q"], a["qo"], a["k"], a["v"], a["ko"], a["B"], a["H"], a["d"], a["Tq"], a["Tkv"],
            a["bias"], a["act"], a["causal"])
    tail = (a["scale"], a["out"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], a["ws"],
            a["ws_bytes"], a["stream"])
    if window is None:
        return lib.gdpa_bwd_mxfp8(*head, *tail)
    return lib.gdpa_bwd_mxfp8_window(*head, window, *tail)


def test_mxfp8_backward_rejects_on_host(lib):
    """gdpa_bwd_mxfp8(_window): the checks of gdpa_bwd, then softmax and d = 128
    only, then the workspace; nothing reaches the device."""
    for w in (None, 0, 3):
        assert _bwd_mx(lib, window=w, act=1) == UNSUPPORTED
        assert _bwd_mx(lib, window=w, d=64) == UNSUPPORTED
        assert _bwd_mx(lib, window=w, d=96) == UNSUPPORTED
        assert _bwd_mx(lib, window=w, H=0) == INVALID
        assert _bwd_mx(lib, window=w, causal=2) == INVALID
        assert _bwd_mx(lib, window=w, q=FAKE + 8) == INVALID
        assert _bwd_mx(lib, window=w, do=None) == INVALID
        assert _bwd_mx(lib, window=w, lse=None) == INVALID
        assert _bwd_mx(lib, window=w, out=FAKE + 4) == INVALID
        assert _bwd_mx(lib, window=w, dk=None) == INVALID
        assert _bwd_mx(lib, window=w, ws=None) == WORKSPACE
        assert _bwd_mx(lib, window=w, ws_bytes=4096) == WORKSPACE
        assert _bwd_mx(lib, window=w, B=0, Tq=0, Tkv=0) == OK
    assert _bwd_mx(lib, window=-1) == INVALID


def test_mxfp8_quantiser_modes_on_host(lib):
    """GDPA_MX_NOSAT combines with either block shape and leaves the scale
    buffer's size unchanged; any other mode bit is refused before a launch."""
    sb = lib.gdpa_mxfp8_scale_bytes
    B, H, d, T = 5, 3, 128, 1000
    for shape in (binding.MX_ALONG_CHANNELS, binding.MX_ALONG_TOKENS):
        assert sb(B, H, d, T, shape | binding.MX_NOSAT) == sb(B, H, d, T, shape) > 0
    assert sb(B, H, d, T, 4) == 0 and sb(B, H, d, T, 7) == 0
    q = lib.gdpa_quantize_mxfp8
    assert q(FAKE, FAKE, B, H, d, T, 4, FAKE, FAKE, None) == INVALID
    assert q(FAKE, FAKE, B, H, d, T, 8 | binding.MX_NOSAT, FAKE, FAKE, None) == INVALID
    assert q(FAKE, None, B, H, d, T, binding.MX_ALONG_TOKENS | binding.MX_NOSAT, FAKE, FAKE,
             None) == INVALID                       # along tokens needs the offsets
    assert q(FAKE, FAKE, B, H, d, 0, binding.MX_NOSAT, FAKE, FAKE, None) == OK  # nothing to do


def test_mxfp8_backward_workspace_size(lib):
    """Seven E4M3 operand versions (Q, K, dO twice, V once), their scales, the
    fp32 dQ accumulator, D and the work list."""
    s = lib.gdpa_bwd_mxfp8_workspace_size
    B, H, d, Tq, Tkv = 32, 4, 128, 69091, 69091
    codes = (4 * Tq + 3 * Tkv) * H * d
    assert s(B, H, d, Tq, Tkv) >= codes + Tq * H * d * 4 + Tq * H * 4
    assert s(B, H, d, Tq, Tkv) < codes * 1.3 + Tq * H * d * 4 + (1 << 20)
    assert s(-1, H, d, 1, 1) == 0 and s(B, 0, d, 1, 1) == 0 and s(B, H, 96, 1, 1) == 0


def test_dense_bias_rejections_on_host(lib):
    """A dense bias needs its values and its int64 offsets (4- and 8-byte
    aligned); every entry point takes it once those are valid."""
    D = binding.BIAS_DENSE
    dense = lambda table=FAKE, off=FAKE + 64: ctypes.byref(binding.gdpa_bias(D, table, 0, off))
    assert _fwd(lib, bias=dense(off=None)) == INVALID
    assert _fwd(lib, bias=dense(table=None)) == INVALID
    assert _fwd(lib, bias=dense(table=FAKE + 2)) == INVALID
    assert _fwd(lib, bias=dense(off=FAKE + 4)) == INVALID
    assert _bwd(lib, bias=dense(off=None)) == INVALID
    assert _fwd(lib, bias=dense(), ws=None) == WORKSPACE      # valid bias: the next check fires
    # with a window it passes validation (the missing workspace is the next check)
    assert lib.gdpa_fwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, dense(), 0, 0, 4,
                               0.125, FAKE, FAKE, None, 0, None) == WORKSPACE
    assert lib.gdpa_bwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, dense(), 0, 0, 4,
                               0.125, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0,
                               None) == WORKSPACE
    # a misaligned gradient is refused
    assert lib.gdpa_bwd_window(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, dense(), 0, 0, 0,
                               0.125, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, 1 << 20,
                               None) == INVALID
    # the block kernels take it (the missing workspace is the next check), and
    # the block backward returns its gradient
    assert lib.gdpa_block_fwd(FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, dense(), 0, 0, 0.125, FAKE,
                              None, 0, None) == WORKSPACE
    blk_bwd = lambda dbias: lib.gdpa_block_bwd_dbias(FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, dense(),
                                                     0, 0, 0.125, 0.0, FAKE, FAKE, FAKE, FAKE,
                                                     dbias, None, 0, None)
    assert blk_bwd(FAKE) == WORKSPACE
    assert blk_bwd(FAKE + 2) == INVALID
    # the MXFP8 forward and backward take it too
    assert lib.gdpa_fwd_mxfp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 128, 10, 10,
                              dense(), 0, 0, 0.125, FAKE, FAKE, None, 0, None) == WORKSPACE
    assert _bwd_mx(lib, bias=dense(), ws=None) == WORKSPACE


def test_rope_backward_rejects_a_bad_base(lib):
    def rope(base):
        return lib.gdpa_bwd_rope(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, None, 0, 0, 0,
                                 0.125, base, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                                 1 << 20, None)
    assert rope(-1.0) == INVALID
    assert rope(float("nan")) == INVALID
    assert rope(float("inf")) == INVALID
    # a bias gradient needs a bias, with or without the rotary backward
    for base in (0.0, 1e4):
        assert lib.gdpa_bwd_rope(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, None, 0, 0, 0,
                                 0.125, base, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 1 << 20, None) == INVALID
    # a dense bias with a window and the rotary backward passes validation
    dense = ctypes.byref(binding.gdpa_bias(binding.BIAS_DENSE, FAKE, 0, FAKE + 64))
    assert lib.gdpa_bwd_rope(FAKE, FAKE, FAKE, FAKE, FAKE, 2, 2, 64, 10, 10, dense, 0, 0, 4, 0.125,
                             1e4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0,
                             None) == WORKSPACE


def test_binding_marshals_both_bias_forms():
    """The binding's gdpa_bias: a table tensor gives the relative-position kind,
    a (values, offsets) pair the dense kind with both pointers."""
    import torch

    table = torch.zeros(2, 15)
    s = binding._bias(table, 8)._obj
    assert (s.kind, s.table, s.max_rel, s.offsets) == (binding.BIAS_RELPOS, table.data_ptr(), 8, None)
    vals, off = torch.zeros(12), torch.zeros(3, dtype=torch.int64)
    s = binding._bias((vals, off), 0)._obj
    assert (s.kind, s.table, s.offsets) == (binding.BIAS_DENSE, vals.data_ptr(), off.data_ptr())
    assert binding._bias(None, 0) is None


def test_bias_struct_layout_matches_the_header(tmp_path):
    """The ctypes gdpa_bias has the C compiler's size and field offsets for the
    struct declared in include/gdpa.h."""
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdpa.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu", sizeof(gdpa_bias), '
                   'offsetof(gdpa_bias, kind), offsetof(gdpa_bias, table), '
                   'offsetof(gdpa_bias, max_rel), offsetof(gdpa_bias, offsets)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    B = binding.gdpa_bias
    assert got == [ctypes.sizeof(B), B.kind.offset, B.table.offset, B.max_rel.offset,
                   B.offsets.offset]


def test_header_compiles_as_c_and_links(tmp_path, lib):
    """A C program that includes include/gdpa.h and takes the address of every
    declared function compiles as C11 and links against the library."""
    names = declared_functions()
    src = tmp_path / "uses_abi.c"
    src.write_text('#include <stdio.h>\n#include "gdpa.h"\n'
                   "int main(void) {\n  void* fns[] = {\n"
                   + "".join(f"    (void*){n},\n" for n in names)
                   + "  };\n  int n = 0;\n"
                   "  for (unsigned i = 0; i < sizeof(fns) / sizeof(fns[0]); ++i) n += fns[i] != 0;\n"
                   '  printf("%d", n);\n  return 0;\n}\n')
    exe = tmp_path / "uses_abi"
    libdir = os.path.dirname(build.LIB)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), f"-L{libdir}", "-l:" + os.path.basename(build.LIB),
                    f"-Wl,-rpath,{libdir}", "-Wl,--unresolved-symbols=ignore-in-shared-libs"],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, check=True)
    assert int(r.stdout) == len(names)


def test_selftest_rejects_a_bad_limit(lib):
    assert lib.gdpa_selftest_timeout(0, None) == INVALID
    assert lib.gdpa_selftest_timeout(2_000_000, None) == INVALID
