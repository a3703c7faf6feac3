"""The C-ABI library loads and exports every entry point that include/kq.h declares.

Runs without a GPU: only size helpers and argument checks that fail before any
CUDA call are exercised here.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kq.h")


@pytest.fixture(scope="module")
def kqlib():
    from quantized_decode_gemv_block_gb300 import build
    build.build()
    import quantized_decode_gemv_block_gb300 as kq
    return kq


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kq_gemv", "kq_gemm", "kq_gemm_workspace_size", "kq_quantize", "kq_block_bytes",
              "kq_block_weights", "kq_row_bytes", "kq_last_error", "kq_version"):
        assert n in names


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as strict C99 and links against the library's
    symbols by name only (no C++ types, no torch)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_kq.c"
    src.write_text('#include "kq.h"\nint main(void) { return kq_block_bytes(KQ_Q4_K) == 144 ? 0 : 1; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-fsyntax-only", str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_calls_the_library(kqlib, tmp_path):
    """A plain C caller links libkq.so and gets sizes, the version and argument errors (every
    call below returns before any CUDA work, so no GPU is needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "call_kq.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "kq.h"
int main(void) {
  if (kq_row_bytes(KQ_Q4_K, 2560) != 1440 || kq_row_bytes(KQ_Q8_0, 2048) != 2176) return 1;
  if (strstr(kq_version(), "sm_103a") == NULL) return 2;
  if (kq_gemv(KQ_Q4_K, NULL, KQ_BF16, NULL, NULL, 1, 8, 300, NULL) != KQ_ERR_ARG) return 3;
  if (strlen(kq_last_error()) == 0) return 4;
  if (kq_gemv(KQ_Q4_K, NULL, KQ_BF16, NULL, NULL, 0, 8, 256, NULL) != KQ_OK) return 5;
  if (kq_shortlist_bytes(151936, 2048) != (size_t)151936 * 8 * 144 + (size_t)151936 * 4) return 6;
  puts("ok");
  return 0;
}
""")
    lib_dir = os.path.dirname(kqlib.LIB_PATH)
    exe = tmp_path / "call_kq"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", lib_dir, "-lkq", "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stdout, run.stderr)


def test_library_exports_every_declared_symbol(kqlib):
    L = ctypes.CDLL(kqlib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_size_helpers(kqlib):
    assert (kqlib.block_bytes("q8_0"), kqlib.block_weights("q8_0")) == (34, 32)
    assert (kqlib.block_bytes("q4_k"), kqlib.block_weights("q4_k")) == (144, 256)
    assert (kqlib.block_bytes("affine4"), kqlib.block_weights("affine4")) == (20, 32)
    assert (kqlib.block_bytes("q5_k"), kqlib.block_weights("q5_k")) == (176, 256)
    assert (kqlib.block_bytes("q6_k"), kqlib.block_weights("q6_k")) == (210, 256)
    assert kqlib.row_bytes("q5_k", 2560) == 1760
    assert kqlib.row_bytes("q6_k", 2560) == 2100
    assert kqlib.block_bytes(99) == 0
    assert kqlib.row_bytes("q4_k", 2560) == 1440
    assert kqlib.row_bytes("q8_0", 2048) == 2176
    assert kqlib.row_bytes("affine4", 2560) == 1600
    assert kqlib.row_bytes("q4_k", 100) == 0
    assert "sm_103a" in kqlib.version()


def test_argument_errors_before_any_cuda_call(kqlib):
    L = kqlib.lib()
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    cases = [
        ((7, fake, kqlib.BF16, fake, fake, 1, 8, 256, None), kqlib.KQ_ERR_UNSUPPORTED),
        ((kqlib.Q4_K, fake, 9, fake, fake, 1, 8, 256, None), kqlib.KQ_ERR_UNSUPPORTED),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake, fake, 17, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake, fake, -1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake, fake, 1, 8, 300, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, None, kqlib.BF16, fake, fake, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, None, fake, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake, None, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake + 8, kqlib.BF16, fake, fake, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake + 4, fake, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
        ((kqlib.Q4_K, fake, kqlib.BF16, fake, fake + 2, 1, 8, 256, None), kqlib.KQ_ERR_ARG),
    ]
    for args, code in cases:
        assert L.kq_gemv(*args) == code, args
        assert L.kq_last_error().decode() != ""
    # empty problems succeed without launching anything
    assert L.kq_gemv(kqlib.Q4_K, None, kqlib.BF16, None, None, 0, 8, 256, None) == 0
    assert L.kq_gemv(kqlib.Q4_K, None, kqlib.BF16, None, None, 4, 0, 256, None) == 0
    assert L.kq_last_error().decode() == ""
    assert L.kq_quantize(kqlib.Q4_K, fake, fake, 4, 100, None) == kqlib.KQ_ERR_ARG
    assert L.kq_quantize(99, fake, fake, 4, 256, None) == kqlib.KQ_ERR_UNSUPPORTED
    # decode attention: shape and pointer checks before any CUDA call
    bad = [(0, 10, 16, 4, 128), (33, 10, 16, 4, 128), (4, -1, 16, 4, 128), (4, 10, 6, 4, 128),
           (4, 10, 16, 4, 96), (32, 10, 32, 4, 128)]
    for (M, Lc, nq, nkv, hd) in bad:
        assert L.kq_attention_workspace_size(M, Lc, nq, nkv, hd) == 0
        assert L.kq_attention(fake, fake, fake, fake, M, Lc, nq, nkv, hd, None, 1.0, fake, 1 << 30, None) \
            == kqlib.KQ_ERR_ARG, (M, Lc, nq, nkv, hd)
    need = L.kq_attention_workspace_size(8, 100, 16, 4, 128)
    assert need == 4 * 1 * 32 * 130 * 4  # kv heads x (108 positions: one 128-position chunk) x rows x (d + m, l)
    assert L.kq_attention(fake, fake, fake, fake, 8, 100, 16, 4, 128, None, 1.0, fake, need - 1, None) \
        == kqlib.KQ_ERR_WORKSPACE
    assert L.kq_attention(None, fake, fake, fake, 8, 100, 16, 4, 128, None, 1.0, fake, need, None) == kqlib.KQ_ERR_ARG


def test_shortlist_head_argument_checks(kqlib):
    L = kqlib.lib()
    fake = 1 << 20
    # buffer sizes: the small copy rounded up to 256 bytes, then N fp32 bounds
    assert L.kq_shortlist_bytes(151936, 2048) == 151936 * 8 * 144 + 151936 * 4
    assert L.kq_shortlist_bytes(3, 256) == 512 + 256  # 432 bytes of copy, 12 of bounds
    for N, K in ((0, 256), (4, 0), (4, 300), (-1, 256)):
        assert L.kq_shortlist_bytes(N, K) == 0
        assert L.kq_shortlist_build(fake, N, K, fake, 1 << 30, None) == kqlib.KQ_ERR_ARG
    assert L.kq_shortlist_build(fake, 4, 256, fake, 511, None) == kqlib.KQ_ERR_ARG       # buffer too small
    assert L.kq_shortlist_build(fake, 4, 256, fake + 16, 1 << 20, None) == kqlib.KQ_ERR_ARG  # not 256-aligned
    # workspace: M*N scores, 2 x 16 words per chunk of 1024 rows, the state
    assert L.kq_head_argmax_workspace_size(1, 151936) == 607744 + 19200 + 256  # 149 x 128 B rounded up to 256
    assert L.kq_head_argmax_workspace_size(0, 100) == 0 and L.kq_head_argmax_workspace_size(17, 100) == 0
    need = L.kq_head_argmax_workspace_size(2, 1000)
    ok_args = dict(w=fake, sl=fake, xd=kqlib.BF16, x=fake, M=2, N=1000, K=256, tok=fake, sc=fake, rs=None,
                   ws=fake, wsn=need, fl=0)

    def call(**kw):
        a = dict(ok_args, **kw)
        return L.kq_head_argmax(a["w"], a["sl"], a["xd"], a["x"], a["M"], a["N"], a["K"], a["tok"], a["sc"],
                                a["rs"], a["ws"], a["wsn"], a["fl"], None)
    assert call(fl=2) == kqlib.KQ_ERR_ARG
    assert call(M=0) == kqlib.KQ_ERR_ARG and call(M=17) == kqlib.KQ_ERR_ARG
    assert call(K=300) == kqlib.KQ_ERR_ARG and call(N=0) == kqlib.KQ_ERR_ARG
    assert call(xd=7) == kqlib.KQ_ERR_UNSUPPORTED
    assert call(sl=None) == kqlib.KQ_ERR_ARG
    assert call(x=fake + 8) == kqlib.KQ_ERR_ARG and call(sl=fake + 16) == kqlib.KQ_ERR_ARG
    assert call(wsn=need - 1) == kqlib.KQ_ERR_WORKSPACE and call(ws=None) == kqlib.KQ_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(tmp_path):
    import quantized_decode_gemv_block_gb300 as kq
    with pytest.raises(ImportError):
        kq._lib, saved = None, kq._lib
        try:
            kq.load_library(str(tmp_path / "missing.so"))
        finally:
            kq._lib = saved
