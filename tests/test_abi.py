"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every symbol include/fp8pa.h declares, and argument errors come
back as status codes before anything touches a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8pa.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_quantised_paged_gb300 import build
    build.build()
    from fp8_quantised_paged_gb300 import _native
    return _native.lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8pa_\w+)\s*\(", text)))


def test_header_declares_the_two_calls():
    names = declared_functions()
    assert "fp8pa_kv_append_quant" in names and "fp8pa_paged_decode_attention" in names


def test_every_declared_symbol_is_exported(lib):
    from fp8_quantised_paged_gb300 import _native
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _native._SIGS, f"binding lacks {name}"


def test_status_strings_and_version(lib):
    assert lib.fp8pa_version() >> 16 == 1
    for code in range(-7, 1):
        assert lib.fp8pa_error_string(code)
    assert lib.fp8pa_error_string(-99) == b"unknown status"


def test_argument_errors_need_no_device(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # bad enum
    assert lib.fp8pa_kv_append_quant(fake, None, fake, 4, 1, 64, 7, 0, 64, fake, None, fake, None,
                                     8, 16, None) == -2
    # bad shape
    assert lib.fp8pa_kv_append_quant(fake, None, fake, 4, 0, 64, 0, 0, 64, fake, None, fake, None,
                                     8, 16, None) == -3
    # head_dim not a multiple of 16
    assert lib.fp8pa_kv_append_quant(fake, None, fake, 4, 1, 40, 0, 0, 64, fake, None, fake, None,
                                     8, 16, None) == -4
    # null pointers
    assert lib.fp8pa_kv_append_quant(None, None, fake, 4, 1, 64, 0, 0, 64, fake, None, fake, None,
                                     8, 16, None) == -1
    # misaligned
    assert lib.fp8pa_kv_append_quant(P(0x1001), None, fake, 4, 1, 64, 0, 0, 64, fake, None, fake,
                                     None, 8, 16, None) == -6
    # no tokens: nothing to do
    assert lib.fp8pa_kv_append_quant(None, None, None, 0, 1, 64, 0, 0, 64, None, None, None, None,
                                     8, 16, None) == 0
    # INT8 codes with power-of-two (MX) block scales: not a defined pairing
    assert lib.fp8pa_kv_append_quant(fake, None, fake, 4, 1, 64, 2, 3, 32, fake, None, fake, None,
                                     8, 16, None) == -4

    def dec(**kw):
        a = dict(q=fake, kc=fake, vc=fake, ks=fake, vs=fake, bt=fake, mb=4, sl=fake, B=2, bs=16,
                 hq=8, hkv=2, d=128, dv=128, fmt=0, mode=0, gs=64, sm=0.1, nb=16, out=fake,
                 odt=0, ws=fake, wsb=1 << 30, st=None)
        a.update(kw)
        return lib.fp8pa_paged_decode_attention(
            a["q"], a["kc"], a["vc"], a["ks"], a["vs"], a["bt"], a["mb"], a["sl"], a["B"],
            a["bs"], a["hq"], a["hkv"], a["d"], a["dv"], a["fmt"], a["mode"], a["gs"],
            ctypes.c_float(a["sm"]), a["nb"], a["out"], a["odt"], a["ws"], a["wsb"], a["st"])

    assert dec(hq=7) == -3          # Hq % Hkv != 0
    assert dec(fmt=3) == -2
    assert dec(fmt=2, mode=3, gs=32) == -4  # INT8 codes with MX block scales
    assert dec(mode=5) == -2
    assert dec(odt=2) == -2
    assert dec(d=96, dv=96) == -4   # head_dim not served
    assert dec(hq=32, hkv=2) == -4  # 16 heads per KV head
    assert dec(bs=8) == -4
    assert dec(q=None) == -1
    assert dec(vc=None) == -1
    assert dec(B=0) == 0
    assert dec(d=576, dv=512, hkv=1, hq=128, mode=2, bs=64, vc=P(0x2000)) == -4  # MLA needs v==k


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fp8pa.h"

/* Host-only use of the C ABI from plain C: version, status strings and
 * argument errors (none of these touch a device). */
int main(void) {
  const int major = fp8pa_version() >> 16;
  if (major != 1) { printf("version %d\n", major); return 1; }
  if (strcmp(fp8pa_error_string(FP8PA_ERR_WORKSPACE), "workspace missing or too small") != 0)
    return 2;
  static uint16_t k[4 * 64];
  static int32_t slots[4];
  static uint8_t cache[8 * 16 * 64];
  static float scale[8 * 16];
  int rc = fp8pa_kv_append_quant(k, NULL, slots, 4, 1, 64, 7 /* no such format */,
                                 FP8PA_SCALE_TOKEN_HEAD, 64, cache, NULL, scale, NULL, 8, 16,
                                 NULL);
  if (rc != FP8PA_ERR_BAD_ENUM) { printf("append rc %d\n", rc); return 3; }
  rc = fp8pa_kv_append_quant(k, NULL, slots, 4, 1, 64, FP8PA_INT8, FP8PA_SCALE_MX_BLOCK, 32,
                             cache, NULL, scale, NULL, 8, 16, NULL);
  if (rc != FP8PA_ERR_UNSUPPORTED) { printf("int8+mx rc %d\n", rc); return 4; }
  rc = fp8pa_paged_decode_attention(NULL, NULL, NULL, NULL, NULL, NULL, 4, NULL, 0, 16, 8, 2,
                                    128, 128, FP8PA_E4M3, FP8PA_SCALE_TOKEN_HEAD, 64, 0.1f, 16,
                                    NULL, FP8PA_OUT_BF16, NULL, 0, NULL);
  if (rc != FP8PA_OK) { printf("empty batch rc %d\n", rc); return 5; }
  puts("ok");
  return 0;
}
"""


def test_plain_c_program_builds_against_the_header_and_runs(lib, tmp_path):
    """The boundary is a C ABI: a C11 program (pedantic, warnings as errors)
    compiles against include/fp8pa.h, links libfp8pa.so and runs."""
    import shutil
    import subprocess
    from fp8_quantised_paged_gb300 import _native
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(_native.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lfp8pa",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
