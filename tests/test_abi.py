"""The C-ABI library without a GPU: it loads, exports every function that
include/attnq.h declares, and its host-only helpers behave as documented.
No compute call is made here."""
import ctypes as C
import os
import shutil
import subprocess

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def aq():
    from precision_attention_numerics_gb300 import _build
    _build.build()
    import precision_attention_numerics_gb300 as aq
    aq.load_library()
    return aq


def test_exports_every_declared_symbol(aq):
    names = aq.exported_symbols()
    assert {"attnq_prepare", "attnq_fwd", "attnq_fwd_ponly", "attnq_err", "attnq_device_status",
            "attnq_status_string", "attnq_hadamard_signs", "attnq_version", "attnq_prepare_workspace",
            "attnq_vt_ld"} <= set(names)
    L = aq.load_library()
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(aq):
    assert aq.attnq_version() >= 100
    for code, name in aq.STATUS.items():
        assert aq.attnq_status_string(code).startswith(name)


def test_vt_ld(aq):
    assert [aq.attnq_vt_ld(n) for n in (0, 1, 15, 16, 17, 32768)] == [0, 16, 16, 16, 32, 32768]


@pytest.mark.parametrize("seed", [0, 7, 123456789])
def test_hadamard_signs_follow_splitmix64(aq, seed):
    assert np.array_equal(aq.attnq_hadamard_signs(seed, 128), synth.hadamard_signs(seed, 128))


def test_argument_checks_before_any_cuda_call(aq):
    L = aq.load_library()
    bad = [aq.AttnqDesc(1, 4, 3, 16, 64), aq.AttnqDesc(1, 1, 1, 16, 96), aq.AttnqDesc(0, 1, 1, 16, 64),
           aq.AttnqDesc(1, 1, 1, 0, 64), aq.AttnqDesc(1, 1, 1, 16, 64, flags=64),
           aq.AttnqDesc(1, 1, 1, 16, 64, stat_len=-1), aq.AttnqDesc(1, 1, 1, 16, 64, stat_len=17)]
    want = [1, 2, 1, 1, 1, 1, 1]
    for desc, code in zip(bad, want):
        d = desc._c()
        assert L.attnq_prepare_workspace(C.byref(d)) == 0
        fake = C.c_void_p(4096)
        rc = L.attnq_fwd(C.byref(d), fake, fake, fake, None, C.c_float(256.0), 0, 1, 128, fake, 0, None, 4, None)
        assert rc == code, (desc, rc)


def test_pcast_scales_on_an_e4m3_rounding_point_are_refused(aq):
    """attnq_fwd forms P * S in one exp2, so S must round as P * S at P = 1
    does: S within 2^-20 of an E4M3 rounding point (100 is halfway between 96
    and 104) is refused before any CUDA call; E4M3 values and S clear of such
    points pass it and stop at the next check (a KV tile of 96: unsupported)."""
    L = aq.load_library()
    d = aq.AttnqDesc(1, 1, 1, 16, 64, flags=aq.ATTNQ_VT_LAYOUT)._c()
    fake = C.c_void_p(4096)
    scales = aq.binding._Scales(4096, 4096, 4096, None)

    def rc(S):
        return L.attnq_fwd(C.byref(d), fake, fake, fake, C.byref(scales), C.c_float(S), 0, 1, 96, fake, 0, None, 4,
                           None)
    for S in (100.0, 50.0, 200.0, 25.0, 100.0 * (1 + 2.0 ** -22), 0.0, 449.0, float("nan")):
        assert rc(S) == 1, S  # ATTNQ_EINVAL
    for S in (1.0, 256.0, 448.0, 96.0, 101.0, 0.5, 3.0, 2.0 ** -8):
        assert rc(S) == 2, S  # past the S check: ATTNQ_EUNSUPPORTED for the tile


def test_workspace_size_grows_with_centring(aq):
    d0 = aq.AttnqDesc(2, 32, 8, 32768, 128, flags=aq.ATTNQ_VT_LAYOUT)
    d1 = aq.AttnqDesc(2, 32, 8, 32768, 128, flags=aq.ATTNQ_VT_LAYOUT | aq.ATTNQ_CENTER_K)
    w0, w1 = aq.attnq_prepare_workspace(d0), aq.attnq_prepare_workspace(d1)
    assert 0 < w0 < w1
    assert w1 - w0 >= 2 * 8 * (32768 // 128) * 128 * 4


def test_descriptor_layout_matches_the_header(aq, tmp_path):
    """The ctypes mirrors have the C structs' sizes and field offsets."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stdio.h>\n#include \"attnq.h\"\n"
        "int main(void) { printf(\"%zu %zu %zu %zu\\n\", sizeof(attnq_desc), offsetof(attnq_desc, signs),"
        " offsetof(attnq_desc, stat_len), sizeof(attnq_scales)); return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(root, "include"), "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    from precision_attention_numerics_gb300 import binding
    want = [C.sizeof(binding._Desc), binding._Desc.signs.offset, binding._Desc.stat_len.offset,
            C.sizeof(binding._Scales)]
    assert got == want


def test_missing_library_fails_loudly(aq, tmp_path):
    """Without the compiled library every call raises: there is no other path."""
    from precision_attention_numerics_gb300 import binding
    saved_path, saved_lib = binding._LIB_PATH, binding._lib
    try:
        binding._LIB_PATH = str(tmp_path / "libattnq.so")
        binding._lib = None
        with pytest.raises(RuntimeError, match="is missing"):
            binding.load_library()
        with pytest.raises(RuntimeError, match="is missing"):
            aq.attnq_version()
    finally:
        binding._LIB_PATH, binding._lib = saved_path, saved_lib
