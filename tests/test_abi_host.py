"""Host-side checks of libamsim (no GPU needed): the library loads, exports
every function include/amsim.h declares, its host-only Algorithm 1 LUT
generator agrees with the oracle's for every mantissa width and both kinds,
user-supplied multiplier models go through the same generator, and argument
errors are reported before any device work."""
import ctypes

import numpy as np
import pytest

import approximate_multiplier_dnn_gb300 as am


@pytest.fixture(scope="module")
def L():
    am.build()
    return am.lib()


def test_exports_every_declared_function(L):
    names = am.header_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(L, n), n


def test_cooperative_switch_values(L):
    """The switch is host state only: 0 and 1 are taken, anything else is
    refused, and it is left on."""
    assert L.amsim_set_cooperative_launches(2) == am.AMSIM_EINVAL
    assert L.amsim_set_cooperative_launches(-1) == am.AMSIM_EINVAL
    assert L.amsim_set_cooperative_launches(0) == am.AMSIM_OK
    assert L.amsim_set_cooperative_launches(1) == am.AMSIM_OK


def test_status_strings(L):
    for s in range(6):
        assert am.status_string(s)
    assert am.status_string(99) == "unknown status"


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
@pytest.mark.parametrize("M", list(range(1, 12)))
def test_lut_generate_matches_oracle(L, orc, kind, M):
    assert np.array_equal(am.amsim_lut_generate(kind, M), orc.lut(kind, M))


def test_lut_generate_errors(L):
    buf = np.zeros(4, np.uint32)
    assert L.amsim_lut_generate(0, 0, buf.ctypes.data) == am.AMSIM_EUNSUPPORTED
    assert L.amsim_lut_generate(0, 12, buf.ctypes.data) == am.AMSIM_EUNSUPPORTED
    assert L.amsim_lut_generate(7, 1, buf.ctypes.data) == am.AMSIM_EUNSUPPORTED
    assert L.amsim_lut_generate(0, 1, None) == am.AMSIM_EINVAL


def test_lut_generate_from_user_function(L, orc):
    """A user model (here: Python callbacks of the two closed forms on floats)
    goes through Algorithm 1 and must reproduce the built-in tables."""
    def exact(a, b):
        return float(np.float32(a) * np.float32(b))

    def mitchell(a, b):
        x, y = a - 1.0, b - 1.0
        return 1.0 + x + y if x + y < 1.0 else 2.0 * (x + y)

    for M in (1, 3, 5):
        assert np.array_equal(am.amsim_lut_generate_from_fn(exact, M), orc.lut("exact", M))
        assert np.array_equal(am.amsim_lut_generate_from_fn(mitchell, M), orc.lut("mitchell", M))


def test_lut_generate_from_fn_rejects_bad_model(L):
    with pytest.raises(am.AmsimError) as e:
        am.amsim_lut_generate_from_fn(lambda a, b: 0.25 * a * b, 3)   # exponent drops below the operands'
    assert e.value.status == am.AMSIM_EUNSUPPORTED
    with pytest.raises(am.AmsimError):
        am.amsim_lut_generate_from_fn(lambda a, b: -a * b, 3)          # negative product


def test_conv_out_hw_matches_oracle(L, orc):
    cases = [(2, 7, 6, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1)), (1, 9, 8, 2, 5, 3, 2, (2, 1), (1, 0), (1, 1)),
             (2, 8, 9, 3, 2, 3, 3, (1, 2), (2, 2), (2, 1)), (128, 32, 32, 64, 64, 3, 3, (1, 1), (1, 1), (1, 1))]
    for N, H, W, C, K, R, S, st, pd, dl in cases:
        d = am.ConvDesc.make(N, H, W, C, K, R, S, st, pd, dl)
        assert am.amsim_conv2d_out_hw(d) == orc.conv_out_hw(orc.conv_desc(N, H, W, C, K, R, S, st, pd, dl))
    with pytest.raises(am.AmsimError):
        am.amsim_conv2d_out_hw(am.ConvDesc.make(1, 2, 2, 1, 1, 5, 5))


def test_calls_reject_null_lut_without_device_work(L):
    vp = ctypes.c_void_p
    assert L.amsim_mul(None, None, None, 4, None, None) == am.AMSIM_EINVAL
    assert L.amsim_gemm(b"N", b"N", 2, 2, 2, 1.0, None, 2, None, 2, 0.0, None, 2, None, None, 0,
                        None) == am.AMSIM_EINVAL
    d = am.ConvDesc.make(1, 4, 4, 1, 1, 3, 3)
    assert L.amsim_conv2d_fwd(ctypes.byref(d), None, None, None, None, None, 0, None) == am.AMSIM_EINVAL
    assert L.amsim_gemm_workspace_size(b"N", b"N", 8, 8, 8, 1, None) == 0
    assert L.amsim_conv2d_workspace_size(ctypes.byref(d), 0, None) == 0
    for fn in ("amsim_dwconv2d_fwd", "amsim_dwconv2d_bwd_data", "amsim_dwconv2d_bwd_filter"):
        assert getattr(L, fn)(ctypes.byref(d), None, None, None, None, None, 0, None) == am.AMSIM_EINVAL
    assert L.amsim_dwconv2d_workspace_size(ctypes.byref(d), 2, None) == 0
    L.amsim_lut_destroy(vp(None))     # NULL is ignored
    assert L.amsim_lut_info(None, None, None, None) == am.AMSIM_EINVAL
    assert L.amsim_lut_entries(None, None) == am.AMSIM_EINVAL
    assert L.amsim_softmax_rows(None, None, -1, 4, None) == am.AMSIM_EINVAL
    assert L.amsim_softmax_rows(None, None, 0, 4, None) == am.AMSIM_OK


def test_lut_build_from_entries_rejects_wide_entries(L):
    e = np.zeros(16, np.uint32)
    e[3] = 1 << 24
    h = ctypes.c_void_p(0)
    assert L.amsim_lut_build_from_entries(e.ctypes.data, 2, ctypes.byref(h)) == am.AMSIM_EUNSUPPORTED
    assert L.amsim_lut_build_from_entries(e.ctypes.data, 0, ctypes.byref(h)) == am.AMSIM_EUNSUPPORTED


def test_gemm_problem_struct_layout_matches_header(tmp_path):
    """The binding's ctypes mirror of amsim_gemm_problem has the C layout."""
    import os
    import subprocess
    src = tmp_path / "layout.c"
    src.write_text("""
#include <stdio.h>
#include <stddef.h>
#include "amsim.h"
int main(void) {
    printf("%zu", sizeof(amsim_gemm_problem));
#define F(x) printf(" %zu", offsetof(amsim_gemm_problem, x));
    F(A) F(B) F(C) F(strideA) F(strideB) F(strideC) F(m) F(n) F(k) F(lda) F(ldb) F(ldc) F(batch)
    F(alpha) F(beta) F(transA) F(transB)
    printf("\\n");
    return 0;
}
""")
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(am.HEADER))
    subprocess.run(["gcc", "-std=c11", f"-I{inc}", str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    G = am.GemmProblem
    want = [ctypes.sizeof(G)] + [getattr(G, f).offset for f, _ in G._fields_]
    assert [int(x) for x in out] == want


def test_grouped_rejects_bad_arguments(L):
    probs = (am.GemmProblem * 1)()
    assert L.amsim_gemm_grouped(1, probs, None, None, 0, None) == am.AMSIM_EINVAL
    assert L.amsim_gemm_grouped_workspace_size(1, probs, None) == 0


def test_closed_form_switch_rejects_null(L):
    assert L.amsim_lut_set_closed_form(None, 1) == am.AMSIM_EINVAL
    assert L.amsim_lut_set_closed_form(None, 0) == am.AMSIM_EINVAL


def test_lut_build_from_fn_rejects_before_device_work(L):
    """amsim_lut_build_from_fn runs Algorithm 1 on the host before it touches a
    device: argument and model errors come back without a GPU."""
    h = ctypes.c_void_p(0)
    cb = am.APPROX_MUL_FN(lambda a, b: a * b)
    assert L.amsim_lut_build_from_fn(am.APPROX_MUL_FN(), 3, ctypes.byref(h)) == am.AMSIM_EINVAL
    assert L.amsim_lut_build_from_fn(cb, 3, None) == am.AMSIM_EINVAL
    assert L.amsim_lut_build_from_fn(cb, 0, ctypes.byref(h)) == am.AMSIM_EUNSUPPORTED
    assert L.amsim_lut_build_from_fn(cb, 12, ctypes.byref(h)) == am.AMSIM_EUNSUPPORTED
    bad = am.APPROX_MUL_FN(lambda a, b: 0.25 * a * b)
    assert L.amsim_lut_build_from_fn(bad, 3, ctypes.byref(h)) == am.AMSIM_EUNSUPPORTED
    assert h.value is None


def test_wait_status_calls_check_arguments_first(L):
    """The wait-status calls reject bad arguments before touching a device."""
    assert L.amsim_device_errors(None, 1) == am.AMSIM_EINVAL
    assert L.amsim_set_flag_wait_limit(-5) == am.AMSIM_EINVAL
    assert L.amsim_set_flag_wait_limit(20_000_000_000) == am.AMSIM_EINVAL


def test_exponent_bits_rejects_null_handle(L):
    assert L.amsim_lut_set_exponent_bits(None, 5) == am.AMSIM_EINVAL
