"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/gptq.h declares, and rejects bad arguments before launching."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gptq.h")


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(gptq_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("gptq_hessian_accumulate", "gptq_factor", "gptq_quantize_layer", "gptq_workspace_size",
                     "gptq_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(g):
    lib = g.library()
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in g.SIGNATURES, f"binding lacks {name}"


def test_status_strings(g):
    assert g.gptq_status_string(0) == "GPTQ_OK"
    assert g.gptq_status_string(2) == "GPTQ_ERR_NOT_PD"
    assert g.gptq_status_string(6) == "GPTQ_ERR_TIMEOUT"
    assert g.gptq_status_string(99) == "GPTQ_ERR_UNKNOWN"
    assert g.gptq_version() >= 100


def test_workspace_sizes(g):
    f1 = g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, 1024)
    f2 = g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, 2048)
    assert f1 >= 1024 * 1024 * 4 and f2 > f1 and f1 % 256 == 0
    q = g.gptq_workspace_size(g.GPTQ_WS_QUANTIZE, 4096, 4096, 4, 128, 128)
    assert q >= 4096 * 4096 * 4
    assert g.gptq_workspace_size(g.GPTQ_WS_QUANTIZE, 4096, 4096, 4, 128, 100) == 0
    assert g.gptq_workspace_size(7, 1, 1, 4, 128, 128) == 0
    assert g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, 0) == 0


# fake, aligned, never dereferenced device addresses: validation must fail first
P = 0x10000000


def _err(g, status):
    return g.gptq_status_string(status)


def test_hessian_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    assert lib.gptq_hessian_accumulate(P, 10, 64, 64, None, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_accumulate(None, 10, 64, 64, P, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_accumulate(P, 10, 60, 64, P, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG   # d % 8
    assert lib.gptq_hessian_accumulate(P, 10, 64, 60, P, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG   # ldx < d
    assert lib.gptq_hessian_accumulate(P + 2, 10, 64, 64, P, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_accumulate(P, 10, 64, 64, P, 66, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG   # ldh % 4
    assert lib.gptq_hessian_accumulate(P, -1, 64, 64, P, 64, 2.0, 1, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_hessian_accumulate(P, 10, 64, 64, P, 64, float("nan"), 1, None) == g.GPTQ_ERR_INVALID_ARG
    assert "X" in g.gptq_last_error() or "alpha" in g.gptq_last_error() or g.gptq_last_error()
    # n == 0 without zero_first is a no-op that launches nothing
    assert lib.gptq_hessian_accumulate(None, 0, 64, 64, P, 64, 2.0, 0, None) == g.GPTQ_OK
    assert g.gptq_launch_count() == before


def test_factor_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    ws = g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, 64)
    info = ctypes.c_int64(0)
    call = lambda H, d, pd, ao, perm, U, w, wb: lib.gptq_factor(H, d, pd, ao, perm, U, w, wb, ctypes.byref(info), None)
    assert call(None, 64, 0.01, 0, None, P, P, ws) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 0, 0.01, 0, None, P, P, ws) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 64, -0.5, 0, None, P, P, ws) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 64, float("nan"), 0, None, P, P, ws) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 64, 0.01, 1, None, P, P, ws) == g.GPTQ_ERR_INVALID_ARG           # act-order without perm
    assert call(P, 64, 0.01, 0, None, P, P, ws - 1) == g.GPTQ_ERR_INVALID_ARG       # workspace too small
    assert call(P, 64, 0.01, 0, None, P, P + 64, ws) == g.GPTQ_ERR_INVALID_ARG      # workspace misaligned
    assert g.gptq_launch_count() == before


def test_quantize_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    m, d = 64, 256
    ws = g.gptq_workspace_size(g.GPTQ_WS_QUANTIZE, m, d, 4, 128, 128)

    def call(bits=4, gs=128, bs=128, perm=None, wsb=ws, W=P, dt=0, ldw=d, dd=d):
        return lib.gptq_quantize_layer(W, dt, m, dd, ldw, P, perm, bits, gs, bs, P, P, P, P, P, wsb, None, None)

    assert call(bits=5) == g.GPTQ_ERR_INVALID_ARG
    assert call(gs=96) == g.GPTQ_ERR_INVALID_ARG            # d % g != 0
    assert call(gs=64, bs=96) == g.GPTQ_ERR_INVALID_ARG     # neither divides the other... 96 % 64 and 64 % 96
    assert call(bs=0) == g.GPTQ_ERR_INVALID_ARG
    assert call(W=None) == g.GPTQ_ERR_INVALID_ARG
    assert call(dt=2) == g.GPTQ_ERR_INVALID_ARG
    assert call(ldw=d - 1) == g.GPTQ_ERR_INVALID_ARG
    assert call(wsb=ws - 1) == g.GPTQ_ERR_INVALID_ARG
    assert call(bs=16, gs=128) == g.GPTQ_ERR_UNSUPPORTED    # valid, not built
    assert call(gs=16, bs=32) == g.GPTQ_ERR_UNSUPPORTED
    assert g.gptq_launch_count() == before


def test_unpack_argument_checks(g):
    lib = g.library()
    assert lib.gptq_unpack_codes(None, 4, 4, 4, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, 4, 4, 5, P, None) == g.GPTQ_ERR_INVALID_ARG


def test_host_pipeline_argument_checks(g):
    """gptq_pipeline_create refuses the settings gptq_quantize_layer refuses, and a bad
    chunk size, before it allocates or launches anything; the other pipeline calls
    refuse a NULL pipeline (destroy accepts it)."""
    lib = g.library()
    before = g.gptq_launch_count()
    out = ctypes.c_void_p(P)

    def create(m=64, d=256, dt=1, bits=4, gs=128, bs=128, damp=0.01, ao=0, chunk=1024, o=True):
        return lib.gptq_pipeline_create(m, d, dt, bits, gs, bs, damp, ao, chunk, ctypes.byref(out) if o else None)

    assert create(o=False) == g.GPTQ_ERR_INVALID_ARG
    assert create(bits=5) == g.GPTQ_ERR_INVALID_ARG and out.value is None
    assert create(dt=2) == g.GPTQ_ERR_INVALID_ARG
    assert create(m=0) == g.GPTQ_ERR_INVALID_ARG
    assert create(d=12, gs=-1) == g.GPTQ_ERR_INVALID_ARG        # d a multiple of 8
    assert create(gs=100) == g.GPTQ_ERR_INVALID_ARG
    assert create(damp=-1.0) == g.GPTQ_ERR_INVALID_ARG
    assert create(damp=float("nan")) == g.GPTQ_ERR_INVALID_ARG
    assert create(chunk=0) == g.GPTQ_ERR_INVALID_ARG
    assert create(chunk=(1 << 24) + 1) == g.GPTQ_ERR_INVALID_ARG
    assert create(bs=16, gs=128) == g.GPTQ_ERR_UNSUPPORTED
    assert lib.gptq_pipeline_run(None, P, 256, P, 10, 256, P, P, P, P, None, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_pipeline_status(None, None, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_pipeline_destroy(None) == g.GPTQ_OK
    assert g.gptq_launch_count() == before


def test_dequant_gemv_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()

    def call(q=P, s=P, z=P, gi=None, m=64, d=256, bits=4, gs=128, X=P, T=3, ldx=256, Y=P, ldy=64):
        return lib.gptq_dequant_gemv(q, s, z, gi, m, d, bits, gs, X, T, ldx, Y, ldy, None)

    assert call(q=None) == g.GPTQ_ERR_INVALID_ARG
    assert call(d=250, ldx=256) == g.GPTQ_ERR_INVALID_ARG          # d not a multiple of 32
    assert call(bits=5) == g.GPTQ_ERR_INVALID_ARG
    assert call(gs=48) == g.GPTQ_ERR_INVALID_ARG
    assert call(gs=96) == g.GPTQ_ERR_INVALID_ARG                    # does not divide d
    assert call(ldx=252) == g.GPTQ_ERR_INVALID_ARG
    assert call(ldx=260) == g.GPTQ_ERR_INVALID_ARG                  # not a multiple of 8
    assert call(ldy=63) == g.GPTQ_ERR_INVALID_ARG
    assert call(q=P + 4) == g.GPTQ_ERR_INVALID_ARG                  # 4-bit words need 16-byte alignment
    assert call(T=0, X=None, Y=None) == g.GPTQ_OK                   # nothing to do
    assert call(T=1 << 31) == g.GPTQ_ERR_INVALID_ARG                # token count beyond int32
    assert call(T=-1) == g.GPTQ_ERR_INVALID_ARG
    assert g.gptq_launch_count() == before


def test_factor_static_argument_checks(g):
    lib = g.library()
    info = ctypes.c_int64(0)
    call = lambda H, d, pd, ao, perm, U: lib.gptq_factor_static(H, d, pd, ao, perm, U, ctypes.byref(info), None)
    before = g.gptq_launch_count()
    assert call(None, 64, 0.01, 0, None, P) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 0, 0.01, 0, None, P) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 2049, 0.01, 0, None, P) == g.GPTQ_ERR_INVALID_ARG
    assert "2048" in g.gptq_last_error()
    assert call(P, 64, float("nan"), 0, None, P) == g.GPTQ_ERR_INVALID_ARG
    assert call(P, 64, 0.01, 1, None, P) == g.GPTQ_ERR_INVALID_ARG       # act-order without perm_out
    assert "perm_out" in g.gptq_last_error()
    # without info the outcome could not be read back (the shared scratch holds it)
    assert lib.gptq_factor_static(P, 64, 0.01, 0, None, P, None, None) == g.GPTQ_ERR_INVALID_ARG
    assert "info" in g.gptq_last_error()
    assert g.gptq_launch_count() == before


def test_unpack_codes_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    assert lib.gptq_unpack_codes(None, 4, 64, 4, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, 4, 64, 5, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, -1, 64, 4, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, 4, 65537, 4, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, (1 << 30) + 1, 64, 4, P, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_unpack_codes(P, 1 << 30, 65536, 4, P, None) == g.GPTQ_ERR_INVALID_ARG    # m * d > 2^36
    assert g.gptq_launch_count() == before


def _prototypes():
    """name -> parameter count of every function include/gptq.h declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(gptq_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_signatures_match_the_header(g):
    """Every declared function has a ctypes signature with the same number of parameters."""
    protos = _prototypes()
    assert protos, "no prototypes parsed"
    for name, nargs in protos.items():
        assert name in g.SIGNATURES, f"{name} has no binding"
        assert len(g.SIGNATURES[name][1]) == nargs, (name, nargs, len(g.SIGNATURES[name][1]))


def test_wait_selftest_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    assert lib.gptq_wait_selftest(2, 1000000, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_wait_selftest(0, 999, None) == g.GPTQ_ERR_INVALID_ARG
    assert lib.gptq_wait_selftest(1, 1000000001, None) == g.GPTQ_ERR_INVALID_ARG
    assert g.gptq_launch_count() == before


def test_dequant_gemm_argument_checks(g):
    lib = g.library()
    before = g.gptq_launch_count()
    ws = 1 << 30
    call = lambda q=P, s=P, z=P, m=64, d=256, bits=4, gs=128, X=P, T=16, ldx=256, Y=P, yb=0, ldy=64, w=P, wb=ws: \
        lib.gptq_dequant_gemm(q, s, z, m, d, bits, gs, X, T, ldx, Y, yb, ldy, w, wb, None)
    assert call(q=None) == g.GPTQ_ERR_INVALID_ARG
    assert call(w=None) == g.GPTQ_ERR_INVALID_ARG
    assert call(d=250, ldx=256) == g.GPTQ_ERR_INVALID_ARG           # d not a multiple of 32
    assert call(bits=5) == g.GPTQ_ERR_INVALID_ARG
    assert call(gs=96) == g.GPTQ_ERR_INVALID_ARG                    # does not divide d
    assert call(yb=2) == g.GPTQ_ERR_INVALID_ARG
    assert call(ldx=260) == g.GPTQ_ERR_INVALID_ARG                  # not a multiple of 8
    assert call(ldy=63) == g.GPTQ_ERR_INVALID_ARG
    assert call(X=P + 8) == g.GPTQ_ERR_INVALID_ARG                  # X must be 16-byte aligned
    assert call(w=P + 128) == g.GPTQ_ERR_INVALID_ARG                # ws must be 256-byte aligned
    assert call(wb=64 * 256 * 2 - 1) == g.GPTQ_ERR_INVALID_ARG      # workspace too small
    assert call(T=0, X=None, Y=None) == g.GPTQ_OK                   # nothing to do
    assert call(T=-1) == g.GPTQ_ERR_INVALID_ARG
    assert g.gptq_launch_count() == before
    assert g.gptq_workspace_size(g.GPTQ_WS_DEQUANT_GEMM, 64, 256) >= 64 * 256 * 2
    assert g.gptq_workspace_size(g.GPTQ_WS_DEQUANT_GEMM, 64, 250) == 0
