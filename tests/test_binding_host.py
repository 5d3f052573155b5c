"""The Python binding's argument marshalling, on CPU: a recording stand-in takes the
library's place and receives the pointers, sizes, strides and workspace bytes that each
call passes; shape, dtype, device and workspace checks raise before any library call.
Only the "is a CUDA tensor" requirement is lifted (there is no GPU here); the calls use
the shapes the package's own callers pass."""
import os

import pytest
import torch


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


class _Recorder:
    """Stands in for the CDLL: compute entry points record their arguments and return OK;
    the host-only helpers (workspace sizes, status strings) are the real library's."""

    REAL = ("gptq_workspace_size", "gptq_status_string", "gptq_last_error")

    def __init__(self, real):
        self.real = real
        self.calls = []

    def __getattr__(self, name):
        if name in self.REAL:
            return getattr(self.real, name)

        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


@pytest.fixture
def fake(g, monkeypatch):
    rec = _Recorder(g.library())
    monkeypatch.setattr(g, "_lib", rec)

    def need_cuda(t, name, dtypes):              # dtype still checked; CPU tensors allowed
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a tensor")
        if t.dtype not in dtypes:
            raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    monkeypatch.setattr(g, "_need_cuda", need_cuda)
    monkeypatch.setattr(g, "_stream", lambda s: None)
    return rec


def _layer(g, m, d, bits, gs):
    G = 1 if gs == -1 else d // gs
    return g.QuantizedLayer(torch.zeros((m, (d * bits + 31) // 32), dtype=torch.int32),
                            torch.zeros((m, G)), torch.zeros((m, G)), torch.zeros(d), bits, gs, d)


def test_hessian_marshalling(g, fake):
    X = torch.zeros((100, 64), dtype=torch.int16)
    H = torch.zeros((72, 80))[:64, :64]                 # a view: row stride 80
    g.gptq_hessian_accumulate(X, H, alpha=2.0, zero_first=True)
    name, a = fake.calls[-1]
    assert name == "gptq_hessian_accumulate"
    assert a[1:4] == (100, 64, 64) and a[5] == 80 and a[6] == 2.0 and a[7] == 1
    with pytest.raises(ValueError):
        g.gptq_hessian_accumulate(X, torch.zeros((64, 63)))


def test_factor_marshalling_and_output_checks(g, fake):
    d = 256
    H = torch.zeros((d, d))
    need = g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, d)
    U, perm, info = g.gptq_factor(H, act_order=True, sync=False)
    name, a = fake.calls[-1]
    assert name == "gptq_factor" and a[1] == d and a[3] == 1
    assert U.shape == (d, d) and perm.shape == (d,) and perm.dtype == torch.int32 and info is None
    assert a[7] >= need                                   # workspace bytes
    ws = torch.zeros(need // 4 + 1, dtype=torch.float32)  # any dtype: bytes are counted
    g.gptq_factor(H, Hinv1=U, ws=ws, sync=False)
    assert fake.calls[-1][1][7] == ws.numel() * 4 and fake.calls[-1][1][4] is None
    n = len(fake.calls)
    with pytest.raises(ValueError):
        g.gptq_factor(H, ws=torch.zeros(need - 1, dtype=torch.uint8))
    with pytest.raises(ValueError):
        g.gptq_factor(H, Hinv1=torch.zeros((d, d - 1)))
    with pytest.raises(ValueError):
        g.gptq_factor(H, Hinv1=torch.zeros((d, d)).t())   # not contiguous
    with pytest.raises(TypeError):
        g.gptq_factor(H, Hinv1=torch.zeros((d, d), dtype=torch.float64))
    with pytest.raises(ValueError):
        g.gptq_factor(H, act_order=True, perm_out=torch.zeros(d - 1, dtype=torch.int32))
    with pytest.raises(ValueError):
        g.gptq_factor_static(H, torch.zeros((d, d)), act_order=True, perm_out=torch.zeros(2 * d, dtype=torch.int32))
    assert len(fake.calls) == n


@pytest.mark.parametrize("bits,gs", [(4, 128), (3, -1), (2, 64), (8, 32)])
def test_quantize_marshalling_and_output_checks(g, fake, bits, gs):
    m, d = 96, 256
    W = torch.zeros((m, d), dtype=torch.bfloat16)
    U = torch.zeros((d, d))
    q = g.gptq_quantize_layer(W, U, None, bits=bits, group_size=gs, blocksize=32 if gs == 32 else 64)
    name, a = fake.calls[-1]
    assert name == "gptq_quantize_layer" and a[1] == 1 and a[2:5] == (m, d, d) and a[7:10] == (
        bits, gs, 32 if gs == 32 else 64)
    assert q.qweight.shape == (m, (d * bits + 31) // 32) and (q.bits, q.group_size, q.d) == (bits, gs, d)
    out = _layer(g, m, d, bits, gs)
    g.gptq_quantize_layer(W, U, None, bits=bits, group_size=gs, blocksize=32 if gs == 32 else 64, out=out)
    n = len(fake.calls)
    bad = _layer(g, m, d, bits, gs)
    bad.scales = torch.zeros((m + 1, bad.scales.shape[1]))
    with pytest.raises(ValueError):
        g.gptq_quantize_layer(W, U, None, bits=bits, group_size=gs, out=bad)
    with pytest.raises(ValueError):                       # metadata of another layout
        g.gptq_quantize_layer(W, U, None, bits=bits, group_size=gs, out=_layer(g, m, d, 8 if bits != 8 else 4, gs))
    with pytest.raises(ValueError):
        g.gptq_quantize_layer(W, U, torch.zeros(d + 1, dtype=torch.int32), bits=bits, group_size=gs)
    assert len(fake.calls) == n


def test_unpack_and_gemv_marshalling(g, fake):
    m, d = 64, 256
    q = _layer(g, m, d, 4, 128)
    g.gptq_unpack_codes(q.qweight, m, d, 4)
    assert fake.calls[-1][0] == "gptq_unpack_codes" and fake.calls[-1][1][1:4] == (m, d, 4)
    g.gptq_unpack_codes(q.qweight, m - 8, d, 4)         # the first rows of a larger layer
    X = torch.zeros((5, 264), dtype=torch.int16)[:, :d]  # row stride 264
    Y = g.gptq_dequant_gemv(q, X, m)
    name, a = fake.calls[-1]
    assert name == "gptq_dequant_gemv" and a[4:8] == (m, d, 4, 128) and a[9:11] == (5, 264) and a[12] == m
    assert Y.shape == (5, m) and Y.dtype == torch.float32
    gi = torch.zeros(d, dtype=torch.int32)
    g.gptq_dequant_gemv(q, X, m, g_idx=gi, Y=torch.zeros((5, m)))
    n = len(fake.calls)
    with pytest.raises(ValueError):
        g.gptq_unpack_codes(q.qweight, m + 1, d, 4)      # more rows than stored
    with pytest.raises(ValueError):
        g.gptq_unpack_codes(q.qweight, m, d, 8)          # another width
    with pytest.raises(ValueError):
        g.gptq_dequant_gemv(q, X, m + 1)
    with pytest.raises(ValueError):
        g.gptq_dequant_gemv(q, X, m, Y=torch.zeros((4, m)))
    with pytest.raises(TypeError):
        g.gptq_dequant_gemv(q, X, m, Y=torch.zeros((5, m), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        g.gptq_dequant_gemv(q, X, m, g_idx=torch.zeros(d - 32, dtype=torch.int32))
    short = _layer(g, m, d, 4, 128)
    short.scales = torch.zeros((m, 1))
    with pytest.raises(ValueError):
        g.gptq_dequant_gemv(short, X, m)
    assert len(fake.calls) == n


def test_gemm_marshalling(g, fake):
    M, N, K = 48, 40, 24
    for ak in (True, False):
        for bk in (True, False):
            A = torch.zeros((M, K) if ak else (K, M))
            B = torch.zeros((N, K) if bk else (K, N))
            C = torch.zeros((M, N))
            g.gptq_gemm_f32(A, B, C, ak, bk)
            assert fake.calls[-1][1][3:6] == (M, N, K)
            with pytest.raises(ValueError):
                g.gptq_gemm_f32(A, torch.zeros((N + 1, K) if bk else (K, N + 1)), C, ak, bk)
            with pytest.raises(ValueError):
                g.gptq_gemm_f32(torch.zeros((M + 1, K) if ak else (K, M + 1)), B, C, ak, bk)


def test_tensors_on_two_devices_are_refused(g, fake):
    H = torch.zeros((64, 64))
    with pytest.raises(ValueError):
        g.gptq_factor(H, Hinv1=torch.zeros((64, 64), device="meta"), sync=False)


def test_dequant_gemm_marshalling(g, fake):
    m, d, T = 96, 256, 300
    q = _layer(g, m, d, 4, 128)
    X = torch.zeros((T, d + 8), dtype=torch.int16)[:, :d]          # row stride d + 8
    Y = g.gptq_dequant_gemm(q, X, m, out_bf16=True)
    name, a = fake.calls[-1]
    assert name == "gptq_dequant_gemm"
    assert a[3:7] == (m, d, 4, 128) and a[8:10] == (T, d + 8) and a[11] == 1 and a[12] == m
    assert a[14] == g.gptq_workspace_size(g.GPTQ_WS_DEQUANT_GEMM, m, d)
    assert Y.dtype == torch.bfloat16 and tuple(Y.shape) == (T, m)
    g.gptq_dequant_gemm(q, X, m, Y=torch.zeros((T, m)))
    assert fake.calls[-1][1][11] == 0
    n = len(fake.calls)
    with pytest.raises(TypeError):
        g.gptq_dequant_gemm(q, X, m, Y=torch.zeros((T, m)), out_bf16=True)       # dtype of Y
    with pytest.raises(ValueError):
        g.gptq_dequant_gemm(q, X, m, Y=torch.zeros((T - 1, m)))
    with pytest.raises(ValueError):
        g.gptq_dequant_gemm(q, X, m, ws=torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        g.gptq_dequant_gemm(q, torch.zeros((T, d - 32), dtype=torch.int16), m)
    assert len(fake.calls) == n


def test_sequential_quantize_marshalling(g, fake):
    """Each layer runs Hessian, factor, column loop, then the dequant GEMM whose bf16
    output is the next layer's Hessian input; a width mismatch raises before any call."""
    n = 512
    X0 = torch.zeros((n, 256), dtype=torch.int16)
    Ws = [torch.zeros((128, 256), dtype=torch.bfloat16), torch.zeros((64, 128), dtype=torch.bfloat16)]
    layers, inputs, out = g.sequential_quantize(X0, Ws, bits=4, group_size=128)
    names = [c[0] for c in fake.calls]
    per_layer = ["gptq_hessian_accumulate", "gptq_factor", "gptq_quantize_layer", "gptq_dequant_gemm"]
    assert names == per_layer * 2
    h1, gemm1, h2, gemm2 = fake.calls[0][1], fake.calls[3][1], fake.calls[4][1], fake.calls[7][1]
    assert h1[0] == X0.data_ptr() and h1[1:3] == (n, 256)
    assert gemm1[3:5] == (128, 256) and gemm1[7] == X0.data_ptr() and gemm1[11] == 1
    assert h2[0] == gemm1[10] and h2[1:3] == (n, 128)           # layer 2 sees layer 1's bf16 outputs
    assert gemm2[3:5] == (64, 128) and gemm2[7] == gemm1[10] and gemm2[10] == out.data_ptr()
    assert [x.data_ptr() for x in inputs] == [X0.data_ptr(), gemm1[10]]
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == (n, 64) and len(layers) == 2
    k = len(fake.calls)
    with pytest.raises(ValueError):
        g.sequential_quantize(X0, [torch.zeros((64, 128), dtype=torch.bfloat16)])
    assert len(fake.calls) == k


def test_host_pipeline_marshalling(g, fake):
    """HostPipeline hands the library its settings at creation, then per run the host
    pointers with their row strides (views into wider arrays keep their stride), the
    token count and the output buffers (the permutation only with act-order); bad
    shapes and dtypes raise before any call."""
    m, d = 48, 256
    pipe = g.HostPipeline(m, d, bits=3, group_size=-1, blocksize=64, percdamp=0.02, act_order=True,
                          chunk_tokens=1000, w_dtype=torch.float32, device="cpu")
    name, a = fake.calls[-1]
    assert name == "gptq_pipeline_create"
    assert a[:6] == (m, d, 0, 3, -1, 64) and abs(a[6] - 0.02) < 1e-7 and a[7:9] == (1, 1000)
    Wwide = torch.zeros((m, d + 8))
    Xwide = torch.zeros((700, d + 16), dtype=torch.int16)
    out = pipe.run(Wwide[:, :d], Xwide[:, :d])
    name, a = fake.calls[-1]
    assert name == "gptq_pipeline_run"
    assert a[1] == Wwide.data_ptr() and a[2] == d + 8
    assert a[3] == Xwide.data_ptr() and a[4:6] == (700, d + 16)
    assert a[6:10] == (out.qweight.data_ptr(), out.scales.data_ptr(), out.zeros.data_ptr(), out.col_losses.data_ptr())
    assert a[10] == pipe.perm.data_ptr() and pipe.perm.shape == (d,)
    assert out.qweight.shape == (m, (d * 3 + 31) // 32) and out.scales.shape == (m, 1)
    assert pipe.bytes_h2d(700) == 700 * d * 2 + m * d * 4
    assert pipe.bytes_d2h() == out.qweight.numel() * 4 + 2 * m * 4 + d * 4 + d * 4
    n_calls = len(fake.calls)
    with pytest.raises(ValueError):
        pipe.run(torch.zeros((m, d), dtype=torch.bfloat16), Xwide[:, :d])     # W dtype
    with pytest.raises(ValueError):
        pipe.run(Wwide[:, :d], torch.zeros((10, d + 1), dtype=torch.int16))  # X width
    with pytest.raises(TypeError):
        pipe.run(Wwide[:, :d], torch.zeros((10, d), dtype=torch.float32))    # X dtype
    assert len(fake.calls) == n_calls
    pipe2 = g.HostPipeline(m, d, bits=4, group_size=128, device="cpu")
    assert fake.calls[-1][1][2] == 1 and pipe2.perm is None                  # bf16 W by default
    pipe2.run(torch.zeros((m, d), dtype=torch.bfloat16), torch.zeros((5, d), dtype=torch.int16))
    assert fake.calls[-1][1][10] is None
