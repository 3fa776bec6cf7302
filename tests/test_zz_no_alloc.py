"""la_gemm_noalloc (the GEMM whose workspace is a fixed array inside the
library) against la_debug_gemm (the same kernel with a workspace allocated per
call), through the C ABI, two calls in a row per case so that the second call
runs on the workspace the first one left behind.

This file is collected last on purpose: it must pass both in a fresh process
(where its first call sets the workspace up) and after every other GPU test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16_REL = 2.0 ** -7     # two bf16 ulps: the stored results are rounded to bf16
F32_REL = 1e-5


def L():
    from lookahead_decoding_gb300 import _lib
    return _lib


def bf16_bits(rng, shape, scale):
    v = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return v.to(torch.bfloat16)


def run(mode, w, w2, x, y):
    s = torch.cuda.current_stream()
    L().la_gemm_noalloc(mode, w.data_ptr(), w2.data_ptr() if w2 is not None else None, w.shape[0], w.shape[1],
                        x.data_ptr(), x.shape[0], y.data_ptr(), s.cuda_stream)


@pytest.mark.parametrize("mode,n_out,K,rows", [(0, 4096, 4096, 64),     # the 7B attention output shape
                                               (0, 1280, 704, 1),
                                               (2, 1408, 512, 17)])
def test_bf16_modes_match_debug_gemm_twice(mode, n_out, K, rows):
    rng = np.random.default_rng(1000 + mode * 7 + rows)
    w = bf16_bits(rng, (n_out, K), 0.02)
    w2 = bf16_bits(rng, (n_out, K), 0.02) if mode == 2 else None
    x = bf16_bits(rng, (rows, K), 1.0)
    ref = L().la_debug_gemm(w, x, 0, mode, w2_bf16=w2)
    dw, dx = w.cuda(), x.cuda()
    dw2 = w2.cuda() if w2 is not None else None
    for call in range(2):
        y = torch.full((rows, n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
        run(mode, dw, dw2, dx, y)
        got = y.float().cpu().numpy()
        tol = BF16_REL * np.abs(ref) + 1e-6
        assert np.all(np.abs(got - ref) <= tol), (call, float(np.max(np.abs(got - ref))))


def test_resid_matches_debug_gemm_twice():
    """Ragged rows over two 256-row chunks; the second call accumulates onto the first."""
    mode, n_out, K, rows = 1, 512, 1024, 300
    rng = np.random.default_rng(77)
    w = bf16_bits(rng, (n_out, K), 0.02)
    x = bf16_bits(rng, (rows, K), 1.0)
    y0 = rng.standard_normal((rows, n_out)).astype(np.float32)
    r1 = L().la_debug_gemm(w, x, 0, mode, y_in=y0)
    r2 = L().la_debug_gemm(w, x, 0, mode, y_in=r1)
    y = torch.from_numpy(y0).cuda()
    dw, dx = w.cuda(), x.cuda()
    for ref in (r1, r2):
        run(mode, dw, None, dx, y)
        got = y.cpu().numpy()
        assert np.all(np.abs(got - ref) <= F32_REL * np.abs(ref) + 1e-5), float(np.max(np.abs(got - ref)))


def test_rejects_before_device_work():
    _lib = L()
    w = torch.zeros((12288, 4096), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((1024, 4096), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1024, 12288), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # four 256-row chunks of a 12288 x 4096 weight need far more than 64 MiB of partial sums
    rc = _lib.LIB.la_gemm_noalloc(0, w.data_ptr(), None, 12288, 4096, x.data_ptr(), 1024, y.data_ptr(), s)
    assert rc == _lib.LA_ECAPACITY
    # misaligned activations, a missing second weight, an unsupported mode
    rc = _lib.LIB.la_gemm_noalloc(0, w.data_ptr(), None, 12288, 4096, x.data_ptr() + 2, 4, y.data_ptr(), s)
    assert rc == _lib.LA_EINVAL
    assert _lib.LIB.la_gemm_noalloc(2, w.data_ptr(), None, 128, 64, x.data_ptr(), 4, y.data_ptr(), s) == _lib.LA_EINVAL
    assert _lib.LIB.la_gemm_noalloc(3, w.data_ptr(), None, 128, 64, x.data_ptr(), 4, y.data_ptr(), s) == _lib.LA_EINVAL
    # the workspace is intact after the rejections
    rng = np.random.default_rng(5)
    wb = bf16_bits(rng, (256, 128), 0.05)
    xb = bf16_bits(rng, (3, 128), 1.0)
    ref = _lib.la_debug_gemm(wb, xb, 0, 0)
    out = torch.zeros((3, 256), dtype=torch.bfloat16, device="cuda")
    run(0, wb.cuda(), None, xb.cuda(), out)
    assert np.all(np.abs(out.float().cpu().numpy() - ref) <= BF16_REL * np.abs(ref) + 1e-6)
