"""The tcgen05 GEMM alone against a float64 matmul of the same bf16 inputs:
shapes with many K slices per CTA (the shared-memory ring wraps), tiles
shared by several persistent CTAs, CTAs that own several tiles, ragged row
counts, several row chunks; plus row-count invariance."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def L():
    from lookahead_decoding_gb300 import lib
    return lib()


def case(n_out, K, rows, seed):
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(n_out, K, generator=g) * 0.05).to(torch.bfloat16)
    x = torch.randn(rows, K, generator=g).to(torch.bfloat16)
    ref = x.double().numpy() @ w.double().numpy().T
    return w, x, ref


@pytest.mark.parametrize("n_out,K,rows,n_cta", [
    (128, 64, 1, 1), (256, 512, 16, 0), (128, 4096, 76, 1), (384, 4096, 120, 0), (256, 4096, 33, 4),
    (128, 11008, 7, 0), (256, 1024, 256, 3), (128, 2048, 300, 7), (128, 640, 512, 0), (4096, 4096, 60, 0),
    (1024, 4096, 60, 148), (32000 // 125 * 4, 4096, 1, 0),
])
def test_gemm_matches_float64(n_out, K, rows, n_cta):
    w, x, ref = case(n_out, K, rows, n_out + K + rows)
    y = L().la_debug_gemm(w, x, n_cta)
    err = np.max(np.abs(y - ref)) / (np.max(np.abs(ref)) + 1e-9)
    assert err < 2e-5, err


def bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("K,rows,n_cta", [(4096, 24, 0), (4096, 60, 5), (512, 7, 0), (11008, 76, 2)])
def test_store_segments(K, rows, n_cta):
    w, x, ref = case(3 * 256, K, rows, 3 + K)
    y = L().la_debug_gemm(w, x, n_cta, mode=0, n_seg=3)
    assert np.max(np.abs(y - bf16(ref))) <= np.max(np.abs(ref)) * 2 ** -7


@pytest.mark.parametrize("K,rows,n_cta", [(4096, 24, 0), (4096, 60, 4), (512, 7, 0), (1408, 300, 2)])
def test_swiglu(K, rows, n_cta):
    w, x, g = case(256, K, rows, 5 + K)
    w2, _, _ = case(256, K, rows, 6 + K)
    u = x.double().numpy() @ w2.double().numpy().T
    ref = g / (1 + np.exp(-g)) * u
    y = L().la_debug_gemm(w, x, n_cta, mode=2, w2_bf16=w2)
    assert np.max(np.abs(y - ref)) <= np.max(np.abs(ref)) * 2 ** -7


@pytest.mark.parametrize("K,rows,n_cta", [(4096, 24, 0), (11008, 60, 4), (512, 7, 0)])
def test_resid(K, rows, n_cta):
    w, x, ref = case(256, K, rows, 7 + K)
    y0 = np.random.default_rng(1).normal(size=ref.shape).astype(np.float32)
    y = L().la_debug_gemm(w, x, n_cta, mode=1, y_in=y0)
    assert np.max(np.abs(y - (y0 + ref))) < 1e-4 * (np.max(np.abs(ref)) + 1)


def test_rows_do_not_change_other_rows_bits():
    w, x, _ = case(256, 4096, 200, 1)
    full = L().la_debug_gemm(w, x, 0)
    for r in (1, 13, 64, 199):
        part = L().la_debug_gemm(w, x[:r].clone(), 0)
        assert np.array_equal(part.view(np.uint32), full[:r].view(np.uint32))


PAIR = 16   # LA_GEMM_PAIR: units of one atom of two adjacent output tiles


@pytest.mark.parametrize("n_out,K,rows,n_cta", [
    (256, 64, 1, 1), (512, 4096, 60, 0), (256, 11008, 76, 3), (4096, 4096, 60, 0), (1024, 1024, 256, 5),
    (512, 2048, 300, 7), (32000 // 125 * 4, 4096, 13, 0),
])
def test_pair_units_logits_match_float64(n_out, K, rows, n_cta):
    """Units of two output tiles (as the model's QKV, O, down and head GEMMs
    stream them): fp32 results against a float64 matmul, with tiles shared by
    up to a dozen CTAs, the split reduction and ragged rows."""
    w, x, ref = case(n_out, K, rows, 11 + n_out + K + rows)
    y = L().la_debug_gemm(w, x, n_cta, mode=3 | PAIR)
    err = np.max(np.abs(y - ref)) / (np.max(np.abs(ref)) + 1e-9)
    assert err < 2e-5, err


@pytest.mark.parametrize("K,rows,n_cta", [(4096, 24, 0), (4096, 60, 5), (512, 7, 0), (11008, 76, 2)])
def test_pair_units_store_segments(K, rows, n_cta):
    w, x, ref = case(3 * 512, K, rows, 13 + K)
    y = L().la_debug_gemm(w, x, n_cta, mode=0 | PAIR, n_seg=3)
    assert np.max(np.abs(y - bf16(ref))) <= np.max(np.abs(ref)) * 2 ** -7


@pytest.mark.parametrize("K,rows,n_cta", [(4096, 24, 0), (11008, 60, 4), (512, 7, 0)])
def test_pair_units_resid(K, rows, n_cta):
    w, x, ref = case(512, K, rows, 17 + K)
    y0 = np.random.default_rng(2).normal(size=ref.shape).astype(np.float32)
    y = L().la_debug_gemm(w, x, n_cta, mode=1 | PAIR, y_in=y0)
    assert np.max(np.abs(y - (y0 + ref))) < 1e-4 * (np.max(np.abs(ref)) + 1)


def test_pair_units_rows_do_not_change_other_rows_bits():
    w, x, _ = case(512, 4096, 200, 3)
    full = L().la_debug_gemm(w, x, 0, mode=3 | PAIR)
    for r in (1, 13, 64, 199):
        part = L().la_debug_gemm(w, x[:r].clone(), 0, mode=3 | PAIR)
        assert np.array_equal(part.view(np.uint32), full[:r].view(np.uint32))
