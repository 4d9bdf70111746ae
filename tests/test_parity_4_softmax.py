"""GPU parity of softmax_rows (the Gluon Multi-CTA tutorial's multi-CTA row
softmax) against the fp64 oracle: the tutorial's test shapes (64 x 64,
64 x 256, 16 x 65536), every cluster size (1, 2, 4, 8, 16 CTAs per row),
ragged and misaligned rows, in-place use, large-magnitude rows and long
rows with many more rows than resident clusters.
Acceptance: |y - y_ref| <= 1e-5 * y_ref + 1e-30 per element (fp32 exp and a
tree sum of at most 2^18 terms stay well inside 1e-5 relative; the absolute
term only covers results that underflow fp32)."""

import numpy as np
import pytest

import datagen
import dense_gemm_06_gb300 as lg
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lg.load()


def run_softmax(M, N, ld_pad=0, scale=1.0, dist="normal", seed=0, inplace=False, offset=0):
    import torch
    ldx = N + ld_pad
    x = (datagen.logical(M, ldx, dtype="f32", dist=dist, seed=seed) * scale).astype(np.float32)
    flat = np.concatenate([np.zeros(offset, np.float32), x.ravel()])
    dx = torch.from_numpy(flat).cuda()
    xp = int(dx.data_ptr()) + 4 * offset
    if inplace:
        dy, yp, ldy = dx, xp, ldx
    else:
        ldy = N + 3
        dy = torch.full((M * ldy,), float("nan"), device="cuda")
        yp = int(dy.data_ptr())
    lg.check(lg.softmax_rows(M, N, xp, ldx, yp, ldy), "softmax_rows")
    lg.check(lg.gemm_check_device_error(), "device error word")
    torch.cuda.synchronize()
    out = dy.cpu().numpy()
    if inplace:
        out = out[offset:]
    y = out.reshape(M, -1)[:, :N].astype(np.float64)
    y_ref = oracle.softmax_ref(M, N, x.ravel(), ldx)
    err = np.abs(y - y_ref)
    lim = 1e-5 * y_ref + 1e-30
    assert np.all(np.isfinite(y)) and np.all(err <= lim), \
        f"{M}x{N}: worst err/bound {np.max(err / lim):.3g}"
    if not inplace and ldy > N:
        assert np.all(np.isnan(out.reshape(M, ldy)[:, N:])), "padding of y was written"
    return y


@pytest.mark.parametrize("M,N", [(64, 64), (64, 256), (16, 2 ** 16)])
def test_tutorial_shapes(M, N):
    run_softmax(M, N, seed=M + N)


@pytest.mark.parametrize("N", [16384, 16385, 32768, 32769, 65537, 131072, 200003, 262144,
                               524288])
def test_every_cluster_size(N):
    # 1 CTA per row up to 32768 columns, then clusters of 2, 4, 8, 16
    run_softmax(3, N, seed=N % 97)


@pytest.mark.parametrize("M,N", [(1, 1), (5, 3), (37, 1000), (7, 4097), (2, 30001)])
def test_ragged_rows(M, N):
    run_softmax(M, N, ld_pad=5, seed=M * N % 101)


def test_misaligned_scalar_path_and_inplace():
    run_softmax(9, 5000, ld_pad=1, offset=1, seed=3)           # 4-byte aligned only
    run_softmax(9, 40000, ld_pad=0, seed=4, inplace=True)       # y is x
    run_softmax(4, 100000, ld_pad=2, offset=3, seed=5, inplace=True)


def test_large_magnitudes_are_stable():
    y = run_softmax(6, 70000, scale=40.0, seed=6)    # |x| up to ~200: exp would overflow unshifted
    assert np.allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-5)
    run_softmax(6, 3000, dist="pm1", scale=1e-3, seed=7)  # nearly uniform rows


@pytest.mark.parametrize("M,N,ld_pad", [(1000, 40000, 0), (300, 65540, 4), (64, 262144, 0),
                                        (200, 131073, 3), (152, 98304, 0)])
def test_long_rows_many_per_cluster(M, N, ld_pad):
    # more rows than resident clusters: each cluster walks several rows and
    # prefetches the next one while reducing the current one
    run_softmax(M, N, ld_pad=ld_pad, seed=(M + N) % 89)
