"""Batches past the grid's 65535 limit in y (70,000 tiny frames per launch).

The direct-load kernels walk images as blockIdx.y, blockIdx.y + gridDim.y,
...; the staged and streaming kernels fold images into their unit index.
Frames on both sides of the 65535 boundary (and the last) are compared with
the oracle for every kernel family: exact 2x down and up, any ratio, float32
(staged; wrap on the direct kernel), normalise, gray, and the filter
epilogues (streaming 3x3 and 5x5, the tile kernel for K = 1).
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N = 70000
PICK = [0, 1, 65534, 65535, 65536, N - 1]


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


def frames_u8(H, W, C, seed):
    return np.random.default_rng(seed).integers(0, 256, (N, H, W, C), dtype=np.uint8)


@pytest.mark.parametrize("geom", [(8, 8, 4, 4), (4, 4, 8, 8), (8, 8, 5, 7), (6, 10, 11, 13)])
@pytest.mark.parametrize("mode", [0, 1])
def test_u8_batch_past_grid_limit(rz, geom, mode):
    H, W, OH, OW = geom
    f = frames_u8(H, W, 3, H + W + mode)
    src = torch.from_numpy(f).cuda()
    dst = torch.zeros((N, OH, OW, 3), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(H, W, OH, OW, mode) as plan:
        rz.resize_u8_batch(plan, src, dst)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in PICK:
        want = oracle.linear_u8(f[n], OH, OW) if mode else oracle.nearest_u8(f[n], OH, OW)
        np.testing.assert_array_equal(got[n], want, err_msg=f"frame {n}")


@pytest.mark.parametrize("border", [0, 2])
def test_f32_batch_past_grid_limit(rz, border):
    f = (np.random.default_rng(3).random((N, 6, 7, 1)) * 255).astype(np.float32)
    src = torch.from_numpy(f).cuda()
    dst = torch.zeros((N, 9, 5, 1), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(6, 7, 9, 5, rz.RZ_LINEAR, border=border) as plan:
        rz.resize_f32_batch(plan, src, dst)
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in PICK:
        assert np.abs(got[n] - oracle.linear_f32(f[n], 9, 5, border)).max() <= 1e-4, n


def test_normalize_and_gray_batches_past_grid_limit(rz):
    f = frames_u8(8, 8, 3, 11)
    src = torch.from_numpy(f).cuda()
    mean, std = (0.485, 0.456, 0.406), (0.229, 0.224, 0.225)
    norm = torch.zeros((N, 3, 5, 5), dtype=torch.float32, device="cuda")
    gray = torch.zeros((N, 4, 4), dtype=torch.uint8, device="cuda")
    with rz.resize_plan_create(8, 8, 5, 5, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, norm, rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=mean, std=std))
    with rz.resize_plan_create(8, 8, 4, 4, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, gray, rz.make_epilogue(rz.RZ_EPI_GRAY_RGB))
    torch.cuda.synchronize()
    gn, gg = norm.cpu().numpy(), gray.cpu().numpy()
    for n in PICK:
        assert np.abs(gn[n] - oracle.linear_u8_normalize(f[n], 5, 5, mean, std)).max() <= 1e-4, n
        np.testing.assert_array_equal(gg[n], oracle.gray_resize_u8(f[n], 4, 4))


@pytest.mark.parametrize("K", [1, 3, 5])
def test_filter_batches_past_grid_limit(rz, K):
    f = (np.random.default_rng(K).random((N, 7, 9, 1)) * 255).astype(np.float32)
    w = np.random.default_rng(K + 1).random((K, K)).astype(np.float32)
    w /= w.sum()
    src = torch.from_numpy(f).cuda()
    dst = torch.zeros((N, 10, 6, 1), dtype=torch.float32, device="cuda")
    with rz.resize_plan_create(7, 9, 10, 6, rz.RZ_LINEAR) as plan:
        rz.resize_fused(plan, src, dst, rz.make_epilogue(rz.RZ_EPI_FILTER, wk=w))
        torch.cuda.synchronize()
    got = dst.cpu().numpy()
    for n in PICK:
        want = oracle.filter_centred(oracle.linear_f32(f[n], 10, 6)[:, :, 0], w)
        assert np.abs(got[n][:, :, 0] - want).max() <= 1e-4 + 2 * K * K * 2.0 ** -24 * 255, n
