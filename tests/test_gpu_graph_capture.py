"""Many resizes captured in one CUDA graph, replayed, checked against the oracle.

CUDA graphs pack many launches into one submission, which cuts the CPU's
scheduling cost per launch (CUDA interpolation page, hnwysp.cn/news/129086,
§8.1; the per-call overhead of many small kernels is the tracking paper's
§4.2 subject).  One graph here holds resize_u8 on an exact 2x, an exact 3:2
and an arbitrary geometry (bilinear) plus an arbitrary nearest one, a
float32 resize, a resize_fused normalise of a two-frame batch, a
resize_u8_multi launch of mixed jobs, and a chain in which each resize reads
the previous one's output.  The graph is replayed several times with new
input contents written in between; after every replay each output must equal
the oracle's result for the inputs of that replay (uint8 bit-exact, float32
within 1e-4).
"""
import numpy as np
import pytest

import oracle
from bilinear_image_resize_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_TOL = 1e-4


@pytest.fixture(scope="module")
def rz():
    import __graft_entry__
    __graft_entry__.build()
    import bilinear_image_resize_gb300 as m
    torch.cuda.set_device(0)
    return m


U8_CALLS = [  # (H, W, OH, OW, C, mode)
    (480, 640, 240, 320, 3, 1),      # exact 2x down
    (540, 960, 360, 640, 3, 1),      # exact 3:2 down
    (701, 1003, 333, 517, 3, 1),     # arbitrary ratio
    (190, 250, 420, 380, 4, 1),      # arbitrary upscale
    (701, 1003, 333, 517, 1, 0),     # nearest
]
MULTI_JOBS = [(100, 80, 33, 50), (64, 64, 128, 128), (37, 41, 37, 41), (90, 160, 45, 80)]


def test_graph_of_mixed_calls_matches_oracle_over_replays(rz):
    rng = np.random.default_rng(2024)
    s = torch.cuda.Stream()
    # inputs (rewritten before every replay) and outputs
    u8_src = [torch.empty((H, W, C), dtype=torch.uint8, device="cuda") for H, W, _, _, C, _ in U8_CALLS]
    u8_dst = [torch.empty((OH, OW, C), dtype=torch.uint8, device="cuda") for _, _, OH, OW, C, _ in U8_CALLS]
    u8_plans = [rz.resize_plan_create(H, W, OH, OW, m) for H, W, OH, OW, _, m in U8_CALLS]
    f_src = torch.empty((300, 200), dtype=torch.float32, device="cuda")
    f_dst = torch.empty((123, 456), dtype=torch.float32, device="cuda")
    f_plan = rz.resize_plan_create(300, 200, 123, 456, rz.RZ_LINEAR)
    n_src = torch.empty((2, 240, 320, 3), dtype=torch.uint8, device="cuda")
    n_dst = torch.empty((2, 3, 224, 224), dtype=torch.float32, device="cuda")
    n_plan = rz.resize_plan_create(240, 320, 224, 224, rz.RZ_LINEAR)
    n_epi = rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=synth.NORM_MEAN, std=synth.NORM_STD)
    m_src = [torch.empty((H, W, 3), dtype=torch.uint8, device="cuda") for H, W, _, _ in MULTI_JOBS]
    m_dst = [torch.empty((OH, OW, 3), dtype=torch.uint8, device="cuda") for _, _, OH, OW in MULTI_JOBS]
    m_jobs, _ = rz.make_jobs(m_src, m_dst)
    m_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # chain: 720p -> 360p (exact 2x) -> 240x427 (arbitrary) -> 480x854 (upscale)
    c_src = torch.empty((720, 1280, 3), dtype=torch.uint8, device="cuda")
    c_mid = torch.empty((360, 640, 3), dtype=torch.uint8, device="cuda")
    c_mid2 = torch.empty((240, 427, 3), dtype=torch.uint8, device="cuda")
    c_out = torch.empty((480, 854, 3), dtype=torch.uint8, device="cuda")
    c_plans = [rz.resize_plan_create(720, 1280, 360, 640, rz.RZ_LINEAR),
               rz.resize_plan_create(360, 640, 240, 427, rz.RZ_LINEAR),
               rz.resize_plan_create(240, 427, 480, 854, rz.RZ_LINEAR)]
    torch.cuda.synchronize()

    def calls():
        for p, a, b, (_, _, _, _, _, m) in zip(u8_plans, u8_src, u8_dst, U8_CALLS):
            rz.resize_u8(p, a, b, stream=s)
        rz.resize_f32(f_plan, f_src, f_dst, stream=s)
        rz.resize_fused(n_plan, n_src, n_dst, n_epi, stream=s)
        rz.resize_u8_multi(m_jobs, len(MULTI_JOBS), 3, rz.RZ_LINEAR, m_status, stream=s)
        rz.resize_u8(c_plans[0], c_src, c_mid, stream=s)
        rz.resize_u8(c_plans[1], c_mid, c_mid2, stream=s)
        rz.resize_u8(c_plans[2], c_mid2, c_out, stream=s)

    # one eager pass first (per-kernel attributes are set on first use)
    with torch.cuda.stream(s):
        calls()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    torch.cuda.synchronize()

    for rep in range(3):
        imgs = [rng.integers(0, 256, (H, W, C), dtype=np.uint8) for H, W, _, _, C, _ in U8_CALLS]
        fimg = (rng.random((300, 200)) * 255.0).astype(np.float32)
        nimg = rng.integers(0, 256, (2, 240, 320, 3), dtype=np.uint8)
        mimgs = [rng.integers(0, 256, (H, W, 3), dtype=np.uint8) for H, W, _, _ in MULTI_JOBS]
        cimg = synth.smooth_rgb(1280, 720, 100 + rep)
        for t, a in zip(u8_src, imgs):
            t.copy_(torch.from_numpy(a))
        f_src.copy_(torch.from_numpy(fimg))
        n_src.copy_(torch.from_numpy(nimg))
        for t, a in zip(m_src, mimgs):
            t.copy_(torch.from_numpy(a))
        c_src.copy_(torch.from_numpy(np.ascontiguousarray(cimg)))
        for t in u8_dst + m_dst + [c_mid, c_mid2, c_out]:
            t.fill_(0x5A)
        f_dst.fill_(-1.0)
        n_dst.fill_(-1.0)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()

        for img, out, (H, W, OH, OW, C, m) in zip(imgs, u8_dst, U8_CALLS):
            want = oracle.linear_u8(img, OH, OW) if m == 1 else oracle.nearest_u8(img, OH, OW)
            np.testing.assert_array_equal(out.cpu().numpy(), want, err_msg=f"replay {rep}: {H}x{W}->{OH}x{OW}")
        werr = np.max(np.abs(f_dst.cpu().numpy().astype(np.float64) - oracle.linear_f32(fimg, 123, 456).reshape(123, 456)))
        assert werr <= F32_TOL, (rep, werr)
        got = n_dst.cpu().numpy()
        for k in range(2):
            want = oracle.linear_u8_normalize(nimg[k], 224, 224, synth.NORM_MEAN, synth.NORM_STD)
            assert np.max(np.abs(got[k].astype(np.float64) - want)) <= F32_TOL, (rep, k)
        assert int(m_status.item()) == rz.RZ_OK
        for img, out, (H, W, OH, OW) in zip(mimgs, m_dst, MULTI_JOBS):
            np.testing.assert_array_equal(out.cpu().numpy(), oracle.linear_u8(img, OH, OW))
        e1 = oracle.linear_u8(cimg, 360, 640)
        e2 = oracle.linear_u8(e1, 240, 427)
        np.testing.assert_array_equal(c_out.cpu().numpy(), oracle.linear_u8(e2, 480, 854), err_msg=f"chain {rep}")

    for p in u8_plans + c_plans + [f_plan, n_plan]:
        assert rz.resize_plan_status(p) == rz.RZ_OK
        p.destroy()


def test_graph_of_many_small_resizes(rz):
    # 64 small resizes of distinct frames in one graph (the launch-bound case
    # graphs are for), replayed twice with new frames
    rng = np.random.default_rng(7)
    n = 64
    geo = (96, 128, 60, 80)
    plan = rz.resize_plan_create(*geo, rz.RZ_LINEAR)
    srcs = [torch.empty((96, 128, 3), dtype=torch.uint8, device="cuda") for _ in range(n)]
    dsts = [torch.empty((60, 80, 3), dtype=torch.uint8, device="cuda") for _ in range(n)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rz.resize_u8(plan, srcs[0], dsts[0], stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for a, b in zip(srcs, dsts):
            rz.resize_u8(plan, a, b, stream=s)
    for rep in range(2):
        imgs = [rng.integers(0, 256, (96, 128, 3), dtype=np.uint8) for _ in range(n)]
        for t, a in zip(srcs, imgs):
            t.copy_(torch.from_numpy(a))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for img, out in zip(imgs, dsts):
            np.testing.assert_array_equal(out.cpu().numpy(), oracle.linear_u8(img, 60, 80))
    plan.destroy()
