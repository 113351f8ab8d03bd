"""The device entry points captured into CUDA graphs.

Once a plan exists, sarbp_backproject, sarbp_range_compress and
sarbp_backproject_raw only enqueue kernels on the caller's stream (no
allocation, no synchronisation), so a
stream capture records them into a graph whose replays must give the eager
result bit for bit: the whole range-compression -> backprojection pipeline
then runs as one graph launch.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from domain_backprojection_sarbp_gb300 import Plan, RangeCompressor  # noqa: E402
from synth import chirp, scenes  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def scene():
    return scenes.make_scene(scenes.CONFIGS[1])


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("interp", ["linear", "sinc8", "nearest"])
def test_backprojection_graph_replays_the_eager_image(scene, interp):
    p = scene.params
    echoes, pos = _dev(scene.echoes), _dev(scene.antenna_pos)
    with Plan(p) as plan:
        eager = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
        plan.backproject(eager, echoes, pos, interp=interp)
        torch.cuda.synchronize()
        img = torch.full_like(eager, complex(5.0, 5.0))
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):               # warm-up outside the capture
            plan.backproject(img, echoes, pos, interp=interp, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.backproject(img, echoes, pos, interp=interp,
                             stream=torch.cuda.current_stream())
        for _ in range(3):
            img.fill_(complex(5.0, 5.0))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(img, eager), interp


def test_pipeline_graph(scene):
    """Raw chirps -> range compression -> backprojection as one graph; the
    replay equals the eager pipeline, and a new raw frame copied into the
    captured input buffer gives that frame's image."""
    p = scene.params
    ref = _dev(chirp.chirp().astype(np.complex64))
    tgt = np.array([[0.0, 0.0, 0.0], [12.0, -20.0, 0.0]])
    frames = []
    for amp in (1.0, 0.5):
        raw = chirp.raw_echoes(scene.antenna_pos, tgt, np.array([amp, 1.0]), p["r0"], p["nr"])
        frames.append(_dev(raw.astype(np.complex64)))
    pos = _dev(scene.antenna_pos)
    raw_buf = frames[0].clone()
    rc_out = torch.empty_like(raw_buf)
    img = torch.empty((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    with RangeCompressor(ref, p["na"], p["nr"]) as rc, Plan(p) as plan:
        def eager(raw):
            out = torch.empty_like(raw)
            rc(out, raw)
            im = torch.empty_like(img)
            plan.backproject(im, out, pos)
            torch.cuda.synchronize()
            return im
        want = [eager(f) for f in frames]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            rc(rc_out, raw_buf, stream=side)
            plan.backproject(img, rc_out, pos, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            s = torch.cuda.current_stream()
            rc(rc_out, raw_buf, stream=s)
            plan.backproject(img, rc_out, pos, stream=s)
        for f, w in zip(frames, want):
            raw_buf.copy_(f)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(img, w)
    assert not torch.equal(want[0], want[1])


def test_raw_entry_point_graph(scene):
    """sarbp_backproject_raw (compression fused with the echo table) captured
    into a graph: replays equal the eager call bit for bit, for two raw frames
    copied into the captured input."""
    p = scene.params
    ref = _dev(chirp.chirp().astype(np.complex64))
    tgt = np.array([[0.0, 0.0, 0.0], [12.0, -20.0, 0.0]])
    frames = [_dev(chirp.raw_echoes(scene.antenna_pos, tgt, np.array([amp, 1.0]), p["r0"],
                                    p["nr"]).astype(np.complex64)) for amp in (1.0, 0.5)]
    pos = _dev(scene.antenna_pos)
    raw_buf = frames[0].clone()
    img = torch.empty((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
    with RangeCompressor(ref, p["na"], p["nr"], "hamming", 0.8) as rc, Plan(p) as plan:
        want = []
        for f in frames:
            im = torch.empty_like(img)
            plan.backproject_raw(im, f, pos, rc)
            torch.cuda.synchronize()
            want.append(im)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            plan.backproject_raw(img, raw_buf, pos, rc, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.backproject_raw(img, raw_buf, pos, rc, stream=torch.cuda.current_stream())
        for f, w in zip(frames, want):
            raw_buf.copy_(f)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(img, w)
    assert not torch.equal(want[0], want[1])


def test_volume_and_height_map_graphs(scene):
    p = scene.params
    echoes, pos = _dev(scene.echoes), _dev(scene.antenna_pos)
    h = _dev(scenes.terrain(p["nx"], p["ny"], p["dx"], 5, relief=10.0, mean=5.0).astype(np.float32))
    with Plan(p) as vplan, Plan(p, height_range=(0.0, 10.0)) as hplan:
        def run(vol, img, stream=None):
            vplan.backproject_volume(vol, echoes, pos, 0.5, stream=stream)
            hplan.backproject_heights(img, echoes, pos, h, stream=stream)
        vol0 = torch.zeros((3, p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
        img0 = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
        run(vol0, img0)
        torch.cuda.synchronize()
        vol, img = torch.empty_like(vol0), torch.empty_like(img0)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run(vol, img, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(vol, img, stream=torch.cuda.current_stream())
        vol.zero_()
        img.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(vol, vol0) and torch.equal(img, img0)


def test_two_plans_on_two_streams_at_once(scene):
    """Plans are independent: two plans enqueued on two streams at the same
    time (linear and sinc, different images) give the images each computes
    alone, bit for bit."""
    p = scene.params
    echoes, pos = _dev(scene.echoes), _dev(scene.antenna_pos)
    with Plan(p) as pa, Plan(p) as pb:
        solo = []
        for plan, interp in ((pa, "linear"), (pb, "sinc8")):
            img = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
            plan.backproject(img, echoes, pos, interp=interp)
            torch.cuda.synchronize()
            solo.append(img)
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        both = [torch.zeros_like(solo[0]), torch.zeros_like(solo[1])]
        for _ in range(3):
            pa.backproject(both[0], echoes, pos, interp="linear", stream=sa)
            pb.backproject(both[1], echoes, pos, interp="sinc8", stream=sb)
        torch.cuda.synchronize()
        assert torch.equal(both[0], solo[0]) and torch.equal(both[1], solo[1])


def test_sinc_plan_captures_its_first_call(scene):
    """A plan made for sinc holds its coefficient rows from the start, so its
    very first sinc call can be captured; the replay equals an eager call on a
    plan that allocated them on first use."""
    p = scene.params
    echoes, pos = _dev(scene.echoes), _dev(scene.antenna_pos)
    with Plan(p) as lazy:
        eager = torch.zeros((p["ny"], p["nx"]), dtype=torch.complex64, device=DEV)
        lazy.backproject(eager, echoes, pos, interp="sinc8")
        torch.cuda.synchronize()
    with Plan(p, interp="sinc8") as plan:
        img = torch.zeros_like(eager)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.backproject(img, echoes, pos, interp="sinc8",
                             stream=torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(img, eager)
