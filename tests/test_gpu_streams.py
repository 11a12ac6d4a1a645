"""Every call runs on the caller's stream.

For each group of calls: every buffer the calls write (scratch included) is
overwritten with a fill pattern and the device synchronised, then the calls
run on the default stream.  The buffers are filled again, and the calls are
enqueued on a non-blocking side stream behind a spin kernel that keeps that
stream busy for a few milliseconds.  A kernel or memset that went to another
stream would run before its producers on the side stream and read the fill
pattern (or leave it in place); every buffer must instead come out identical
to the first run.  The groups: the layer step (24 experts, the full-size
tokens per expert), a decode-shaped forward, the MXFP8 forward, the FP4
backward's requantisations and the combine receive.  All are deterministic:
their random bits are counter-based.
"""
import numpy as np
import pytest
import torch

from precision_moe_numerics_gb300 import workloads as W

pytestmark = pytest.mark.gpu

STEP_BUFFERS = ("w1q", "w2q", "xq", "h", "hq", "z", "xt", "ht", "w1t", "w2t", "dy_r", "dy_t", "dy1_r", "dy1_t",
                "dh", "dx", "dw1", "dw2")


def flat(obj, names):
    """(name, tensor) for the named attributes (tuples of tensors flattened)"""
    out = []
    for n in names:
        v = getattr(obj, n)
        out.extend((n, t) for t in (v if isinstance(v, tuple) else (v,)))
    return out


def check_on_side_stream(pmn, run, outs, scratch=()):
    """outs: [(name, tensor)] that run() writes; scratch: tensors it uses as workspace"""
    def fill():  # the same pattern before both runs, so bytes no call writes compare equal too
        for t in [t for _, t in outs] + list(scratch):
            t.view(torch.uint8).fill_(0xA5)
        torch.cuda.synchronize()

    fill()
    run()
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    first = [t.clone() for _, t in outs]
    fill()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        torch.cuda._sleep(20_000_000)  # bounded spin: the side stream stays busy while the calls are enqueued
        run()
    side.synchronize()
    torch.cuda.synchronize()
    assert pmn.get_device_error() == 0
    for (name, b), a in zip(outs, first):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), "%s differs after the side-stream run" % name


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from precision_moe_numerics_gb300 import build, layer, pmn
    build.build()
    inp = W.moe_device(3, device="cuda", experts=24, tokens=1024)
    r = inp["routing"]
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    L = layer.ExpertLayerStep(inp["x"], inp["w1"], inp["w2"], inp["dy"], inp["dy1"], offs, r.real_rows, seed=5)
    L.step()
    torch.cuda.synchronize()
    return {"pmn": pmn, "layer": layer, "inp": inp, "r": r, "offs": offs, "L": L}


def test_step_runs_on_the_callers_stream(env):
    L = env["L"]
    check_on_side_stream(env["pmn"], L.step, flat(L, STEP_BUFFERS), scratch=(L.ws,))


def test_decode_forward_runs_on_the_callers_stream(env):
    """16 tokens routed top-8 over the layer's 24 experts (unpadded segments
    of a few rows: the 32-row tiles), against the step's NVFP4 weights"""
    L = env["L"]
    rng = np.random.default_rng(9)
    r = W.route_topk(rng.standard_normal((16, 24), dtype=np.float32), W.TOP_K, pad=1)
    x = torch.from_numpy(W.decode_x(r, 9, L.w1.shape[2]).view(np.int16)).view(torch.bfloat16).cuda()
    offs = torch.from_numpy(r.offsets.astype(np.int32)).cuda()
    dec = env["layer"].DecodeForward(x, L.w1q3(), L.w2q3(), offs, seed=5)
    check_on_side_stream(env["pmn"], dec.forward, flat(dec, ("xq", "h", "hq", "z")))


def test_mxfp8_forward_runs_on_the_callers_stream(env):
    inp = env["inp"]
    fw = env["layer"].MXFP8Forward(inp["x"], inp["w1"], inp["w2"], env["offs"])
    check_on_side_stream(env["pmn"], fw.forward, flat(fw, ("w1q", "w2q", "xq", "y", "hq", "z")))


def test_fp4_backward_requant_runs_on_the_callers_stream(env):
    """the NVFP4 requantisations of the saved W1 (per expert) and X (per
    token): a memset and three kernels each, the outer-scale output doubling
    as the reduction's scratch"""
    pmn, L = env["pmn"], env["L"]
    E, F2, D = L.w1.shape
    T = L.xq[0].shape[0]
    w = (torch.empty((E, D, F2 // 2), dtype=torch.uint8, device="cuda"),
         torch.empty((E, D, F2 // 16), dtype=torch.uint8, device="cuda"),
         torch.empty((E,), dtype=torch.float32, device="cuda"))
    x = (torch.empty((1, D, T // 2), dtype=torch.uint8, device="cuda"),
         torch.empty((1, D, T // 16), dtype=torch.uint8, device="cuda"),
         torch.empty((1,), dtype=torch.float32, device="cuda"))

    def run():
        pmn.requant_transpose_sr_nvfp4(*L.w1q, False, E, F2, D, 5, pmn.TAG_W1, out=w)
        pmn.requant_transpose_sr_nvfp4(*L.xq, True, 1, T, D, 5, pmn.TAG_X, out=x)

    check_on_side_stream(pmn, run, [("w1 requant", t) for t in w] + [("x requant", t) for t in x])


def test_combine_receive_runs_on_the_callers_stream(env):
    pmn, L, r = env["pmn"], env["L"], env["r"]
    idx = torch.from_numpy(r.token_rows()).cuda()
    gates = torch.from_numpy(r.gates).cuda()
    out = torch.empty((idx.shape[0], L.z[0].shape[1]), dtype=torch.bfloat16, device="cuda")
    check_on_side_stream(pmn, lambda: pmn.combine_receive_s2f6(L.z, 5, idx, gates, out=out), [("combine", out)])
