"""The library's calls inside a captured CUDA graph.

Each call only launches kernels on the caller's stream (no synchronisation,
no allocation inside the library, workspaces passed in), so a sequence of
calls can be captured once and replayed.  Every replay must give the bits of
the eager calls (the kernels are deterministic).  The persistent BatchNorm
kernel carries a launch epoch in its workspace, so replaying the same
captured launch never matches a stale flag.  The device is prepared
(gbn_init) before capture."""

import pytest
import torch

from bwd_bn_pass_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _replay_matches(run, outs, reps=3):
    """run() issues the calls writing into `outs`; eager, then captured and
    replayed `reps` times, each replay bit-identical to the eager result."""
    torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(reps):
        for t in outs:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for t, r in zip(outs, ref):
            assert torch.equal(t, r)


@pytest.mark.parametrize("path", ["two-launch", "small-channel", "persistent"])
def test_batchnorm_in_a_graph(gbn, path):
    gbn.init(0)
    prev = gbn.bn_set_persistent_min_bytes(0 if path == "persistent" else 1 << 62)
    prev_small = gbn.bn_set_small_max_elems(0 if path == "two-launch" else 2048)
    try:
        inp = synth.bn_inputs(synth.BNCase("graph_bn", (16, 24, 14, 14), "bf16",
                                           mu_range=(-5.0, 5.0), seed=1101))
        x, dy = inp["x"].to(DEV), inp["dy"].to(DEV)
        g, b = inp["gamma"].to(DEV), inp["beta"].to(DEV)
        C = x.shape[1]
        y, dx = torch.empty_like(x), torch.empty_like(x)
        stats = gbn.bn_stats_tensor(C, x.device)
        grads = torch.empty(4 * C, device=DEV)
        ws = gbn.bn_workspace(x)

        def run():
            gbn.bn_forward_train(x, g, b, None, None, 0.1, 1e-5, y=y, stats=stats, ws=ws,
                                 act="relu")
            gbn.bn_backward(x, dy, stats, dx=dx, grads=grads, ws=ws, beta=b, act="relu")

        _replay_matches(run, [y, stats, dx, grads])
    finally:
        gbn.bn_set_persistent_min_bytes(prev)
        gbn.bn_set_small_max_elems(prev_small)


def test_rows_and_channels_last_in_a_graph(gbn):
    gbn.init(0)
    r = synth.rms_inputs(synth.RMSCase("graph_rms", 64, 4096, "bf16", seed=1103))
    x, dy, w = r["x"].to(DEV), r["dy"].to(DEV), r["w"].to(DEV)
    rstd = torch.rsqrt(x.float().pow(2).mean(dim=1) + 1e-5)
    dxr, dwr = torch.empty_like(x), torch.empty_like(w)
    wsr = gbn.rowwise_workspace(64, 4096, gbn.GBN_ROW_RMS, x.dtype, x.device)
    ln = synth.ln_inputs(synth.LNCase("graph_ln", 96, 1600, "bf16", seed=1105))
    d = {k: v.to(DEV) for k, v in ln.items() if torch.is_tensor(v)}
    mean = torch.zeros(96, device=DEV)
    lrstd = torch.ones(96, device=DEV)
    yl = torch.empty_like(d["inp"])
    zl = torch.empty_like(d["inp"])
    ni = synth.bn_inputs(synth.BNCase("graph_nhwc", (8, 32, 6, 6), "f32", seed=1107))
    xn = ni["x"].permute(0, 2, 3, 1).contiguous().to(DEV)
    dyn = ni["dy"].permute(0, 2, 3, 1).contiguous().to(DEV)
    yn, dxn = torch.empty_like(xn), torch.empty_like(xn)
    sn = gbn.bn_stats_tensor(32, xn.device)
    gn = torch.empty(4 * 32, device=DEV)
    wsn = gbn.bn_nhwc_workspace(xn)

    def run():
        gbn.rmsnorm_backward(dy, x, w, rstd, dx=dxr, dw=dwr, ws=wsr)
        gbn.layernorm_forward(d["inp"], d["gamma"], d["beta"], 1e-5, residual=d["residual"],
                              bias=d["bias"], mask=d["mask"], dropout_scale=ln["dropout_scale"],
                              y=yl, z=zl, mean=mean, rstd=lrstd)
        gbn.bn_nhwc_forward_train(xn, None, None, None, None, 0.1, 1e-5, y=yn, stats=sn,
                                  ws=wsn)
        gbn.bn_nhwc_backward(xn, dyn, sn, dx=dxn, grads=gn, ws=wsn)

    _replay_matches(run, [dxr, dwr, yl, zl, mean, lrstd, yn, sn, dxn, gn])
