"""proj_gemv_static -- the entry point that allocates no device memory.

It serves callers that may not allocate: a plugin or custom operator that a
host framework hands only its input and output buffers (the framework's
allocator owns the device memory), or latency-critical code that cannot
afford cudaMalloc/cudaFree (they can stall the whole device and can fail at
run time).  Its scratch is a small static array inside the library, shared
by every call on a device.

Each case calls it twice in a row on fresh inputs -- so the second call
runs on the scratch the first one left behind -- and checks both outputs
against the FP64 oracle under the parity tests' contract (relative L2,
per-row bound, probe rows equal to the scaled weight column), against
proj_run's output under the same contract, and bit for bit against the
ring-form GEMV of proj_run_ex, which runs the same kernel on the same
partition of W.  This file is named to be collected last; it passes alone
in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_projection_layers_gb300 import binding as B
from gemv_projection_layers_gb300 import workloads as wl
from oracle import oracle

pytestmark = pytest.mark.gpu


def _device_weights(spec, seed):
    W = wl.make_weights(spec, seed)
    if spec.weight_dtype == "fp32":
        return torch.from_numpy(W).cuda(), B.PROJ_FP32, torch.float32
    return (torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16), B.PROJ_BF16,
            torch.bfloat16)


@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("layer", [s.name for s in wl.LAYERS])
def test_static_scratch_gemv_matches_proj_run(layer, m):
    assert torch.cuda.is_available()
    B.load()
    spec = wl.LAYER_BY_NAME[layer]
    Wd, dt, odt = _device_weights(spec, 3)
    h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, dt, 0, 16)
    try:
        n_out = B.proj_out_features(h, m)  # the unpooler computes its first 1024 rows
        acts = [wl.make_activations(spec, m, seed, outliers=bool(seed % 2)) for seed in (5, 6)]
        xs = [torch.from_numpy(a.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
              for a in acts]
        got = [torch.full((m, n_out), float("nan"), dtype=odt, device="cuda") for _ in xs]
        for x, o in zip(xs, got):  # two calls in a row
            B.proj_gemv_static(Wd, dt, n_out, spec.K, x, m, o)
        ref = [torch.full((m, n_out), float("nan"), dtype=odt, device="cuda") for _ in xs]
        for x, o in zip(xs, ref):
            B.proj_run(h, x, m, o)
        # the ring-form GEMV over the same partition (min(SMs, 256, N) CTAs)
        ring = [torch.full((m, n_out), float("nan"), dtype=odt, device="cuda") for _ in xs]
        grid = min(B.proj_num_sms(), 256)
        for x, o in zip(xs, ring):
            B.proj_run_ex(h, x, m, o, kernel=B.PROJ_KERNEL_GEMV, grid=grid)
        torch.cuda.synchronize()
        assert B.proj_device_status(h) == 0
        B.proj_gemv_static(Wd, dt, n_out, spec.K, xs[1], m, got[1])  # the last static call
        assert B.proj_gemv_static_status() == 0
        W = wl.make_weights(spec, 3)
        for call, (a, g, r, q) in enumerate(zip(acts, got, ref, ring)):
            g64 = g.float().cpu().numpy().astype(np.float64)
            exact = oracle.reference(layer, a.x_bits, W)[:, :n_out]
            res = oracle.check(layer, g64, exact, a.probe_rows)
            assert res["ok"], (layer, m, call, "oracle", res)
            r64 = r.float().cpu().numpy().astype(np.float64)
            res = oracle.check(layer, g64, r64, a.probe_rows)
            assert res["ok"], (layer, m, call, "proj_run", res)
            assert torch.equal(g.view(torch.int32 if odt == torch.float32 else torch.int16),
                               q.view(torch.int32 if odt == torch.float32 else torch.int16)), \
                (layer, m, call, "ring-form GEMV differs")
    finally:
        B.proj_destroy(h)


@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("layer", ["qkv_gate", "router"])
def test_static_scratch_gemv_in_a_cuda_graph(layer, m):
    """After one eager call (the per-device set-up), two calls captured on a
    side stream -- each a memset node and the kernel -- replay with fresh x
    copied into the captured input buffers and give, bit for bit, the eager
    call's output on the same x."""
    assert torch.cuda.is_available()
    B.load()
    spec = wl.LAYER_BY_NAME[layer]
    Wd, dt, odt = _device_weights(spec, 4)
    N, K = spec.N, spec.K
    ibits = torch.int32 if odt == torch.float32 else torch.int16

    def xs_for(seed):
        a = wl.make_activations(spec, m, seed)
        return torch.from_numpy(a.x_bits.view(np.int16)).cuda().view(torch.bfloat16)

    def eager(x):
        o = torch.full((m, N), float("nan"), dtype=odt, device="cuda")
        B.proj_gemv_static(Wd, dt, N, K, x, m, o)
        torch.cuda.synchronize()
        return o

    eager(xs_for(10))  # set-up happens outside the capture
    xin = [torch.empty((m, K), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs = [torch.full((m, N), float("nan"), dtype=odt, device="cuda") for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for x, o in zip(xin, outs):
            B.proj_gemv_static(Wd, dt, N, K, x, m, o, stream=s)
    for replay, seeds in enumerate(((11, 12), (13, 14))):
        fresh = [xs_for(sd) for sd in seeds]
        for dst, src in zip(xin, fresh):
            dst.copy_(src)
        for o in outs:
            o.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert B.proj_gemv_static_status(s) == 0
        for x, o in zip(fresh, outs):
            want = eager(x)
            assert torch.equal(o.view(ibits), want.view(ibits)), (layer, m, replay)


def test_static_scratch_gemv_rejects_sizes_beyond_its_limits():
    assert torch.cuda.is_available()
    B.load()
    W = torch.zeros((64, 1024), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((3, 1024), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_gemv_static(W, B.PROJ_BF16, 64, 1024, x, 3, out)
    assert e.value.status == B.PROJ_EUNSUPPORTED
    assert "m > 2" in B.last_cuda_error()
    for K in (1536, 16384):  # not a multiple of 1024; beyond the 8192 columns x staging holds
        with pytest.raises(B.ProjError) as e:
            B.proj_gemv_static(W, B.PROJ_BF16, 4, K, x, 1, out)
        assert e.value.status == B.PROJ_EUNSUPPORTED
        assert "K must be" in B.last_cuda_error()
