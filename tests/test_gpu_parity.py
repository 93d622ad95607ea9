"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Contract (muse_bf16_proj guide, ch. 1, §1.5 "What counts as correct"):
relative L2 per output <= 1e-2 (router 1e-4), probe rows within 1e-3 (and,
stronger, exactly equal to the scaled weight column), no row over 5x the
bound, no NaN/Inf.  Shapes: the five layers at the six scored token counts
and the awkward ones (§1.2), two weight seeds, normal and outlier inputs.
Small m and the scored 128 and 256 tokens are compared in full; the other
large m on sampled token rows (all of their outputs), which always include
the probe rows.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from gemv_projection_layers_gb300 import binding as B
from gemv_projection_layers_gb300 import workloads as wl
from oracle import oracle

pytestmark = pytest.mark.gpu

FULL_ORACLE_MAX_M = 33
FULL_ORACLE_M = (128, 256)  # the scored wide token counts: every output checked
SAMPLED_ROWS = 20
M_SCORED = (1, 8, 16, 32, 128, 256)
M_AWKWARD = (2, 3, 5, 7, 9, 33, 130, 512, 1000)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    B.load()
    return torch.device("cuda:0")


_cache = {}


def prepared(layer, seed, flags=0):
    key = (layer, seed, flags)
    if key not in _cache:
        spec = wl.LAYER_BY_NAME[layer]
        Wnp = wl.make_weights(layer, seed)
        if spec.weight_dtype == "fp32":
            Wd = torch.from_numpy(Wnp).cuda()
            dt = B.PROJ_FP32
        else:
            Wd = torch.from_numpy(Wnp.view(np.int16)).cuda().view(torch.bfloat16)
            dt = B.PROJ_BF16
        h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, dt, flags, 1024)
        _cache[key] = (h, Wnp, Wd)
    return _cache[key]


def to_dev_x(x_bits):
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda().view(torch.bfloat16)


def run(layer, h, x_dev, m, **kw):
    spec = wl.LAYER_BY_NAME[layer]
    n_out = B.proj_out_features(h, m)
    dt = torch.float32 if spec.out_dtype == "fp32" else torch.bfloat16
    out = torch.full((m, n_out), float("nan"), dtype=dt, device="cuda")
    if kw:
        B.proj_run_ex(h, x_dev, m, out, torch.cuda.current_stream(), **kw)
    else:
        B.proj_run(h, x_dev, m, out, torch.cuda.current_stream())
    torch.cuda.synchronize()
    return out


def out_f64(out):
    return out.float().cpu().numpy().astype(np.float64)


def reference_rows(layer, act, W, rows):
    """FP64 reference of whole output rows (tokens) `rows`."""
    return oracle.reference(layer, act.x_bits[rows], W)


def check_case(layer, seed, outliers, m, h=None, W=None, **kw):
    if h is None:
        h, W, _ = prepared(layer, seed)
    act = wl.make_activations(layer, m, seed, outliers)
    out = out_f64(run(layer, h, to_dev_x(act.x_bits), m, **kw))
    if m <= FULL_ORACLE_MAX_M or m in FULL_ORACLE_M:
        rows = np.arange(m)
    else:
        rng = np.random.default_rng(m * 7 + seed)
        pick = rng.choice(m, size=min(SAMPLED_ROWS, m), replace=False)
        rows = np.unique(np.concatenate([pick, [m - 1], act.probe_rows])).astype(np.int64)
    ref = reference_rows(layer, act, W, rows)
    probe_local = [int(np.flatnonzero(rows == p)[0]) for p in act.probe_rows]
    res = oracle.check(layer, out[rows], ref, probe_local)
    assert res["ok"], (layer, seed, outliers, m, res)
    # probe rows: exactly the scaled weight column (bf16 out: exact in bf16)
    n_out = out.shape[1]
    for r, c, e, s in zip(act.probe_rows, act.probe_cols, act.probe_exp, act.probe_sign):
        if W.dtype == np.float32:
            col = W[:n_out, c].astype(np.float64)
        else:
            col = oracle.bf16_bits_to_f64(W[:n_out, c])
        assert np.array_equal(out[r], float(s) * 2.0 ** int(e) * col), (layer, m, int(r))
    return out


@pytest.mark.parametrize("m", M_SCORED + M_AWKWARD)
@pytest.mark.parametrize("layer", [s.name for s in wl.LAYERS])
def test_parity_all_shapes(dev, layer, m):
    combos = [(0, False), (1, True)]
    if m <= FULL_ORACLE_MAX_M or m in FULL_ORACLE_M:
        combos += [(0, True), (1, False)]
    for seed, outl in combos:
        check_case(layer, seed, outl, m)


@pytest.mark.parametrize("layer,m", [("o", 1), ("o", 33), ("unpooler", 8), ("qkv_gate", 130),
                                     ("pooler", 16)])
def test_split_partitions_and_determinism(dev, layer, m):
    """Every partition and both split-K combine modes of the stream-K
    tensor-core kernel meet the contract and are bitwise reproducible."""
    h, W, _ = prepared(layer, 0)
    sms = B.proj_num_sms()
    modes = [B.PROJ_REDUCE_DISTRIBUTED]
    if m <= 32:
        modes.append(B.PROJ_REDUCE_OWNER)
    for reduce in modes:
        for grid in (1, 7, 64, sms - 1, sms):
            kw = dict(grid=grid, reduce=reduce, kernel=B.PROJ_KERNEL_TILE)
            a = check_case(layer, 0, True, m, h=h, W=W, **kw)
            b = check_case(layer, 0, True, m, h=h, W=W, **kw)
            assert np.array_equal(a, b), (layer, m, grid, reduce)
    assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer,m", [("o", 1), ("pooler", 16), ("qkv_gate", 32), ("o", 33),
                                     ("unpooler", 64), ("qkv_gate", 130), ("pooler", 256),
                                     ("qkv_gate", 512), ("o", 1000), ("router", 1),
                                     ("router", 3), ("router", 16), ("router", 130),
                                     ("router", 256), ("router", 1000)])
def test_cluster_sizes_and_determinism(dev, layer, m):
    """The cluster split-K kernel at every cluster size (1..16 CTAs sharing K)
    meets the contract and is bitwise reproducible; for the router this is the
    FP32-FMA cluster kernel (fp32 weights as they are)."""
    h, W, _ = prepared(layer, 0)
    if layer == "router" and m >= 25:
        assert "cluster" in B.proj_describe(h, m)
    elif layer == "o" and m >= 129:
        assert B.proj_describe(h, m).startswith("tc_pair")
    elif layer != "router" and m >= 33:
        assert "cluster" in B.proj_describe(h, m)
    for cs in range(1, 17):
        kw = dict(grid=cs, kernel=B.PROJ_KERNEL_CLUSTER)
        a = check_case(layer, 0, True, m, h=h, W=W, **kw)
        b = check_case(layer, 0, True, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (layer, m, cs)
    assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer,m", [("router", 3), ("router", 256), ("qkv_gate", 16),
                                     ("unpooler", 8), ("o", 130), ("pooler", 64)])
def test_cluster_groups_and_determinism(dev, layer, m):
    """Several clusters per output tile, their partials summed through global
    memory by whichever finishes last, in a fixed order: meets the contract,
    is bitwise reproducible, and leaves its counters at zero (a second call
    would go wrong otherwise)."""
    h, W, _ = prepared(layer, 1)
    sms = B.proj_num_sms()
    # a forced cluster shape keeps the smallest token tile covering m
    spec = wl.LAYER_BY_NAME[layer]
    # (the router's FP32-FMA kernel takes token tiles of at most 64)
    bn = next(b for b in (16, 32, 64, 128, 256) if m <= b or b == 256)
    if layer == "router":
        bn = min(bn, 64)
    tiles = B.proj_out_features(h, m) // 128 * -(-m // bn)
    kb = spec.K // 64
    ran = 0
    for cs, kg in ((1, 2), (2, 3), (4, 2), (8, 4), (16, 2), (3, 5), (1, 16), (5, 7)):
        if tiles * cs * kg > sms or cs * kg > kb:
            continue
        kw = dict(grid=cs, groups=kg, kernel=B.PROJ_KERNEL_CLUSTER)
        a = check_case(layer, 1, True, m, h=h, W=W, **kw)
        b = check_case(layer, 1, True, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (layer, m, cs, kg)
        ran += 1
    assert ran >= 1
    assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer,m", [("o", 128), ("qkv_gate", 128), ("pooler", 256),
                                     ("unpooler", 256), ("qkv_gate", 130), ("pooler", 65),
                                     ("o", 512), ("unpooler", 1000), ("qkv_gate", 33),
                                     ("unpooler", 96)])
def test_pair_shapes_and_determinism(dev, layer, m):
    """The CTA-pair tensor-core kernel (two CTAs per M = 256 MMA, K split
    across the pairs of a cluster whose partials meet in L2): the dispatch
    form on o above 128 tokens and on the unpooler from 192; at every token
    tile and several K splits it meets the contract and is bitwise
    reproducible (two calls in a row)."""
    want_pair = (layer == "o" and m >= 129) or (layer == "unpooler" and m >= 192)
    for seed in (0, 1):
        h, W, _ = prepared(layer, seed)
        assert B.proj_describe(h, m).startswith("tc_pair") == want_pair, B.proj_describe(h, m)
        ran = 0
        for bn in (64, 128, 256):
            for kg in (0, 1, 2, 3, 5, 8):
                kw = dict(kernel=B.PROJ_KERNEL_PAIR, tile_n=bn, groups=kg)
                try:
                    B.proj_describe_ex(h, m, **kw)
                except B.ProjError as e:  # < 4 k-blocks per CTA, or a split over > 1 wave
                    assert e.status == B.PROJ_EUNSUPPORTED
                    continue
                a = check_case(layer, seed, seed == 1, m, h=h, W=W, **kw)
                b = check_case(layer, seed, seed == 1, m, h=h, W=W, **kw)
                assert np.array_equal(a, b), (layer, m, seed, kw)
                ran += 1
        assert ran >= 3
        assert B.proj_device_status(h) == 0


def test_pair_rejections(dev):
    h, _, _ = prepared("o", 0)
    x = torch.zeros((128, 1024), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((128, 8192), dtype=torch.bfloat16, device="cuda")
    for kw in (dict(kernel=B.PROJ_KERNEL_PAIR, tile_n=32),        # token tiles of 64..256
               dict(kernel=B.PROJ_KERNEL_PAIR, grid=4),           # no grid for the pair kernel
               dict(kernel=B.PROJ_KERNEL_PAIR, groups=9),         # clusters of at most 16 CTAs
               dict(kernel=B.PROJ_KERNEL_PAIR, groups=5),         # o: 16 k-blocks, < 4 per CTA
               dict(kernel=B.PROJ_KERNEL_PAIR, variant=B.PROJ_VARIANT_EXPWIN12)):
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x, 128, out, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED, kw
    hr, _, _ = prepared("router", 0)
    xr = torch.zeros((128, 8192), dtype=torch.bfloat16, device="cuda")
    orr = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(hr, xr, 128, orr, kernel=B.PROJ_KERNEL_PAIR)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("layer,m", [(l, m) for l in ("qkv_gate", "o", "pooler", "unpooler")
                                     for m in (1, 2, 3, 5, 7, 8)] +
                         [("o", 9), ("o", 16), ("o", 17), ("o", 32), ("unpooler", 9),
                          ("unpooler", 16)])
def test_mma_gemv(dev, layer, m):
    """The bf16 layers' few-token GEMV on the warp-level tensor-core MMA (W in
    fragment order, whole 16-row blocks per CTA): the dispatch form at
    3 <= m <= 8, forced at m <= 8 and at several CTA counts (up to four
    blocks per CTA); meets the contract and is bitwise reproducible."""
    for seed in (0, 1):
        h, W, _ = prepared(layer, seed)
        nb = B.proj_out_features(h, m) // 16
        if (3 <= m <= 8 and layer in ("o", "unpooler")) or (layer == "o" and 9 <= m <= 16):
            assert "gemv_mma" in B.proj_describe(h, m)
        for kw in (dict(), dict(kernel=B.PROJ_KERNEL_MMA),
                   dict(kernel=B.PROJ_KERNEL_MMA, grid=-(-nb // 4)),
                   dict(kernel=B.PROJ_KERNEL_MMA, grid=37)):
            if m <= 2 and not kw:
                continue
            if kw.get("grid") and -(-nb // kw["grid"]) > 4:
                continue
            a = check_case(layer, seed, seed == 1, m, h=h, W=W, **kw)
            b = check_case(layer, seed, seed == 1, m, h=h, W=W, **kw)
            assert np.array_equal(a, b), (layer, m, seed, kw)
        assert B.proj_device_status(h) == 0


def test_mma_gemv_rejections(dev):
    h, _, _ = prepared("pooler", 0)
    x = torch.zeros((16, 8192), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((16, 4096), dtype=torch.bfloat16, device="cuda")
    for m, kw in ((9, dict(kernel=B.PROJ_KERNEL_MMA)),    # x for 16 tokens does not fit at K = 8192
                  (8, dict(kernel=B.PROJ_KERNEL_MMA, grid=16)),   # 16 blocks per CTA
                  (8, dict(kernel=B.PROJ_KERNEL_MMA, variant=B.PROJ_VARIANT_EXPWIN12))):
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x, m, out, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED
    hr, _, _ = prepared("router", 0)
    xr = torch.zeros((8, 8192), dtype=torch.bfloat16, device="cuda")
    orr = torch.zeros((8, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(hr, xr, 8, orr, kernel=B.PROJ_KERNEL_MMA)
    assert e.value.status == B.PROJ_EUNSUPPORTED


def check_outputs(layer, seed, outliers, m, h, W, configs):
    """Run every config (proj_run_ex keyword sets) on one seeded input; check
    each against one FP64 reference, probe rows exactly, each config twice
    for bitwise reproducibility.  Configs the library rejects with
    PROJ_EUNSUPPORTED are skipped; returns the configs that ran."""
    act = wl.make_activations(layer, m, seed, outliers)
    x = to_dev_x(act.x_bits)
    ref = oracle.reference(layer, act.x_bits, W)
    ran = []
    for kw in configs:
        try:
            B.proj_describe_ex(h, m, **{k: v for k, v in kw.items() if k != "stamps"})
        except B.ProjError as e:
            assert e.status == B.PROJ_EUNSUPPORTED, (layer, m, kw)
            continue
        a = out_f64(run(layer, h, x, m, **kw))
        b = out_f64(run(layer, h, x, m, **kw))
        assert np.array_equal(a, b), (layer, m, seed, kw)
        res = oracle.check(layer, a, ref, list(act.probe_rows))
        assert res["ok"], (layer, seed, outliers, m, kw, res)
        n_out = a.shape[1]
        for r, c, e, sg in zip(act.probe_rows, act.probe_cols, act.probe_exp, act.probe_sign):
            col = oracle.bf16_bits_to_f64(W[:n_out, c])
            assert np.array_equal(a[r], float(sg) * 2.0 ** int(e) * col), (layer, m, kw, int(r))
        ran.append(kw)
    return ran


@pytest.mark.parametrize("m", [3, 5, 7, 8, 9, 16, 17, 31, 32])
@pytest.mark.parametrize("layer", ["qkv_gate", "o", "pooler", "unpooler"])
def test_rows_gemv(dev, layer, m):
    """The row-run warp-MMA GEMV (whole row runs per CTA streamed into a
    shared-memory ring -- from the packed run layout at the SM-count grid,
    through 3-D tensor copies of the row-major W at other grids -- and x
    fragments from global memory, the in-step column assignment shared by
    both operands): the chosen ring shape and forced stages of 1 and 2 steps
    per warp (many ring laps), the SM-count grid and two odd grids (runs one
    row shorter than the longest, partial last blocks), all four
    seed/outlier inputs; the contract, exact probe rows, bitwise
    reproducibility."""
    sms = B.proj_num_sms()
    if layer in ("qkv_gate", "pooler") and 3 <= m <= 8:  # the dispatch form there
        assert B.proj_describe(prepared(layer, 0)[0], m).startswith("gemv_rows")
    for seed, outl in ((0, False), (0, True), (1, False), (1, True)):
        h, W, _ = prepared(layer, seed)
        configs = [dict(kernel=B.PROJ_KERNEL_ROWS, groups=ks, grid=grid)
                   for ks in (0, 1, 2) for grid in (0, sms - 3, 131)]
        ran = check_outputs(layer, seed, outl, m, h, W, configs)
        assert any(kw["grid"] == 0 and kw["groups"] == 0 for kw in ran), (layer, m)
        assert B.proj_device_status(h) == 0


def test_rows_gemv_stamps_and_rejections(dev):
    """The phase stamps are written per CTA in order (the row-run kernel and
    the tensor-core cluster and CTA-pair kernels); shapes outside the
    row-run kernel's range are rejected before any launch."""
    h, W, _ = prepared("pooler", 0)
    m = 16
    act = wl.make_activations("pooler", m, 0, False)
    x = to_dev_x(act.x_bits)
    G = B.proj_num_sms()
    st = torch.zeros((G, 8), dtype=torch.int64, device="cuda")
    out = run("pooler", h, x, m, kernel=B.PROJ_KERNEL_ROWS, stamps=st)
    ref = oracle.reference("pooler", act.x_bits, W)
    assert oracle.check("pooler", out_f64(out), ref, list(act.probe_rows))["ok"]
    t = st.cpu().numpy()[:, [0, 1, 5, 7]]  # entry, wait passed, main loop done, exit
    assert (t > 0).all()
    assert (np.diff(t, axis=1) >= 0).all()
    # the tensor-core kernels: every phase stamped, in order, per CTA
    for layer, mm, kw in (("pooler", 128, {}), ("o", 256, {}),
                          ("pooler", 256, dict(kernel=B.PROJ_KERNEL_PAIR, groups=2))):
        hh, WW, _ = prepared(layer, 0)
        desc = B.proj_describe_ex(hh, mm, **kw)
        ctas = int(desc.split("CTAs=")[1].split()[0])
        a2 = wl.make_activations(layer, mm, 0, False)
        st2 = torch.zeros((ctas, 8), dtype=torch.int64, device="cuda")
        o2 = run(layer, hh, to_dev_x(a2.x_bits), mm, stamps=st2, **kw)
        rows = np.arange(0, mm, 16)
        assert oracle.check(layer, out_f64(o2)[rows], oracle.reference(layer, a2.x_bits[rows], WW),
                            [])["ok"]
        t2 = st2.cpu().numpy()
        assert (t2[:, [0, 1, 4, 5, 6, 7]] > 0).all(), (layer, mm, desc)
        # in order where one thread writes them (thread 0: entry, combine, exit);
        # %globaltimer readings of different warps need not be ordered
        assert (np.diff(t2[:, [0, 6, 7]], axis=1) >= 0).all(), (layer, mm, desc)
        # first stage / last MMA: stamped by the CTAs that issue MMAs (in a CTA
        # pair, the even one)
        issuers = t2[:, 2] > 0
        assert issuers.sum() * (2 if desc.startswith("tc_pair") else 1) == ctas, (layer, mm, desc)
        assert (t2[issuers][:, 3] > 0).all(), (layer, mm, desc)
    x33 = torch.zeros((33, 8192), dtype=torch.bfloat16, device="cuda")
    o33 = torch.zeros((33, 4096), dtype=torch.bfloat16, device="cuda")
    for mm, kw in ((33, dict(kernel=B.PROJ_KERNEL_ROWS)),             # more than 32 tokens
                   (8, dict(kernel=B.PROJ_KERNEL_ROWS, grid=40)),     # 103 rows per CTA
                   (8, dict(kernel=B.PROJ_KERNEL_ROWS, groups=3)),    # not a power of two
                   (8, dict(kernel=B.PROJ_KERNEL_ROWS, variant=B.PROJ_VARIANT_EXPWIN12))):
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x33, mm, o33, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED, (mm, kw)
    hr, _, _ = prepared("router", 0)
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(hr, x33, 8, torch.zeros((8, 256), dtype=torch.float32, device="cuda"),
                      kernel=B.PROJ_KERNEL_ROWS)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("m", [3, 5, 7, 8, 9, 15, 16])
def test_router_gemv(dev, m):
    """The router's few-token FP32-FMA GEMV (whole rows per CTA, weights in
    registers, x in passes of eight tokens): the dispatch form at 3 <= m <= 8
    (forced to 16), at several CTA counts; meets the router's 1e-4 contract
    (probe rows exactly) and is bitwise reproducible."""
    for seed in (0, 1):
        h, W, _ = prepared("router", seed)
        desc = B.proj_describe(h, m)
        assert desc.startswith("router_gemv_f32w") == (m <= 8), desc
        assert desc.startswith("router_gemv_splitk") == (9 <= m <= 24), desc
        # fp32 weights as they are: the dense variant is the automatic one
        assert B.proj_describe_ex(h, m, variant=B.PROJ_VARIANT_DENSE) == desc
        for kw in (dict(), dict(kernel=B.PROJ_KERNEL_GEMV_REG, grid=128),
                   dict(kernel=B.PROJ_KERNEL_GEMV_REG, grid=150)):
            a = check_case("router", seed, seed == 1, m, h=h, W=W, **kw)
            b = check_case("router", seed, seed == 1, m, h=h, W=W, **kw)
            assert np.array_equal(a, b), (m, seed, kw)
        assert B.proj_device_status(h) == 0
    h, _, _ = prepared("router", 0)
    x = torch.zeros((32, 8192), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((32, 256), dtype=torch.float32, device="cuda")
    for mm, kw in ((17, dict(kernel=B.PROJ_KERNEL_GEMV_REG)),
                   (8, dict(kernel=B.PROJ_KERNEL_GEMV_REG, grid=64))):  # 32 chunks per CTA
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x, mm, out, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("m", [1, 2, 3, 8, 9, 16, 17, 31, 32])
def test_router_gemv_splitk(dev, m):
    """The router GEMV with K split across a cluster (one 1024-column chunk
    per CTA, eight rows per cluster, partials summed in rank order through
    distributed shared memory; the dispatch form at 9 <= m <= 24): the 1e-4
    contract, probe rows exactly, and bitwise reproducible; refused for the
    bf16 layers and above 32 tokens."""
    for seed in (0, 1):
        h, W, _ = prepared("router", seed)
        assert B.proj_describe(h, m).startswith("router_gemv_splitk") == (9 <= m <= 24)
        kw = dict(kernel=B.PROJ_KERNEL_GEMV_SPLITK)
        a = check_case("router", seed, seed == 1, m, h=h, W=W, **kw)
        b = check_case("router", seed, seed == 1, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (m, seed)
        assert B.proj_device_status(h) == 0
    h, _, _ = prepared("router", 0)
    x = torch.zeros((33, 8192), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((33, 256), dtype=torch.float32, device="cuda")
    for mm, kw in ((33, dict(kernel=B.PROJ_KERNEL_GEMV_SPLITK)),
                   (8, dict(kernel=B.PROJ_KERNEL_GEMV_SPLITK, variant=B.PROJ_VARIANT_PLANES3))):
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x, mm, out, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED
    hq, _, _ = prepared("o", 0)
    xq = torch.zeros((8, 1024), dtype=torch.bfloat16, device="cuda")
    oq = torch.zeros((8, 8192), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(hq, xq, 8, oq, kernel=B.PROJ_KERNEL_GEMV_SPLITK)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("m", [1, 3, 16, 130, 256])
def test_router_planes_variant(dev, m):
    """The router's opt-in tensor-core form -- its fp32 weights as three exact
    bf16 planes -- meets the router's 1e-4 contract (probe rows exactly) at
    several cluster shapes, reproducibly."""
    h, W, _ = prepared("router", 1)
    for kw in (dict(), dict(grid=4), dict(grid=2, groups=4), dict(grid=16)):
        kw = dict(kw, variant=B.PROJ_VARIANT_PLANES3)
        if kw.get("grid") or kw.get("groups"):
            kw["kernel"] = B.PROJ_KERNEL_CLUSTER
        a = check_case("router", 1, True, m, h=h, W=W, **kw)
        b = check_case("router", 1, True, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (m, kw)
    assert B.proj_device_status(h) == 0


def test_cluster_kernel_rejections(dev):
    h, _, _ = prepared("router", 0)
    x = torch.zeros((64, 8192), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((64, 256), dtype=torch.float32, device="cuda")
    for kw in (dict(kernel=B.PROJ_KERNEL_TILE),
               dict(kernel=B.PROJ_KERNEL_TILE, variant=B.PROJ_VARIANT_PLANES3),
               dict(kernel=B.PROJ_KERNEL_GEMV, variant=B.PROJ_VARIANT_PLANES3),
               dict(kernel=B.PROJ_KERNEL_CLUSTER, tile_n=256),
               dict(variant=B.PROJ_VARIANT_EXPWIN12)):
        with pytest.raises(B.ProjError) as e:
            B.proj_run_ex(h, x, 2 if kw.get("kernel") == B.PROJ_KERNEL_GEMV else 64, out, **kw)
        assert e.value.status == B.PROJ_EUNSUPPORTED, kw
    h, _, _ = prepared("o", 0)
    x = torch.zeros((64, 1024), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((64, 8192), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(h, x, 64, out, kernel=B.PROJ_KERNEL_CLUSTER, grid=17)
    assert e.value.status == B.PROJ_EINVAL
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(h, x, 64, out, variant=B.PROJ_VARIANT_PLANES3)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("layer", [s.name for s in wl.LAYERS])
@pytest.mark.parametrize("m", [1, 2])
def test_gemv_partitions_and_determinism(dev, layer, m):
    """The streaming GEMV over several partitions (rows shared by neighbouring
    CTAs at every boundary) meets the contract and is reproducible."""
    h, W, _ = prepared(layer, 1)
    sms = B.proj_num_sms()
    assert "gemv" in B.proj_describe(h, m)
    for grid in (1, 3, 37, 100, sms - 1, sms):
        kw = dict(grid=grid, kernel=B.PROJ_KERNEL_GEMV)
        a = check_case(layer, 1, True, m, h=h, W=W, **kw)
        b = check_case(layer, 1, True, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (layer, m, grid)
    assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer", [s.name for s in wl.LAYERS])
@pytest.mark.parametrize("m", [1, 2])
def test_register_gemv_partitions_and_determinism(dev, layer, m):
    """The register-streaming GEMV (the dispatch table's m <= 2 form for the
    shorter weight streams) over
    several partitions meets the contract and is reproducible."""
    h, W, _ = prepared(layer, 1)
    sms = B.proj_num_sms()
    for grid in (16, 37, 100, sms - 1, sms):
        kw = dict(grid=grid, kernel=B.PROJ_KERNEL_GEMV_REG)
        a = check_case(layer, 1, True, m, h=h, W=W, **kw)
        b = check_case(layer, 1, True, m, h=h, W=W, **kw)
        assert np.array_equal(a, b), (layer, m, grid)
    assert B.proj_device_status(h) == 0


def test_owner_mode_rejected_for_wide_token_tiles(dev):
    h, W, _ = prepared("pooler", 0)
    x = torch.zeros((64, 8192), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((64, 4096), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(h, x, 64, out, reduce=B.PROJ_REDUCE_OWNER)
    assert e.value.status == B.PROJ_EUNSUPPORTED
    with pytest.raises(B.ProjError) as e:
        B.proj_run_ex(h, x, 3, out, kernel=B.PROJ_KERNEL_GEMV)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("layer,m", [("qkv_gate", 16), ("router", 1), ("pooler", 256),
                                     ("unpooler", 8), ("router", 130)])
def test_graph_replay_with_fresh_inputs(dev, layer, m):
    """Split-K counters must return to zero: replays on new x stay correct
    (muse_bf16_proj notebook, n. 19 "Split-K and the cost of combining work")."""
    spec = wl.LAYER_BY_NAME[layer]
    h, W, _ = prepared(layer, 1)
    n_out = B.proj_out_features(h, m)
    dt = torch.float32 if spec.out_dtype == "fp32" else torch.bfloat16
    xs = torch.zeros((m, spec.K), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((m, n_out), dtype=dt, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        B.proj_run(h, xs, m, out, s)  # warm-up (tensor map cached for this buffer)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.proj_run(h, xs, m, out, torch.cuda.current_stream())
    for rep in range(4):
        act = wl.make_activations(layer, m, 100 + rep, outliers=bool(rep & 1))
        xs.copy_(to_dev_x(act.x_bits))
        g.replay()
        torch.cuda.synchronize()
        o = out_f64(out)
        rows = np.arange(m) if m <= FULL_ORACLE_MAX_M else np.unique(
            np.concatenate([np.arange(0, m, max(1, m // 16)), act.probe_rows]))
        ref = reference_rows(layer, act, W, rows)
        probe_local = [int(np.flatnonzero(rows == p)[0]) for p in act.probe_rows]
        res = oracle.check(layer, o[rows], ref, probe_local)
        assert res["ok"], (layer, m, rep, res)
    assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer", ["qkv_gate", "o", "pooler", "unpooler", "router"])
def test_unpack_is_lossless(dev, layer):
    h, W, Wd = prepared(layer, 0)
    back = torch.empty_like(Wd)
    B.proj_unpack_weights(h, B.PROJ_VARIANT_DENSE, back)
    torch.cuda.synchronize()
    assert torch.equal(back.view(torch.int16) if back.dtype == torch.bfloat16 else back,
                       Wd.view(torch.int16) if Wd.dtype == torch.bfloat16 else Wd)
    if layer == "router":
        # the three bf16 planes sum back to the fp32 weights bit for bit
        B.proj_unpack_weights(h, B.PROJ_VARIANT_PLANES3, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int32), Wd.view(torch.int32))
        with pytest.raises(B.ProjError):
            B.proj_unpack_weights(h, B.PROJ_UNPACK_FRAG16, back)
    else:
        # the few-token GEMV's copy in warp-MMA fragment order
        back.zero_()
        B.proj_unpack_weights(h, B.PROJ_UNPACK_FRAG16, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        # the row-run GEMV's copy (each CTA's rows step-major)
        back.zero_()
        B.proj_unpack_weights(h, B.PROJ_UNPACK_RUNS, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        if layer == "unpooler":
            part = torch.zeros((1024, Wd.shape[1]), dtype=Wd.dtype, device="cuda")
            B.proj_unpack_weights(h, B.PROJ_UNPACK_RUNS_SLICE, part)
            torch.cuda.synchronize()
            assert torch.equal(part.view(torch.int16), Wd[:1024].view(torch.int16))
        else:
            with pytest.raises(B.ProjError):
                B.proj_unpack_weights(h, B.PROJ_UNPACK_RUNS_SLICE, back)


@pytest.mark.parametrize("layer", ["qkv_gate", "o", "pooler", "unpooler"])
def test_expwin12_lossless_and_bit_identical(dev, layer):
    """12-bit exponent-window weights (muse_bf16_proj project report, Round 5):
    window and escapes as the oracle's codec, lossless decode, and outputs
    bit-identical to the uncompressed kernel at the same partition -- also at
    the wide token counts, where the tile kernel decodes records into
    swizzled bf16 tiles for 64- and 128-token tensor-core tiles (project
    report, Round 6: decode to shared memory, then the same MMAs)."""
    for seed in (0, 1):
        h, W, Wd = prepared(layer, seed, B.PROJ_ENCODE_EXPWIN12)
        info = B.proj_info(h)
        assert info["expwin12"] == 1 and info["expwin12_declined"] == 0
        e0 = oracle.expwin12_window(W)
        _, _, esc, _ = oracle.expwin12_encode(W, e0)
        assert info["expwin12_e0"] == e0
        assert info["expwin12_escapes"] == esc.size
        back = torch.empty_like(Wd)
        B.proj_unpack_weights(h, B.PROJ_VARIANT_EXPWIN12, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        for m in (1, 8, 16, 32, 64, 128, 130, 256):
            act = wl.make_activations(layer, m, seed + 5, outliers=True)
            x = to_dev_x(act.x_bits)
            combos = ((0, 0), (37, B.PROJ_REDUCE_OWNER), (0, B.PROJ_REDUCE_DISTRIBUTED))
            if m > 32:  # 64- and 128-token tiles: the distributed combine only
                combos = ((0, 0), (101, B.PROJ_REDUCE_DISTRIBUTED))
            tn = 0 if m <= 32 else (64 if m <= 64 else 128)  # the same token tiles
            for grid, reduce in combos:
                a = run(layer, h, x, m, variant=B.PROJ_VARIANT_DENSE, grid=grid, reduce=reduce,
                        kernel=B.PROJ_KERNEL_TILE, tile_n=tn)
                b = run(layer, h, x, m, variant=B.PROJ_VARIANT_EXPWIN12, grid=grid,
                        reduce=reduce, kernel=B.PROJ_KERNEL_TILE, tile_n=tn)
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
                    (layer, seed, m, grid, reduce)
            check_case(layer, seed, True, m, h=h, W=W, variant=B.PROJ_VARIANT_EXPWIN12)
        # one-hot rows on escaped columns reproduce the column exactly
        K = W.shape[1]
        n_out = B.proj_out_features(h, 8)
        cols = np.unique(esc[(esc // K) < n_out] % K)[:8]
        x = np.zeros((len(cols), K), np.uint16)
        x[np.arange(len(cols)), cols] = 0x3F80  # 1.0
        o = out_f64(run(layer, h, to_dev_x(x), len(cols), variant=B.PROJ_VARIANT_EXPWIN12))
        for i, c in enumerate(cols):
            assert np.array_equal(o[i], oracle.bf16_bits_to_f64(W[:o.shape[1], c]))
        assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer", ["qkv_gate", "o", "pooler", "unpooler"])
def test_expwin12_register_gemv(dev, layer):
    """The 12-bit row-chunk records on the register GEMV (m <= 2): the copy
    decodes to W bit for bit, and the outputs are bit-identical to the dense
    register GEMV at the same partition (same products, same order)."""
    for seed in (0, 1):
        h, W, Wd = prepared(layer, seed, B.PROJ_ENCODE_EXPWIN12)
        back = torch.zeros_like(Wd)
        B.proj_unpack_weights(h, B.PROJ_UNPACK_RC12, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        for m in (1, 2):
            act = wl.make_activations(layer, m, seed + 3, outliers=True)
            x = to_dev_x(act.x_bits)
            for grid in (0, 37, 151):
                a = run(layer, h, x, m, variant=B.PROJ_VARIANT_DENSE,
                        kernel=B.PROJ_KERNEL_GEMV_REG, grid=grid)
                b = run(layer, h, x, m, variant=B.PROJ_VARIANT_EXPWIN12, grid=grid)
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (layer, seed, m, grid)
            check_case(layer, seed, True, m, h=h, W=W, variant=B.PROJ_VARIANT_EXPWIN12)
            # the dispatch table keeps the dense register form at m <= 2
            assert B.proj_describe(h, m).startswith("gemv_reg_bf16w")
        assert B.proj_device_status(h) == 0


@pytest.mark.parametrize("layer,m", [("qkv_gate", 3), ("qkv_gate", 8), ("o", 5), ("o", 16),
                                     ("o", 32), ("pooler", 8), ("unpooler", 8),
                                     ("unpooler", 16)])
def test_expwin12_mma_gemv(dev, layer, m):
    """The warp-MMA GEMV on the 12-bit recode of its fragment-order copy:
    outputs bit-identical to the dense warp-MMA GEMV at the same partition
    (the same MMAs on the same decoded fragments), and the oracle's contract."""
    for seed in (0, 1):
        h, W, Wd = prepared(layer, seed, B.PROJ_ENCODE_EXPWIN12)
        back = torch.zeros_like(Wd)
        B.proj_unpack_weights(h, B.PROJ_UNPACK_FRAG12, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        desc = B.proj_describe_ex(h, m, variant=B.PROJ_VARIANT_EXPWIN12)
        assert desc.startswith("gemv_mma16x8_expwin12rc"), desc
        act = wl.make_activations(layer, m, seed + 7, outliers=True)
        x = to_dev_x(act.x_bits)
        a = run(layer, h, x, m, variant=B.PROJ_VARIANT_DENSE, kernel=B.PROJ_KERNEL_MMA)
        b = run(layer, h, x, m, variant=B.PROJ_VARIANT_EXPWIN12)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (layer, seed, m)
        check_case(layer, seed, True, m, h=h, W=W, variant=B.PROJ_VARIANT_EXPWIN12)
        assert B.proj_device_status(h) == 0


def _fragment_positions():
    """(row, column) within a 16 x 16 tile of lane l's eight A-fragment
    elements of mma.sync m16n8k16 (row-major A), in register order."""
    l = np.arange(32)
    g, c = l // 4, 2 * (l % 4)
    rows = np.stack([g, g, g + 8, g + 8, g, g, g + 8, g + 8], 1)
    cols = np.stack([c, c + 1, c, c + 1, c + 8, c + 9, c + 8, c + 9], 1)
    return rows, cols


def test_expwin12_mma_gemv_planted_escapes(dev):
    """o's weights with up to 7 escapes in every 12-bit fragment record (four
    16 x 16 tiles of a row block) at every tile, lane and register position:
    the 12-bit warp-MMA GEMV equals the dense one bit for bit at 3..32 tokens;
    8 escapes in one record make prepare decline that copy."""
    spec = wl.LAYER_BY_NAME["o"]
    rows, cols = _fragment_positions()
    for cap in (7, 8):
        W = wl.make_weights(spec, 2).copy()
        e0 = oracle.expwin12_window(W)
        h7 = (W >> 8) & 0x7F
        nat = (h7 < e0) | (h7 > e0 + 7)
        W[nat] = 0x3C00 | (W[nat] & 0x8000)
        rng = np.random.default_rng(21 + cap)
        KT = spec.K // 16
        vals = np.array([0x4080, 0xC0A0, 0x0000, 0x8000, 0x4200, 0xC110], np.uint16)
        n_rec = spec.N * spec.K // 1024
        for r in range(n_rec):
            n = cap if r == 0 else int(rng.integers(0, 8))
            pos = rng.choice(1024, size=n, replace=False)  # 256 tile + 8 lane + element
            t, ln, b = pos >> 8, (pos >> 3) & 31, pos & 7
            rb, kb = (4 * r) // KT, (4 * r) % KT + t
            W[rb * 16 + rows[ln, b], kb * 16 + cols[ln, b]] = vals[rng.integers(0, len(vals), n)]
        Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
        h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, B.PROJ_BF16,
                              B.PROJ_ENCODE_EXPWIN12, 64)
        try:
            for m in (3, 8, 16, 32):
                x = to_dev_x(wl.make_activations(spec, m, 5, outliers=True).x_bits)
                try:
                    desc = B.proj_describe_ex(h, m, variant=B.PROJ_VARIANT_EXPWIN12)
                except B.ProjError:
                    desc = ""
                assert desc.startswith("gemv_mma16x8_expwin12rc") == (cap == 7), (cap, m, desc)
                if cap == 7 and m == 3:
                    back = torch.zeros_like(Wd)
                    B.proj_unpack_weights(h, B.PROJ_UNPACK_FRAG12, back)
                    torch.cuda.synchronize()
                    assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
                if cap == 7:
                    a = run("o", h, x, m, variant=B.PROJ_VARIANT_DENSE, kernel=B.PROJ_KERNEL_MMA)
                    b = run("o", h, x, m, variant=B.PROJ_VARIANT_EXPWIN12)
                    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), m
            assert B.proj_device_status(h) == 0
        finally:
            B.proj_destroy(h)


def _planted_escape_weights(n_per_chunk, seed=0):
    """o's weights with escapes planted at chosen columns of each 1024-column
    chunk (row): large values above the window, signed zeros below it, at
    even and odd columns of every lane and group position."""
    spec = wl.LAYER_BY_NAME["o"]
    W = wl.make_weights(spec, seed).copy()
    # the matrix's own escapes move into the window (2^-7, same sign), so
    # every chunk holds exactly the planted ones
    e0 = oracle.expwin12_window(W)
    h7 = (W >> 8) & 0x7F
    nat = (h7 < e0) | (h7 > e0 + 7)
    W[nat] = 0x3C00 | (W[nat] & 0x8000)
    rng = np.random.default_rng(seed + 11)
    fixed = np.array([0, 1, 9, 255, 263, 767, 1023, 512])
    vals = np.array([0x4080, 0xC0A0, 0x0000, 0x8000, 0x4200, 0xC110, 0x0000, 0x4080], np.uint16)
    for n in range(spec.N):
        if n == 0:
            cols = fixed[:n_per_chunk]
        else:
            cols = rng.choice(1024, size=int(rng.integers(0, n_per_chunk + 1)), replace=False)
        W[n, cols] = vals[rng.integers(0, len(vals), size=len(cols))]
    return spec, W


def test_expwin12_register_gemv_planted_escapes(dev):
    """Chunks with up to the block's 7 escapes decode exactly and give the
    dense register GEMV's outputs bit for bit; one chunk with 8 escapes makes
    prepare decline the row-chunk copy (the dense forms serve instead)."""
    spec, W = _planted_escape_weights(7)
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, B.PROJ_BF16, B.PROJ_ENCODE_EXPWIN12, 64)
    try:
        back = torch.zeros_like(Wd)
        B.proj_unpack_weights(h, B.PROJ_UNPACK_RC12, back)
        torch.cuda.synchronize()
        assert torch.equal(back.view(torch.int16), Wd.view(torch.int16))
        for m in (1, 2):
            act = wl.make_activations(spec, m, 4, outliers=False)
            x = to_dev_x(act.x_bits)
            a = run("o", h, x, m, variant=B.PROJ_VARIANT_DENSE, kernel=B.PROJ_KERNEL_GEMV_REG)
            b = run("o", h, x, m, variant=B.PROJ_VARIANT_EXPWIN12)
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), m
            ref = oracle.reference("o", act.x_bits, W)
            res = oracle.check("o", out_f64(b), ref, [])
            assert res["ok"], res
        # one-hot rows on the planted columns of row 0 reproduce W's column
        for c in (0, 1, 9, 255, 263, 767, 1023):
            x = np.zeros((1, spec.K), np.uint16)
            x[0, c] = 0x3F80
            o = out_f64(run("o", h, to_dev_x(x), 1, variant=B.PROJ_VARIANT_EXPWIN12))
            assert np.array_equal(o[0], oracle.bf16_bits_to_f64(W[:, c])), c
        assert B.proj_device_status(h) == 0
    finally:
        B.proj_destroy(h)
    spec, W = _planted_escape_weights(8)
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, B.PROJ_BF16, B.PROJ_ENCODE_EXPWIN12, 64)
    try:
        assert B.proj_info(h)["expwin12_declined"] == 1  # the tile records overflow too
        back = torch.zeros_like(Wd)
        with pytest.raises(B.ProjError) as e:
            B.proj_unpack_weights(h, B.PROJ_UNPACK_RC12, back)
        assert e.value.status == B.PROJ_EUNSUPPORTED
        act = wl.make_activations(spec, 1, 4, outliers=False)
        with pytest.raises(B.ProjError) as e:
            run("o", h, to_dev_x(act.x_bits), 1, variant=B.PROJ_VARIANT_EXPWIN12)
        assert e.value.status == B.PROJ_EUNSUPPORTED
        out = run("o", h, to_dev_x(act.x_bits), 1)
        res = oracle.check("o", out_f64(out), oracle.reference("o", act.x_bits, W), [])
        assert res["ok"], res
    finally:
        B.proj_destroy(h)


@pytest.mark.parametrize("pinned", [True, False])
def test_run_host_matches_device_run(dev, pinned):
    """proj_run_host equals proj_run bit for bit: a page-locked x moves in
    through a copy kernel on its device mapping and the projection kernel
    stores straight into a page-locked output's mapping; pageable buffers go
    through cudaMemcpyAsync (then synchronous).  One shape per kernel family
    (register GEMV, router GEMVs, warp-MMA and row-run GEMVs, cluster, CTA
    pair, FP32-FMA router)."""
    for layer, m in (("o", 1), ("router", 16), ("unpooler", 8), ("pooler", 130),
                     ("qkv_gate", 8), ("router", 5), ("router", 64), ("o", 256),
                     ("unpooler", 256), ("qkv_gate", 32)):
        spec = wl.LAYER_BY_NAME[layer]
        h, W, _ = prepared(layer, 0)
        act = wl.make_activations(layer, m, 3, False)
        dev_out = run(layer, h, to_dev_x(act.x_bits), m)
        x_host = torch.from_numpy(act.x_bits.view(np.int16).copy()).view(torch.bfloat16)
        host_out = torch.full(dev_out.shape, float("nan"), dtype=dev_out.dtype)
        if pinned:
            x_host, host_out = x_host.pin_memory(), host_out.pin_memory()
        s = torch.cuda.current_stream()
        for _ in range(2):  # the second call overwrites the first call's buffers
            B.proj_run_host(h, x_host, m, host_out, s)
        s.synchronize()
        if pinned and layer == "o":
            # one call's host output is the next call's host input (o's 8192
            # outputs feed qkv_gate's K = 8192): the copy in must see it
            hq, Wq, _ = prepared("qkv_gate", 0)
            chained = torch.full((m, 2304), float("nan"), dtype=torch.bfloat16).pin_memory()
            host_out.fill_(float("nan"))  # the chain must see the new output, not a stale one
            B.proj_run_host(h, x_host, m, host_out, s)
            B.proj_run_host(hq, host_out, m, chained, s)
            s.synchronize()
            ref = run("qkv_gate", hq, dev_out, m)
            assert torch.equal(chained.view(torch.int16), ref.cpu().view(torch.int16))
        assert torch.equal(host_out.view(torch.int16) if spec.out_dtype == "bf16" else host_out,
                           dev_out.cpu().view(torch.int16) if spec.out_dtype == "bf16"
                           else dev_out.cpu())


def test_edge_arguments(dev):
    h, W, _ = prepared("o", 0)
    x = torch.zeros((4, 1024), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((4, 8192), dtype=torch.bfloat16, device="cuda")
    B.proj_run(h, x, 0, out)  # m = 0: no launch, no error
    with pytest.raises(B.ProjError) as e:
        B.proj_run(h, x, 1025, out)
    assert e.value.status == B.PROJ_EUNSUPPORTED
    with pytest.raises(B.ProjError) as e:
        B.proj_run(h, x.data_ptr() + 2, 1, out)
    assert e.value.status == B.PROJ_EALIGN
    assert B.proj_out_features(prepared("unpooler", 0)[0], 8) == 1024
    assert B.proj_out_features(prepared("unpooler", 0)[0], 9) == 8192
    assert "gemv" in B.proj_describe(h, 1)
    assert "gemv_mma" in B.proj_describe(h, 3)
    assert "gemv_mma" in B.proj_describe(h, 9)
    assert "BN=32" in B.proj_describe(h, 17)
    with pytest.raises(B.ProjError) as e:  # a run longer than the register form keeps
        B.proj_run_ex(h, x, 1, out, grid=1, kernel=B.PROJ_KERNEL_GEMV_REG)
    assert e.value.status == B.PROJ_EUNSUPPORTED


@pytest.mark.parametrize("mode", [0, 1, 0 | 4, 1 | 4])
def test_read_floor_checksums(dev, mode):
    nbytes = 48 * 1024 * 1024 + 4096
    g = torch.Generator().manual_seed(5)
    buf = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, generator=g)
    grid = 37
    sink = torch.zeros(grid + 1, dtype=torch.int32, device="cuda")
    B.proj_read_floor(buf.cuda(), nbytes, sink, grid, mode)
    torch.cuda.synchronize()
    words = buf.numpy().view(np.uint32)
    n16 = nbytes // 16
    for c in range(grid):
        b, e = c * n16 // grid, (c + 1) * n16 // grid
        seg = words[4 * b:4 * e]
        if mode & 1 == 0:
            expect = np.bitwise_xor.reduce(seg) if seg.size else 0
        else:
            expect = np.bitwise_xor.reduce(seg[::4096]) if seg.size else 0
        assert int(sink[c].item()) & 0xFFFFFFFF == int(expect), c
    assert int(sink[grid].item()) == 0


@pytest.mark.parametrize("m", [1, 2, 3, 16, 128, 256])
def test_dependent_chain_back_to_back(dev, m):
    """o -> pooler -> unpooler -> router with each layer's input the previous
    layer's output, launched back to back on one stream with no host sync
    (the kernels let their successor start early and wait for their
    predecessor before reading x): every stage meets the contract against the
    oracle applied to the GPU's own input for that stage."""
    chain = ["o", "pooler", "unpooler"] + (["router"] if m > 8 else [])
    hs = {name: prepared(name, 2) for name in chain}
    x0 = to_dev_x(wl.make_activations("o", m, 9).x_bits)
    rows = np.unique(np.linspace(0, m - 1, min(m, 12)).astype(np.int64))
    for rep in range(3):
        outs = []
        for name in chain:
            spec = wl.LAYER_BY_NAME[name]
            dt = torch.float32 if spec.out_dtype == "fp32" else torch.bfloat16
            outs.append(torch.full((m, B.proj_out_features(hs[name][0], m)), float("nan"),
                                   dtype=dt, device="cuda"))
        torch.cuda.synchronize()
        x = x0
        for name, o in zip(chain, outs):
            B.proj_run(hs[name][0], x, m, o)
            x = o
        torch.cuda.synchronize()
        xin = x0
        for name, o in zip(chain, outs):
            h, W, _ = hs[name]
            x_bits = xin.view(torch.int16).cpu().numpy().view(np.uint16)
            ref = oracle.reference(name, x_bits[rows], W)
            res = oracle.check(name, out_f64(o)[rows], ref)
            assert res["ok"], (m, rep, name, res)
            assert B.proj_device_status(h) == 0
            xin = o


def test_fma_peak_probe(dev):
    """The FP32 FMA probe runs, never writes its sink, reports its FLOPs, and
    measures a rate within the part's range: above half the derived peak
    (SMs x 128 FMA lanes x 2 FLOP x the maximum SM clock) and at most a
    little above it."""
    sms = B.proj_num_sms()
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    for _ in range(2):
        flops = B.proj_fma_peak(sink, 2048, 0, s)
    assert flops == 8 * sms * 256 * 8 * 2 * 2 * 2048
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    B.proj_fma_peak(sink, 2048, 0, s)
    e1.record(s)
    e1.synchronize()
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    derived = sms * 128 * 2 * 2.07e9 / 1e12
    assert 0.5 * derived < tflops < 1.1 * derived, (tflops, derived)
    assert int(sink.abs().sum().item()) == 0
    assert B.proj_fma_peak(sink, 16, 3, s) == 3 * 256 * 8 * 2 * 2 * 16
