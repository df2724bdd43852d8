"""CUDA router vs the CPU oracle, element by element, through the C ABI.

Sizes: the router benchmarks' workloads at full size (the oracle handles
8192 x 2304 in a few seconds), the decode sweep, and edge shapes (odd E,
ragged T, K = 1 and K = E, unaligned buffers, heavy ties, every compiled
lanes-per-row width).
"""
import numpy as np
import pytest

import oracle.router_oracle as O
from compare import assert_close, compare_map, record_near_ties
from score_top_expert_gb300.workloads import WORKLOADS, make_case, make_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


DEV = "cuda:0"
PATHS = ["auto", "segment", "staged", "register"]


@pytest.fixture(params=PATHS)
def path(R, request):
    prev = R.force_path(request.param)
    yield request.param
    R.force_path(prev)
    assert R.device_status() == 0
TD = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV).to(TD[dtype])


def np64(t):
    return t.detach().to(torch.float64).cpu().numpy() if t.dtype != torch.bool \
        else t.cpu().numpy()


_REF_CACHE = {}


def oracle_topk(case, K, sf, ng, gk, c, bias, key=None):
    if key is not None and key in _REF_CACHE:
        return _REF_CACHE[key]
    ref = O.topk_fwd(case.logits, K, sf, ng, gk, c, bias)
    ref["grad"] = O.topk_bwd(case.grad_probs, ref["routing_map"], ref["scores"], sf, c)
    if key is not None:
        _REF_CACHE.clear()
        _REF_CACHE[key] = ref
    return ref


def run_and_check_topk(R, case, K, sf, c=1.0, ng=0, gk=0, bias=None, check_bwd=True,
                       tensors=None, ref_key=None):
    """Run fwd (+bwd) on the GPU and compare with the oracle; returns the map report."""
    dt = case.dtype
    x = to_dev(case.logits, dt) if tensors is None else tensors["x"]
    b = None if bias is None else to_dev(bias)
    kw = {} if tensors is None else tensors.get("out", {})
    probs, rmap, scores = R.router_topk_fwd(x, K, sf, ng, gk, c, b, **kw)
    ref = oracle_topk(case, K, sf, ng, gk, c, bias, ref_key)
    rep = compare_map(rmap.cpu().numpy(), ref["routing_map"], ref["near_tie"])
    rep.check(f"topk map {sf} {dt}")
    ok = rep.ok_rows
    assert_close(np64(probs), ref["probs"], dt, ok, "probs")
    assert_close(np64(scores), ref["scores"], "f32", None, "scores")
    assert (rmap.cpu().numpy().sum(axis=1) == K).all()
    if check_bwd:
        g = to_dev(case.grad_probs, dt)
        gx = R.router_topk_bwd(g, rmap, scores, K, sf, c)
        assert_close(np64(gx), ref["grad"], dt, ok, "grad_logits")
    return rep


def run_and_check_aux(R, case, K, sf, ref_key=None):
    dt = case.dtype
    x = to_dev(case.logits, dt)
    q, rmap, inter = R.router_aux_scores_fwd(x, K, sf)
    if ref_key is not None and ref_key in _REF_CACHE:
        ref = _REF_CACHE[ref_key]
    else:
        ref = O.aux_scores_fwd(case.logits, K, sf)
        if ref_key is not None:
            _REF_CACHE.clear()
            _REF_CACHE[ref_key] = ref
    rep = compare_map(rmap.cpu().numpy(), ref["routing_map"], ref["near_tie"])
    rep.check(f"aux map {sf}")
    assert_close(np64(q), ref["scores"], "f32", None, "aux scores")
    assert_close(np64(inter), ref["saved"], "f32", None, "aux intermediate")
    gs = to_dev(case.grad_scores)
    gx = R.router_aux_scores_bwd(gs, inter, K, sf, TD[dt])
    gref = O.aux_scores_bwd(case.grad_scores, ref["saved"], sf)
    assert_close(np64(gx), gref, dt, None, "aux grad_logits")
    return rep


# ---------------------------------------------------------------------------
# the benchmark workloads, full size
# ---------------------------------------------------------------------------
TOPK_CASES = [
    ("t1024_e64_k4", "softmax", "f32"), ("t8192_e256_k8", "softmax_post", "bf16"),
    ("t8192_e512_k22", "softmax_post", "f32"), ("t8192_e2304_k36", "softmax_post", "f32"),
    ("t8192_e256_k4", "softmax", "f32"), ("t8192_e256_k4", "sigmoid", "f32"),
    ("t8192_e256_k8", "softmax", "f32"), ("t8192_e256_k8", "sigmoid", "f32"),
    ("t8192_e256_k4", "softmax", "bf16"), ("t8192_e256_k8", "sigmoid", "bf16"),
    ("t8192_e256_k4", "sigmoid", "bf16"), ("t8192_e256_k8", "softmax", "bf16"),
    ("t8192_e512_k22", "softmax", "f32"), ("t8192_e512_k22", "sigmoid", "f32"),
    ("t8192_e2304_k36", "softmax", "f32"), ("t8192_e2304_k36", "sigmoid", "f32"),
    ("t16384_e256_k8_grouped", "sigmoid", "bf16"),
]


@pytest.mark.parametrize("name,sf,dt", TOPK_CASES, ids=[f"{n}-{s}-{d}" for n, s, d in TOPK_CASES])
def test_topk_workload(R, path, name, sf, dt):
    case, args = make_workload(name, dtype=dt)
    bias = case.expert_bias
    rep = run_and_check_topk(R, case, args["K"], sf, args["scaling_factor"],
                             args["num_groups"], args["group_topk"], bias,
                             ref_key=("topk", name, sf, dt))
    record_near_ties(f"topk {name} {sf} {dt}", rep)


AUX_CASES = [("t8192_e512_k22", "softmax"), ("t8192_e512_k22", "sigmoid"),
             ("t8192_e2304_k36", "softmax"), ("t8192_e2304_k36", "sigmoid")]


@pytest.mark.parametrize("name,sf", AUX_CASES, ids=[f"{n}-{s}" for n, s in AUX_CASES])
def test_aux_workload(R, path, name, sf):
    case, args = make_workload(name)
    rep = run_and_check_aux(R, case, args["K"], sf, ref_key=("aux", name, sf))
    record_near_ties(f"aux {name} {sf} f32", rep)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 3, 129, 1100])
@pytest.mark.parametrize("E", [8, 16, 64, 120, 128, 136, 200, 256, 264, 384, 504, 512])
def test_register_shapes(R, E, T, dt):
    # the register-resident forward on every row shape it serves (E <= 512,
    # E % 8 == 0): padded and full rows, both chunk counts, one to many rows
    # per warp, K from 1 to 36 and K = E
    prev = R.force_path("register")
    try:
        for K in sorted({1, min(E, 4), min(E, 22), min(E, 36), E if E <= 36 else 1}):
            case = make_case(T, E, K, dtype=dt, sigma=1.5, seed=E * 13 + K + T)
            for sf in ("softmax", "sigmoid", "softmax_post"):
                run_and_check_topk(R, case, K, sf, c=2.5, check_bwd=False)
                if sf != "softmax_post":
                    run_and_check_aux(R, case, K, sf)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E", [8, 64, 256, 512, 520, 1000, 1024, 2048, 2304])
def test_staged_shapes(R, E, dt):
    prev = R.force_path("staged")
    try:
        for K in sorted({1, min(E, 4), min(E, 22), min(E, 36)}):
            case = make_case(129, E, K, dtype=dt, sigma=1.5, seed=E + K)
            for sf in ("softmax", "sigmoid", "softmax_post"):
                run_and_check_topk(R, case, K, sf, c=2.5)
                if dt == "f32" and sf != "softmax_post":
                    run_and_check_aux(R, case, K, sf)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


def test_duplicate_rows_select_lower_indices(R, path):
    case, args = make_workload("t8192_e2304_k36")
    assert len(case.dup_rows) >= 82
    x = to_dev(case.logits)
    _, rmap, _ = R.router_topk_fwd(x, 36, "softmax")
    got = rmap.cpu().numpy()[case.dup_rows]
    for r, row in zip(case.dup_rows, got):
        order = np.lexsort((np.arange(2304), -case.logits[r].astype(np.float64)))
        want = np.zeros(2304, bool)
        want[order[:36]] = True
        assert np.array_equal(row, want), r


# ---------------------------------------------------------------------------
# decode sweep: 1, 2, 4 rows, E = 512, K in 1..10
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 4])
def test_decode_sweep(R, T, dt):
    for K in (1, 2, 4, 6, 8, 10):
        case = make_case(T, 512, K, dtype=dt, seed=4242 + T)
        run_and_check_topk(R, case, K, "softmax")


# ---------------------------------------------------------------------------
# edge shapes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("E", [1, 2, 3, 5, 7, 13, 64, 100, 129, 255, 513, 1000, 2303, 2304])
def test_odd_and_ragged_shapes(R, E):
    for sf in ("softmax", "sigmoid", "softmax_post"):
        for K in sorted({1, min(E, 3), min(E, 36), min(E, 17)}):
            case = make_case(37, E, K, sigma=1.5, seed=E * 31 + K)
            run_and_check_topk(R, case, K, sf, c=1.7)
            if sf != "softmax_post":
                run_and_check_aux(R, case, K, sf)


@pytest.mark.parametrize("E", [4, 16, 36])
def test_k_equals_e(R, E):
    for sf in ("softmax", "sigmoid"):
        case = make_case(50, E, E, seed=E)
        run_and_check_topk(R, case, E, sf, c=2.0)


@pytest.mark.parametrize("T", [0, 1, 7, 31, 33, 257, 1001])
def test_ragged_token_counts(R, T):
    for E, K in ((64, 4), (256, 8), (512, 22), (2304, 36)):
        case = make_case(T, E, K, seed=T + E)
        if T == 0:
            x = torch.empty(0, E, device=DEV)
            p, m, s = R.router_topk_fwd(x, K)
            assert p.shape == (0, E)
            continue
        run_and_check_topk(R, case, K, "softmax")


@pytest.mark.parametrize("lanes", [8, 16, 32])
def test_every_lane_width(R, lanes):
    prev = R.force_fwd_lanes(lanes)
    try:
        for E, K in ((64, 4), (128, 16), (256, 8), (512, 22), (1000, 30), (2304, 36)):
            for dt in ("f32", "bf16"):
                case = make_case(300, E, K, dtype=dt, seed=E + lanes)
                for sf in ("softmax", "sigmoid", "softmax_post"):
                    run_and_check_topk(R, case, K, sf, c=2.5)
                    run_and_check_topk(R, case, K, sf, c=2.5,
                                       bias=np.linspace(-0.05, 0.05, E).astype(np.float32))
                run_and_check_aux(R, case, K, "sigmoid")
    finally:
        R.force_fwd_lanes(prev)


def test_unaligned_buffers_take_the_elementwise_path(R):
    T, E, K = 129, 512, 22
    case = make_case(T, E, K, seed=99)
    buf = torch.zeros(T * E + 1, device=DEV)
    x = buf[1:].view(T, E)
    x.copy_(to_dev(case.logits))
    assert x.data_ptr() % 16 != 0
    outs = dict(probs=torch.empty(T * E + 3, device=DEV)[3:].view(T, E))
    run_and_check_topk(R, case, K, "softmax", tensors={"x": x, "out": outs})
    run_and_check_topk(R, case, K, "sigmoid", tensors={"x": x, "out": outs})


# ---------------------------------------------------------------------------
# ties
# ---------------------------------------------------------------------------
def tie_rows(E, rng):
    rows = [np.zeros(E), np.full(E, -3.25), rng.integers(-2, 3, E).astype(float),
            np.where(rng.random(E) < 0.5, 0.0, -0.0),
            np.round(rng.normal(0, 1, E), 1), np.repeat(rng.normal(0, 1, E // 4 + 1), 4)[:E]]
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("E", [8, 64, 256, 512, 2304])
def test_tied_logits(R, path, E):
    from score_top_expert_gb300.workloads import round_to_bf16_values
    rng = np.random.default_rng(E)
    x = tie_rows(E, rng)
    for K in sorted({1, min(E, 4), min(E, 22), min(E, 36)}):
        for dt in ("f32", "bf16"):
            case = make_case(x.shape[0], E, K, dtype=dt, seed=1)
            case.logits = x if dt == "f32" else round_to_bf16_values(x)
            for sf in ("softmax", "sigmoid", "softmax_post"):
                run_and_check_topk(R, case, K, sf)
                if dt == "f32" and sf != "softmax_post":
                    run_and_check_aux(R, case, K, sf)


# ---------------------------------------------------------------------------
# bias and groups
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("sf", ["softmax", "sigmoid", "softmax_post"])
def test_bias(R, path, sf):
    for E, K in ((64, 4), (256, 8), (512, 22), (2304, 36)):
        case = make_case(513, E, K, seed=E, with_bias=True, bias_range=0.1)
        run_and_check_topk(R, case, K, sf, c=2.5, bias=case.expert_bias)


GROUPED = [  # (E, num_groups, group_topk, K)
    (256, 8, 4, 8), (256, 8, 1, 8), (256, 8, 8, 8), (256, 4, 2, 12), (256, 16, 4, 8),
    (256, 32, 8, 16), (64, 2, 1, 6), (512, 8, 2, 22 - 22 % 2), (2304, 16, 4, 36),
    (2304, 8, 1, 36), (120, 3, 2, 10), (12, 4, 2, 2), (60, 5, 5, 15), (1000, 10, 3, 30),
    # groups that align with 4-expert chunks (scored in registers on the staged path)
    (512, 16, 4, 8), (1024, 32, 4, 16), (384, 12, 4, 8), (2304, 18, 9, 36), (256, 32, 2, 8),
    # more chunk-aligned groups: sums of 3 and 4 keys, two-lane and quarter-warp groups
    (256, 8, 4, 12), (512, 32, 4, 12), (128, 4, 2, 8), (512, 16, 8, 32), (136, 17, 1, 2),
]


@pytest.mark.parametrize("E,G,gk,K", GROUPED, ids=[f"E{e}-G{g}-gk{k}-K{K}" for e, g, k, K in GROUPED])
def test_grouped(R, path, E, G, gk, K):
    for dt in ("f32", "bf16"):
        case = make_case(300, E, K, dtype=dt, seed=E + G, with_bias=True)
        for sf in ("sigmoid", "softmax", "softmax_post"):
            run_and_check_topk(R, case, K, sf, 2.5, G, gk, case.expert_bias)
            run_and_check_topk(R, case, K, sf, 1.0, G, gk, None)


# ---------------------------------------------------------------------------
# nothing is written outside the outputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("E", [7, 256, 2304])
def test_canaries(R, E):
    T, K = 65, min(E, 8)
    case = make_case(T, E, K, seed=5)
    n = T * E
    pad = 256
    probs = torch.full((n + pad,), 7.5, device=DEV)
    rmap = torch.full((n + pad,), True, device=DEV)
    scores = torch.full((n + pad,), -9.0, device=DEV)
    out = dict(probs=probs[:n].view(T, E), routing_map=rmap[:n].view(T, E),
               scores=scores[:n].view(T, E))
    run_and_check_topk(R, case, K, "sigmoid", tensors={"x": to_dev(case.logits), "out": out},
                       check_bwd=False)
    assert (probs[n:] == 7.5).all() and (rmap[n:]).all() and (scores[n:] == -9.0).all()
    g = to_dev(case.grad_probs)
    gx = torch.full((n + pad,), 3.0, device=DEV)
    R.router_topk_bwd(g, out["routing_map"], out["scores"], K, "sigmoid",
                      grad_logits=gx[:n].view(T, E))
    q = torch.full((n + pad,), 1.25, device=DEV)
    R.router_aux_scores_fwd(to_dev(case.logits), K, "softmax", scores=q[:n].view(T, E))
    torch.cuda.synchronize()
    assert (gx[n:] == 3.0).all() and (q[n:] == 1.25).all()


def test_errors_raise(R):
    x = torch.zeros(4, 16, device=DEV)
    with pytest.raises(R.RouterError):
        R.router_topk_fwd(x, 17)
    with pytest.raises(R.RouterError):
        R.router_topk_fwd(x, 4, "sigmoid", num_groups=3, group_topk=1)


BWD_SHAPES = [(8, 1, 2), (16, 1, 4), (32, 1, 2), (32, 1, 4), (32, 2, 1), (32, 2, 2), (32, 2, 4),
              (32, 4, 1), (32, 4, 2), (32, 3, 6), (32, 6, 3), (32, 9, 2)]


@pytest.mark.parametrize("shape", BWD_SHAPES, ids=["x".join(map(str, s)) for s in BWD_SHAPES])
def test_every_backward_shape(R, shape, monkeypatch):
    """Each compiled backward row shape (lanes, warps, chunks per lane),
    forced through the tuning override, on rows that fill it and rows that
    leave lanes idle."""
    cap = 4 * shape[0] * shape[1] * shape[2]
    monkeypatch.setenv("MOE_ROUTER_BWD_SHAPE", ",".join(map(str, shape)))
    for E in sorted({cap, max(4, cap - 36), max(3, cap // 2 + 1)}):
        K = min(E, 8)
        for dt in ("f32", "bf16"):
            case = make_case(77, E, K, dtype=dt, seed=E)
            for sf in ("softmax", "sigmoid"):
                run_and_check_topk(R, case, K, sf, c=1.5)
                if dt == "f32":
                    run_and_check_aux(R, case, K, sf)


def adversarial_rows(E, K, rng):
    """Rows that defeat the cheap candidate bound: sorted rows (the top values
    sit in a few lanes), long runs of one value at the K boundary, a value
    tied far more often than the candidate buffer holds."""
    rows = []
    x = np.sort(rng.normal(0, 1, E))
    rows += [x[::-1].copy(), x.copy()]
    y = rng.normal(0, 1, E)
    top = np.sort(y)[::-1]
    v = top[K - 1]
    pos = rng.choice(E, size=min(E, 3 * K + 150), replace=False)
    y2 = np.where(y >= v, y, y - 10.0)
    y2[pos[: min(E, 3 * K + 150)]] = v           # many copies of the K-th value
    rows.append(y2)
    z = np.full(E, -4.0)
    z[: max(K - 3, 0)] = np.linspace(3, 2, max(K - 3, 0))
    z[rng.choice(np.arange(max(K - 3, 0), E), size=min(E - max(K - 3, 0), 200), replace=False)] = 1.5
    rows.append(z)
    w = rng.normal(0, 1, E)
    w[rng.choice(E, size=min(E, 4 * K), replace=False)] = 5.0 + rng.normal(0, 1e-3, min(E, 4 * K))
    rows.append(w)                                  # a dense cluster just above the rest
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("E,K", [(256, 8), (256, 22), (512, 22), (512, 36), (1024, 30), (2304, 36),
                                 (2304, 4)])
def test_adversarial_rows(R, path, E, K):
    rng = np.random.default_rng(E * 7 + K)
    x = adversarial_rows(E, K, rng)
    for dt in ("f32", "bf16"):
        from score_top_expert_gb300.workloads import round_to_bf16_values
        case = make_case(x.shape[0], E, K, dtype=dt, seed=3)
        case.logits = x if dt == "f32" else round_to_bf16_values(x)
        for sf in ("softmax", "sigmoid", "softmax_post"):
            run_and_check_topk(R, case, K, sf, c=2.0)
            if dt == "f32" and sf != "softmax_post":
                run_and_check_aux(R, case, K, sf)


def mixed_rows(T, E, K, seed):
    # a mix of row kinds in a fixed cycle (normal, wide, integer-valued with heavy
    # ties, adversarial, shifted and sorted rows), so that a threshold carried over
    # from a warp's previous row fails and recovers over and over
    rng = np.random.default_rng(seed)
    adv = adversarial_rows(E, K, rng)
    x = np.empty((T, E), dtype=np.float32)
    for i in range(T):
        kind = i % 6
        if kind == 0:
            x[i] = rng.normal(0, 1, E)
        elif kind == 1:
            x[i] = rng.normal(0, 3, E)
        elif kind == 2:
            x[i] = rng.integers(-3, 4, E)
        elif kind == 3:
            x[i] = adv[(i // 6) % adv.shape[0]][rng.permutation(E)]
        elif kind == 4:
            x[i] = rng.normal(0, 1, E) + 10.0  # shifted (sigmoid keys stay distinct in f64)
        else:
            x[i] = np.sort(rng.normal(0, 1, E))
    return x


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E,K", [(256, 8), (512, 22), (512, 36), (384, 30)])
def test_register_rows_in_sequence(R, E, K, dt):
    # many rows per warp, so that each row starts from the previous row's
    # threshold estimate
    from score_top_expert_gb300.workloads import round_to_bf16_values
    T = 12000
    x = mixed_rows(T, E, K, E * 31 + K)
    prev = R.force_path("register")
    try:
        case = make_case(T, E, K, dtype=dt, seed=5)
        case.logits = x if dt == "f32" else round_to_bf16_values(x)
        for sf in ("softmax", "sigmoid"):
            run_and_check_topk(R, case, K, sf, c=2.5, check_bwd=False)
            run_and_check_aux(R, case, K, sf)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E,K", [(1024, 30), (2304, 36), (1000, 24), (2000, 36)])
def test_staged_rows_taken_over(R, E, K, dt):
    # more rows than resident warps: the staged forward launches one one-warp
    # block per row, and running warps take over the rows of blocks that have
    # not started, so the rows a warp sees (and the threshold it carries from
    # one to the next) follow no fixed stride
    from score_top_expert_gb300.workloads import round_to_bf16_values
    T = 6000
    x = mixed_rows(T, E, K, E * 17 + K)
    prev = R.force_path("staged")
    try:
        case = make_case(T, E, K, dtype=dt, seed=6)
        case.logits = x if dt == "f32" else round_to_bf16_values(x)
        for sf in ("softmax", "sigmoid", "softmax_post"):
            run_and_check_topk(R, case, K, sf, c=2.5, check_bwd=False)
            if sf != "softmax_post":
                run_and_check_aux(R, case, K, sf)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E,G,gk,K", [(256, 8, 4, 8), (512, 16, 4, 8), (384, 12, 3, 9),
                                      (256, 0, 0, 8)])
def test_register_biased_rows_in_sequence(R, E, G, gk, K, dt):
    # bias (and groups) on the register path with many rows per warp: rows of
    # normal, wide, integer-valued and adversarial logits in a fixed cycle
    from score_top_expert_gb300.workloads import round_to_bf16_values
    rng = np.random.default_rng(E * 17 + K + G)
    T = 12000
    adv = adversarial_rows(E, K, rng)
    x = np.empty((T, E), dtype=np.float32)
    for i in range(T):
        kind = i % 4
        if kind == 0:
            x[i] = rng.normal(0, 1, E)
        elif kind == 1:
            x[i] = rng.normal(0, 3, E)
        elif kind == 2:
            x[i] = rng.integers(-3, 4, E)
        else:
            x[i] = adv[(i // 4) % adv.shape[0]][rng.permutation(E)]
    prev = R.force_path("register")
    try:
        case = make_case(T, E, K, dtype=dt, seed=9, with_bias=True)
        case.logits = x if dt == "f32" else round_to_bf16_values(x)
        for sf in ("sigmoid", "softmax", "softmax_post"):
            run_and_check_topk(R, case, K, sf, 2.5, G, gk, case.expert_bias, check_bwd=False)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


def test_bounded_wait_reports_a_timeout(R):
    """The bounded mbarrier wait gives up, reports status 1, and the context
    stays usable: a wait that nothing can complete runs out after 2 ms."""
    assert R.device_status() == 0
    R.selftest_bounded_wait(2000)
    torch.cuda.synchronize()
    assert R.device_status() == 1
    assert R.device_status() == 0          # reading cleared it
    case = make_case(64, 512, 8, seed=11)   # the router still works afterwards
    run_and_check_topk(R, case, 8, "softmax")
    assert R.device_status() == 0
    with pytest.raises(R.RouterError):
        R.selftest_bounded_wait(0)


# ---------------------------------------------------------------------------
# load-balancing aux loss
# ---------------------------------------------------------------------------
# fp32 sums: plain over a warp's rows of one block (at most a few hundred at these
# sizes), compensated across the block's warps and across blocks
AUX_LOSS_REL = 1e-5


# the row ranges per launch follow T and the column groups: one row per range (64 x
# 512), empty trailing ranges (65 x 2304: 25 ranges of 3 rows), 57 ranges (1024
# experts), scalar rows (257 experts)
@pytest.mark.parametrize("T,E,K", [(8192, 512, 22), (8192, 2304, 36), (1000, 257, 5), (77, 64, 4),
                                   (300, 2304, 36), (1, 8, 1), (64, 512, 8), (65, 2304, 8),
                                   (4096, 1024, 8)])
def test_aux_loss(R, T, E, K):
    case = make_case(T, E, K, seed=T + E)
    for sf in ("softmax", "sigmoid"):
        q, amap, inter = R.router_aux_scores_fwd(to_dev(case.logits), K, sf)
        loss, tokens = R.router_aux_loss_fwd(q, amap, K, 0.01)
        loss2, tokens2 = R.router_aux_loss_fwd(q, amap, K, 0.01)
        torch.cuda.synchronize()
        # identical bits on a repeat (fixed reduction order)
        assert loss.item() == loss2.item() and torch.equal(tokens, tokens2)
        # the same inputs through the oracle
        qn, mn = np64(q), amap.cpu().numpy()
        ref, ref_tok = O.aux_loss_fwd(qn, mn, K, 0.01)
        assert np.array_equal(tokens.cpu().numpy(), ref_tok)
        assert abs(loss.item() - ref) <= AUX_LOSS_REL * abs(ref) + 1e-12, (loss.item(), ref)
        # the whole pipeline against the oracle's own scores and map
        o = O.aux_scores_fwd(case.logits, K, sf)
        ref_full, _ = O.aux_loss_fwd(o["scores"], o["routing_map"], K, 0.01)
        assert abs(loss.item() - ref_full) <= AUX_LOSS_REL * abs(ref_full) + 1e-12
        # backward
        gl = torch.tensor([1.7], device=DEV)
        g = R.router_aux_loss_bwd(gl, tokens, T, K, 0.01)
        gref = O.aux_loss_bwd(1.7, ref_tok, T, K, 0.01)
        assert np.max(np.abs(np64(g) - gref) - 1e-6 * np.abs(gref)) <= 0.0


def test_aux_loss_unaligned_backward(R):
    T, E, K = 33, 100, 3
    case = make_case(T, E, K, seed=5)
    q, amap, _ = R.router_aux_scores_fwd(to_dev(case.logits), K, "softmax")
    loss, tokens = R.router_aux_loss_fwd(q, amap, K, 0.5)
    buf = torch.zeros(T * E + 1, device=DEV)
    g = R.router_aux_loss_bwd(torch.tensor([2.0], device=DEV), tokens, T, K, 0.5,
                              grad_aux_scores=buf[1:].view(T, E))
    gref = O.aux_loss_bwd(2.0, tokens.cpu().numpy(), T, K, 0.5)
    assert np.max(np.abs(np64(g) - gref) - 1e-6 * np.abs(gref)) <= 0.0
    assert buf[0].item() == 0.0
