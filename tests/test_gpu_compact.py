"""Compact [T, K] router outputs on the GPU against the CPU oracle, through
the C ABI: indices in rank order, weights, expanded rows k T + t, and the
optional dense outputs of the same call against router_topk_fwd."""
import numpy as np
import pytest

import oracle.router_oracle as O
from compare import F32_ABS, MAX_MISMATCH_FRAC
from score_top_expert_gb300.workloads import make_case, make_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
TD = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


@pytest.fixture(params=["auto", "segment", "staged", "register"])
def path(R, request):
    prev = R.force_path(request.param)
    yield request.param
    R.force_path(prev)
    assert R.device_status() == 0


def to_dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV).to(TD[dtype])


def near(a, b):
    d = abs(a - b)
    return 0.0 < d <= O.NEAR_TIE_REL * max(abs(a), abs(b))


def check_compact(R, case, K, sf, c=1.0, ng=0, gk=0, bias=None, strided=False):
    """Run the compact forward (with dense outputs) and compare with the
    oracle; returns the number of rows whose selected set differs."""
    dt = case.dtype
    T, E = case.logits.shape
    x = to_dev(case.logits, dt)
    b = None if bias is None else to_dev(bias)
    w_buf = i_buf = None
    if strided:  # column views of wider buffers: the extra columns stay untouched
        w_buf = torch.full((T, K + 3), -7.0, device=DEV)
        i_buf = torch.full((T, K + 5), -9, dtype=torch.int32, device=DEV)
    w, idx, tei, probs, rmap, scores = R.router_topk_fwd_compact(
        x, K, sf, ng, gk, c, b, dense=True,
        topk_weights=None if w_buf is None else w_buf[:, :K],
        topk_indices=None if i_buf is None else i_buf[:, :K])
    if strided:
        assert (w_buf[:, K:] == -7.0).all() and (i_buf[:, K:] == -9).all()
    # the dense outputs are those of router_topk_fwd on the same input: the
    # map and the scores bit for bit; the renormalised probs up to the order
    # in which the K selected scores are summed (it follows the candidate
    # order, which depends on each launch's rows-per-warp plan)
    p0, m0, s0 = R.router_topk_fwd(x, K, sf, ng, gk, c, b)
    assert torch.equal(rmap, m0) and torch.equal(scores, s0)
    dp = (probs.double() - p0.double()).abs()
    if dt == "f32":
        assert dp.max().item() <= F32_ABS
    else:
        assert (dp <= 2.0 ** -7 * p0.double().abs()).all()
    # compact and dense agree: the indices are the map's support, the
    # weights its probs (bf16 probs are the weights rounded)
    idx_l = idx.long()
    assert torch.equal(torch.gather(rmap, 1, idx_l), torch.ones_like(idx, dtype=torch.bool))
    assert (rmap.sum(dim=1) == K).all()
    assert torch.equal(torch.gather(probs, 1, idx_l), w.to(probs.dtype))
    # expanded rows
    want_tei = (torch.arange(K, device=DEV)[None, :] * T
                + torch.arange(T, device=DEV)[:, None]).to(torch.int32)
    assert torch.equal(tei, want_tei)

    return compare_with_oracle(case, K, sf, c, ng, gk, bias, idx, w)


def compare_with_oracle(case, K, sf, c, ng, gk, bias, idx, w):
    """Compact indices and weights against the oracle: the selected sets
    equal outside near ties, the rank order by key, the weights within the
    fp32 bound; returns the number of rows whose selected set differs."""
    T = case.logits.shape[0]
    ref = O.topk_fwd_compact(case.logits, K, sf, ng, gk, c, bias)
    gi = idx.cpu().numpy().astype(np.int64)
    gw = w.cpu().numpy().astype(np.float64)
    ri, rw, nt = ref["topk_indices"], ref["topk_weights"], ref["near_tie"]
    # oracle keys (s + bias) of every expert, for the order check
    keys = O.topk_fwd(case.logits, K, sf, ng, gk, c, bias)["scores"]
    if bias is not None:
        keys = keys + np.asarray(bias, np.float64)[None, :]
    set_diff = np.any(np.sort(gi, 1) != np.sort(ri, 1), axis=1)
    assert not np.any(set_diff & ~nt), "selected set differs outside near ties"
    assert set_diff.sum() <= MAX_MISMATCH_FRAC * T
    for t in np.nonzero(~set_diff)[0]:
        if not np.array_equal(gi[t], ri[t]):
            # the order may differ only between keys within the near-tie distance
            kk = keys[t][gi[t]]
            for k in range(K - 1):
                a, bb = kk[k], kk[k + 1]
                assert a > bb or (a == bb and gi[t][k] < gi[t][k + 1]) or near(a, bb), \
                    (t, k, gi[t], ri[t])
        # weights, matched by expert
        og, orr = np.argsort(gi[t]), np.argsort(ri[t])
        assert np.max(np.abs(gw[t][og] - rw[t][orr])) <= F32_ABS, t
    return int(set_diff.sum())


WORKLOADS = [("t8192_e2304_k36", "softmax", "f32"), ("t8192_e512_k22", "sigmoid", "f32"),
             ("t8192_e256_k8", "softmax_post", "bf16"),
             ("t16384_e256_k8_grouped", "sigmoid", "bf16")]


@pytest.mark.parametrize("name,sf,dt", WORKLOADS, ids=[f"{n}-{s}-{d}" for n, s, d in WORKLOADS])
def test_compact_workload(R, path, name, sf, dt):
    case, args = make_workload(name, dtype=dt)
    check_compact(R, case, args["K"], sf, args["scaling_factor"], args["num_groups"],
                  args["group_topk"], case.expert_bias, strided=(name == "t8192_e512_k22"))


@pytest.mark.parametrize("E", [1, 5, 64, 100, 256, 513, 1000, 2304])
def test_compact_shapes(R, path, E):
    for dt in ("f32", "bf16"):
        for sf in ("softmax", "sigmoid", "softmax_post"):
            for K in sorted({1, min(E, 4), min(E, 36)}):
                case = make_case(67, E, K, dtype=dt, sigma=1.5, seed=E * 7 + K)
                check_compact(R, case, K, sf, c=2.5, strided=(K == 4))


def test_compact_bias_and_groups(R, path):
    rng = np.random.default_rng(5)
    for E, K, ng, gk in ((256, 8, 8, 4), (64, 6, 4, 2), (512, 22, 0, 0), (2304, 36, 16, 4)):
        case = make_case(129, E, K, sigma=1.0, seed=E + K)
        bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        for sf in ("softmax", "sigmoid", "softmax_post"):
            check_compact(R, case, K, sf, c=1.5, ng=ng, gk=gk, bias=bias)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E,K,ng,gk", [(512, 22, 0, 0), (512, 36, 0, 0), (256, 8, 8, 4),
                                       (384, 12, 12, 4)])
def test_register_compact_rows_in_sequence(R, E, K, ng, gk, dt):
    # compact outputs on the register path with many rows per warp (each row
    # starting from the previous row's threshold): normal, wide and
    # integer-valued rows in a fixed cycle, with a bias
    from score_top_expert_gb300.workloads import round_to_bf16_values
    rng = np.random.default_rng(E + K + ng)
    T = 12000
    x = np.empty((T, E), dtype=np.float32)
    for i in range(T):
        kind = i % 3
        x[i] = (rng.normal(0, 1, E) if kind == 0 else rng.normal(0, 3, E) if kind == 1
                else rng.integers(-3, 4, E))
    case = make_case(T, E, K, dtype=dt, seed=4)
    case.logits = x if dt == "f32" else round_to_bf16_values(x)
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    prev = R.force_path("register")
    try:
        for sf in ("softmax", "sigmoid"):
            check_compact(R, case, K, sf, c=1.5, ng=ng, gk=gk, bias=bias)
            # without dense outputs: the same compact rows
            xd, bd = to_dev(case.logits, dt), to_dev(bias)
            full = R.router_topk_fwd_compact(xd, K, sf, ng, gk, 1.5, bd, dense=True)
            only = R.router_topk_fwd_compact(xd, K, sf, ng, gk, 1.5, bd)
            assert only[3] is None and only[4] is None and only[5] is None
            for a, b in zip(full[:3], only[:3]):
                assert torch.equal(a, b)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_staged_compact_rows_taken_over(R, dt):
    # compact outputs from the staged forward's one-warp blocks that take over
    # the rows of blocks not yet started (more rows than resident warps)
    from score_top_expert_gb300.workloads import round_to_bf16_values
    E, K, T = 2304, 36, 6000
    rng = np.random.default_rng(23)
    x = np.empty((T, E), dtype=np.float32)
    for i in range(T):
        kind = i % 3
        x[i] = (rng.normal(0, 1, E) if kind == 0 else rng.normal(0, 3, E) if kind == 1
                else rng.integers(-3, 4, E))
    case = make_case(T, E, K, dtype=dt, seed=8)
    case.logits = x if dt == "f32" else round_to_bf16_values(x)
    prev = R.force_path("staged")
    try:
        xd = to_dev(case.logits, dt)
        for sf in ("softmax", "sigmoid", "softmax_post"):
            check_compact(R, case, K, sf, c=1.5)
            # without dense outputs (fp32 rows of this width: one stage per
            # warp, refilled before the ranking): the same compact rows, for
            # batches above and below that launch's row threshold
            for t in (T, 3000, 2000):
                full = R.router_topk_fwd_compact(xd[:t], K, sf, scaling_factor=1.5, dense=True)
                only = R.router_topk_fwd_compact(xd[:t], K, sf, scaling_factor=1.5)
                assert only[3] is None and only[4] is None and only[5] is None
                for a, b in zip(full[:3], only[:3]):
                    assert torch.equal(a, b)
        # rows that do not fill the chunk grid (2000 of 2304 slots)
        xp = xd[:, :2000].contiguous()
        for sf in ("softmax", "sigmoid"):
            full = R.router_topk_fwd_compact(xp, K, sf, scaling_factor=1.5, dense=True)
            only = R.router_topk_fwd_compact(xp, K, sf, scaling_factor=1.5)
            for a, b in zip(full[:3], only[:3]):
                assert torch.equal(a, b)
    finally:
        R.force_path(prev)
    assert R.device_status() == 0


@pytest.mark.parametrize("sf", ["softmax", "sigmoid"])
def test_unaligned_compact_rows(R, sf):
    # logits 4 bytes past a 16-byte boundary: no bulk copy can take the rows,
    # which a batch this size would otherwise send to the one-stage launch
    E, K, T = 2304, 36, 3000
    case = make_case(T, E, K, seed=31)
    buf = torch.zeros(T * E + 1, device=DEV)
    x = buf[1:].view(T, E)
    x.copy_(to_dev(case.logits))
    assert x.data_ptr() % 16 != 0
    w, idx, tei, *_ = R.router_topk_fwd_compact(x, K, sf, scaling_factor=1.5)
    assert compare_with_oracle(case, K, sf, 1.5, 0, 0, None, idx, w) == 0
    want_tei = (torch.arange(K, device=DEV)[None, :] * T
                + torch.arange(T, device=DEV)[:, None]).to(torch.int32)
    assert torch.equal(tei, want_tei)
    assert R.device_status() == 0


def test_compact_ties(R, path):
    # integer logits: heavy exact ties inside and at the boundary of the top-K
    rng = np.random.default_rng(9)
    for E, K in ((64, 8), (512, 22), (2304, 36)):
        case = make_case(64, E, K, seed=3)
        case.logits[:] = rng.integers(-2, 3, case.logits.shape).astype(np.float32)
        case.logits[0] = 0.0  # one all-equal row
        for sf in ("softmax", "sigmoid"):
            assert check_compact(R, case, K, sf) == 0


def test_compact_zero_tokens(R):
    x = torch.empty((0, 64), device=DEV)
    w, idx, tei, _, _, _ = R.router_topk_fwd_compact(x, 4)
    assert w.shape == (0, 4) and idx.shape == (0, 4) and tei.shape == (0, 4)
