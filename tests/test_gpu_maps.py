"""(expert, token)-sorted expert maps on the GPU against the CPU oracle,
through the C ABI: the stand-alone maps of given indices (bit-exact), and the
router with maps (the fused one-block decode launch and the composed launch)
end to end."""
import numpy as np
import pytest

import oracle.router_oracle as O
from compare import F32_ABS
from score_top_expert_gb300.workloads import make_case, make_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
TD = {"f32": torch.float32, "bf16": torch.bfloat16}
KEYS = ("expert_first_token_offset", "permuted_to_unpermuted", "unpermuted_to_permuted",
        "permuted_experts")


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


def to_dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV).to(TD[dtype])


def assert_maps_equal(got, idx, E):
    ref = O.expert_maps(idx, E)
    for name, g in zip(KEYS, got):
        assert np.array_equal(g.cpu().numpy().astype(np.int64), ref[name]), name


def random_indices(T, E, K, seed):
    rng = np.random.default_rng(seed)
    # distinct experts per row, skewed towards low expert ids (uneven loads)
    w = 1.0 / (1.0 + np.arange(E)) ** 0.7
    return np.stack([rng.choice(E, K, replace=False, p=w / w.sum()) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,K", [(1, 8, 1), (3, 4, 2), (7, 64, 8), (255, 256, 8), (256, 256, 8),
                                   (257, 100, 5), (1000, 512, 22), (8192, 2304, 36),
                                   (16384, 256, 8), (600, 2304, 1)])
def test_expert_maps_of_given_indices(R, T, E, K):
    idx = random_indices(T, E, K, seed=T + E + K)
    got = R.router_expert_maps(torch.from_numpy(idx).to(DEV), E)
    assert_maps_equal(got, idx, E)
    # a second call on the same workspace gives the same maps
    again = R.router_expert_maps(torch.from_numpy(idx).to(DEV), E)
    for a, b in zip(got, again):
        assert torch.equal(a, b)


def test_expert_maps_beyond_one_wave(R):
    # 131072 tokens are 2048 tiles of 64: more blocks than fit on the GPU at
    # once, so the maps take the three-launch path instead of the cooperative
    # one; both must give the oracle's maps
    T, E, K = 131072, 64, 2
    idx = random_indices(T, E, K, seed=31)
    assert_maps_equal(R.router_expert_maps(torch.from_numpy(idx).to(DEV), E), idx, E)


def test_expert_maps_strided_and_invalid(R):
    T, E, K = 300, 64, 6
    idx = random_indices(T, E, K, seed=4)
    wide = torch.full((T, K + 3), 7, dtype=torch.int32, device=DEV)
    wide[:, :K] = torch.from_numpy(idx).to(DEV)
    assert_maps_equal(R.router_expert_maps(wide[:, :K], E), idx, E)
    # entries outside [0, E) are skipped: -1 in the inverse map, no permuted row
    bad = idx.copy()
    bad[5, 2] = -1
    bad[77, 0] = E
    off, p2u, u2p, pexp = (t.cpu().numpy() for t in
                           R.router_expert_maps(torch.from_numpy(bad).to(DEV), E))
    n_valid = T * K - 2
    assert off[E] == n_valid
    u2p_ok = u2p.copy()
    assert u2p[5 + 2 * T] == -1 and u2p[77 + 0 * T] == -1
    valid = np.ones(T * K, bool)
    valid[[5 + 2 * T, 77]] = False
    assert sorted(p2u[:n_valid].tolist()) == sorted(np.nonzero(valid)[0].tolist())
    assert np.array_equal(u2p_ok[p2u[:n_valid]], np.arange(n_valid))
    for e in range(E):
        tok = p2u[off[e]:off[e + 1]] % T
        assert np.all(np.diff(tok) > 0) and np.all(pexp[off[e]:off[e + 1]] == e)


def check_router_maps(R, case, K, sf, c=1.0, ng=0, gk=0, bias=None):
    """The router with maps against the oracle: the selected set per row (up
    to near ties), the weights matched by expert (fp32 tolerance), the
    expanded rows, and the maps of the GPU's own indices (bit-exact)."""
    dt = case.dtype
    T, E = case.logits.shape
    x = to_dev(case.logits, dt)
    b = None if bias is None else to_dev(bias)
    w, idx, tei, *maps = R.router_topk_fwd_maps(x, K, sf, ng, gk, c, b)
    gi = idx.cpu().numpy().astype(np.int64)
    gw = w.cpu().numpy().astype(np.float64)
    assert_maps_equal(maps, gi, E)
    want_tei = np.arange(K)[None, :] * T + np.arange(T)[:, None]
    assert np.array_equal(tei.cpu().numpy(), want_tei)
    ref = O.topk_fwd_compact(case.logits, K, sf, ng, gk, c, bias)
    ri, rw = ref["topk_indices"], ref["topk_weights"]
    diff = np.any(np.sort(gi, 1) != np.sort(ri, 1), axis=1)
    assert not np.any(diff & ~ref["near_tie"])
    for t in np.nonzero(~diff)[0]:
        og, orr = np.argsort(gi[t]), np.argsort(ri[t])
        assert np.max(np.abs(gw[t][og] - rw[t][orr])) <= F32_ABS, t


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_fused_decode_maps(R, T, dt):
    for K in (1, 2, 4, 6, 8, 10):
        case = make_case(T, 512, K, dtype=dt, seed=77 + T)
        for sf in ("softmax", "sigmoid", "softmax_post"):
            check_router_maps(R, case, K, sf)


def test_fused_decode_maps_shapes(R):
    rng = np.random.default_rng(3)
    for E, K, ng, gk in ((64, 8, 0, 0), (256, 8, 8, 4), (2304, 36, 0, 0), (2304, 36, 16, 4),
                         (4, 4, 0, 0), (1000, 22, 0, 0)):
        case = make_case(5, E, K, seed=E)
        bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if ng else None
        check_router_maps(R, case, K, "sigmoid", 2.5, ng, gk, bias)
        check_router_maps(R, case, K, "softmax", 1.0, ng, gk, bias)


@pytest.mark.parametrize("name", ["t8192_e512_k22", "t16384_e256_k8_grouped"])
def test_composed_maps(R, name):
    case, args = make_workload(name)
    check_router_maps(R, case, args["K"], "sigmoid", args["scaling_factor"], args["num_groups"],
                      args["group_topk"], case.expert_bias)


def test_unaligned_small_batch_uses_the_composed_path(R):
    case = make_case(3, 101, 5, seed=8)  # E % 4 != 0: no fused launch
    check_router_maps(R, case, 5, "softmax")
