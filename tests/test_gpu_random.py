"""Seeded random configurations against the CPU oracle through the C ABI:
expert count, K, batch, score function, dtype, bias, groups, scaling and
kernel path drawn at random, each checked on the dense forward and backward,
the compact outputs and the expert maps."""
import numpy as np
import pytest

import oracle.router_oracle as O
from compare import assert_close, compare_map
from score_top_expert_gb300.workloads import make_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
TD = {"f32": torch.float32, "bf16": torch.bfloat16}
N_CONFIGS = 200


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


def draw(rng):
    E = int(rng.choice([1, 3, 8, 17, 64, 100, 128, 200, 256, 300, 512, 640, 1000, 1024, 2048,
                        2304]))
    K = int(rng.integers(1, min(E, 36) + 1))
    T = int(rng.integers(1, 200))
    sf = str(rng.choice(["softmax", "sigmoid", "softmax_post"]))
    dt = "bf16" if rng.random() < 0.3 else "f32"
    c = float(rng.choice([1.0, 2.5, 0.7]))
    ng = gk = 0
    if rng.random() < 0.3:
        divs = [g for g in range(2, min(E, 32) + 1) if E % g == 0]
        opts = [(g, k) for g in divs for k in range(1, g + 1)
                if K % k == 0 and K // k <= E // g]
        if opts:
            ng, gk = opts[int(rng.integers(len(opts)))]
    bias = rng.uniform(-0.1, 0.1, E).astype(np.float32) if rng.random() < 0.3 else None
    path = str(rng.choice(["auto", "segment", "staged", "register"]))
    lanes = int(rng.choice([0, 0, 8, 16, 32]))
    sigma = float(rng.choice([0.5, 1.0, 2.0]))
    return dict(E=E, K=K, T=T, sf=sf, dt=dt, c=c, ng=ng, gk=gk, bias=bias, path=path,
                lanes=lanes, sigma=sigma)


def to_dev(a, dtype="f32"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV).to(TD[dtype])


@pytest.mark.parametrize("i", range(N_CONFIGS))
def test_random_config(R, i):
    rng = np.random.default_rng(90210 + i)
    cfg = draw(rng)
    E, K, T, sf, dt = cfg["E"], cfg["K"], cfg["T"], cfg["sf"], cfg["dt"]
    c, ng, gk, bias = cfg["c"], cfg["ng"], cfg["gk"], cfg["bias"]
    case = make_case(T, E, K, dtype=dt, sigma=cfg["sigma"], seed=777 + i)
    prev_path = R.force_path(cfg["path"])
    prev_lanes = R.force_fwd_lanes(cfg["lanes"])
    try:
        x = to_dev(case.logits, dt)
        b = None if bias is None else to_dev(bias)
        probs, rmap, scores = R.router_topk_fwd(x, K, sf, ng, gk, c, b)
        ref = O.topk_fwd(case.logits, K, sf, ng, gk, c, bias)
        rep = compare_map(rmap.cpu().numpy(), ref["routing_map"], ref["near_tie"])
        rep.check(f"random config {i}: {cfg}")
        ok = rep.ok_rows
        assert_close(probs.double().cpu().numpy(), ref["probs"], dt, ok, f"probs {cfg}")
        assert_close(scores.double().cpu().numpy(), ref["scores"], "f32", None, f"scores {cfg}")
        g = to_dev(case.grad_probs, dt)
        gx = R.router_topk_bwd(g, rmap, scores, K, sf, c)
        gref = O.topk_bwd(case.grad_probs, ref["routing_map"], ref["scores"], sf, c)
        assert_close(gx.double().cpu().numpy(), gref, dt, ok, f"grad {cfg}")
        # compact outputs and the expert maps of the GPU's own choices
        w, idx, tei, *maps = R.router_topk_fwd_maps(x, K, sf, ng, gk, c, b)
        gi = idx.cpu().numpy().astype(np.int64)
        cref = O.topk_fwd_compact(case.logits, K, sf, ng, gk, c, bias)
        same = np.all(np.sort(gi, 1) == np.sort(cref["topk_indices"], 1), axis=1)
        assert np.all(same | cref["near_tie"]), f"compact set {cfg}"
        gw = w.cpu().numpy().astype(np.float64)
        for t in np.nonzero(same)[0]:
            og, orr = np.argsort(gi[t]), np.argsort(cref["topk_indices"][t])
            assert np.max(np.abs(gw[t][og] - cref["topk_weights"][t][orr])) <= 1e-6, (t, cfg)
        assert np.array_equal(tei.cpu().numpy(), cref["token_expert_indices"])
        mref = O.expert_maps(gi, E)
        for got, name in zip(maps, ("expert_first_token_offset", "permuted_to_unpermuted",
                                    "unpermuted_to_permuted", "permuted_experts")):
            assert np.array_equal(got.cpu().numpy().astype(np.int64), mref[name]), (name, cfg)
    finally:
        R.force_path(prev_path)
        R.force_fwd_lanes(prev_lanes)
    assert R.device_status() == 0
