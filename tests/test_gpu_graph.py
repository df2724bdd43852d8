"""Router kernels captured in a CUDA graph, chained on one stream the way a
training or serving step runs them (each launched with programmatic
dependent launch): replaying the graph on new inputs gives the eager
results bit for bit."""
import pytest

from score_top_expert_gb300.workloads import make_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


@pytest.mark.parametrize("T,E,K,sf", [(8192, 2304, 36, "softmax"), (4096, 512, 22, "sigmoid"),
                                      (6, 256, 8, "softmax_post")])
def test_graph_replay_matches_eager(R, T, E, K, sf):
    case = make_case(T, E, K, seed=E + K)
    src = torch.from_numpy(case.logits).to(DEV)
    g_src = torch.from_numpy(case.grad_probs).to(DEV)
    x = torch.empty_like(src)
    g = torch.empty_like(g_src)
    probs = torch.empty(T, E, device=DEV)
    rmap = torch.empty(T, E, dtype=torch.bool, device=DEV)
    scores = torch.empty(T, E, device=DEV)
    gx = torch.empty(T, E, device=DEV)
    w = torch.empty(T, K, device=DEV)
    idx = torch.empty(T, K, dtype=torch.int32, device=DEV)
    mo = {"expert_first_token_offset": torch.empty(E + 1, dtype=torch.int32, device=DEV)}
    for nm in ("permuted_to_unpermuted", "unpermuted_to_permuted", "permuted_experts"):
        mo[nm] = torch.empty(T * K, dtype=torch.int32, device=DEV)
    ws = torch.empty(R.lib().router_expert_maps_workspace_bytes(T, E), dtype=torch.uint8,
                     device=DEV)
    q = torch.empty(T, E, device=DEV)
    amap = torch.empty(T, E, dtype=torch.bool, device=DEV)
    loss = torch.empty(1, device=DEV)
    tok = torch.empty(E, dtype=torch.int32, device=DEV)
    lws = torch.empty(R.lib().router_aux_loss_workspace_bytes(T, E), dtype=torch.uint8,
                      device=DEV)
    scale = torch.empty(1, device=DEV)

    def step():
        # a torch kernel writes the inputs right before the router kernels read them
        torch.mul(src, scale, out=x)
        torch.mul(g_src, scale, out=g)
        R.router_topk_fwd(x, K, sf, probs=probs, routing_map=rmap, scores=scores)
        R.router_topk_bwd(g, rmap, scores, K, sf, grad_logits=gx)
        R.router_topk_fwd_maps(x, K, sf, topk_weights=w, topk_indices=idx,
                               token_expert_indices=False, out=mo, workspace=ws)
        if sf != "softmax_post":
            R.router_aux_scores_fwd(x, K, "softmax", scores=q, routing_map=amap)
            R.router_aux_loss_fwd(q, amap, K, 0.01, loss=loss, tokens_per_expert=tok,
                                  workspace=lws)

    outs = [probs, rmap, scores, gx, w, idx] + list(mo.values())
    if sf != "softmax_post":
        outs += [q, amap, loss, tok]

    def snapshot():
        torch.cuda.synchronize()
        return [o.clone() for o in outs]

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        scale.fill_(1.0)
        step()
    want_1 = snapshot()
    with torch.cuda.stream(stream):
        scale.fill_(-0.5)
        step()
    want_2 = snapshot()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()  # warm-up on the capture stream
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for fill, want in ((1.0, want_1), (-0.5, want_2), (1.0, want_1)):
        for o in outs:
            o.zero_()
        scale.fill_(fill)
        graph.replay()
        got = snapshot()
        for j, (a, b) in enumerate(zip(got, want)):
            assert torch.equal(a, b), (fill, j)
    assert R.device_status() == 0
