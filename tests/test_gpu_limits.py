"""The largest legal batch: tokens x experts just under INT_MAX (932067 x 2304,
K = 36), through the C ABI.  The oracle checks sampled rows (the first, a
middle stretch and the last rows) of the forward and backward; the maps of
the batch's 33.5 M choices are checked by their defining properties on
sampled choices and in full where cheap."""
import numpy as np
import pytest

import oracle.router_oracle as O
from compare import F32_ABS
from score_top_expert_gb300.workloads import make_device_normals

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DEV = "cuda:0"
E, K = 2304, 36
T = 2147483647 // E  # 932067: T * E <= INT_MAX


@pytest.fixture(scope="module")
def R():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from score_top_expert_gb300 import build
    build.build()
    import score_top_expert_gb300.router as r
    r.lib()
    return r


def sample_rows():
    return np.concatenate([np.arange(0, 8), np.arange(T // 2, T // 2 + 8), np.arange(T - 8, T)])


def test_forward_and_backward_at_the_size_limit(R):
    assert T * E <= 2**31 - 1 and (T + 1) * E > 2**31 - 1
    try:
        x = make_device_normals(torch, (T, E), 4040, DEV)
        g = make_device_normals(torch, (T, E), 4041, DEV)
        probs, rmap, scores = R.router_topk_fwd(x, K, "softmax")
        gx = R.router_topk_bwd(g, rmap, scores, K, "softmax")
        torch.cuda.synchronize()
        rows = torch.from_numpy(sample_rows()).to(DEV)
        xs = x[rows].double().cpu().numpy()
        gs = g[rows].double().cpu().numpy()
        ref = O.topk_fwd(xs, K, "softmax")
        assert np.array_equal(rmap[rows].cpu().numpy(), ref["routing_map"])
        assert np.max(np.abs(probs[rows].double().cpu().numpy() - ref["probs"])) <= F32_ABS
        assert np.max(np.abs(scores[rows].double().cpu().numpy() - ref["scores"])) <= F32_ABS
        gref = O.topk_bwd(gs, ref["routing_map"], ref["scores"], "softmax")
        assert np.max(np.abs(gx[rows].double().cpu().numpy() - gref)) <= F32_ABS
        assert (rmap.sum(dim=1) == K).all()
        del probs, rmap, scores, gx, g
        # compact outputs and the maps of all T K choices (three-launch path)
        w, idx, tei, off, p2u, u2p, pexp = R.router_topk_fwd_maps(x, K, "softmax")
        torch.cuda.synchronize()
        cref = O.topk_fwd_compact(xs, K, "softmax")
        assert np.array_equal(idx[rows].cpu().numpy(), cref["topk_indices"])
        assert np.max(np.abs(w[rows].double().cpu().numpy() - cref["topk_weights"])) <= F32_ABS
        n = T * K
        off_h = off.cpu().numpy().astype(np.int64)
        assert off_h[0] == 0 and off_h[-1] == n and np.all(np.diff(off_h) >= 0)
        counts = torch.bincount(idx.flatten().long(), minlength=E).cpu().numpy()
        assert np.array_equal(np.diff(off_h), counts)
        # sampled choices (t, k): u = t + k T -> p -> expert and back
        ts = torch.from_numpy(sample_rows()).to(DEV).long()
        ks = torch.arange(K, device=DEV).long()
        u = (ts[:, None] + ks[None, :] * T).flatten()
        p = u2p[u].long()
        assert torch.equal(p2u[p].long(), u)
        assert torch.equal(pexp[p], idx[ts].flatten())
        pe = pexp[p].long()
        offd = off.long()
        assert bool(((offd[pe] <= p) & (p < offd[pe + 1])).all())
        # every permuted row maps back: p2u is a permutation and u2p its inverse
        assert torch.equal(u2p[p2u.long()].long(), torch.arange(n, device=DEV))
        assert torch.equal(tei[ts].flatten().long(), u)
    finally:
        torch.cuda.empty_cache()
