"""The staged forward's stealing launch (one-warp blocks that take over the
rows of blocks not yet started) against its persistent launch
(MOE_ROUTER_STEAL=0): the same outputs, bit for bit, for batches with more
rows than the GPU holds warps at once.  The switch is read once per process,
so each launch runs in its own child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import hashlib, sys
import torch
sys.path.insert(0, ".")
from score_top_expert_gb300 import build
build.build()
import score_top_expert_gb300.router as R
from score_top_expert_gb300.workloads import make_case
h = hashlib.sha256()
dts = {"f32": torch.float32, "bf16": torch.bfloat16}
for E, K, sf, dt in ((2304, 36, "softmax", "f32"), (1000, 24, "sigmoid", "f32"),
                     (2304, 36, "softmax_post", "bf16"), (1024, 30, "sigmoid", "bf16")):
    case = make_case(6000, E, K, dtype=dt, seed=E + K)
    x = torch.from_numpy(case.logits).cuda().to(dts[dt])
    outs = list(R.router_topk_fwd(x, K, sf, scaling_factor=2.5))
    outs += [o for o in R.router_topk_fwd_compact(x, K, sf, scaling_factor=2.5)[:3]]
    if sf != "softmax_post":
        outs += list(R.router_aux_scores_fwd(x, K, sf))
    for o in outs:
        h.update(o.contiguous().view(torch.uint8).cpu().numpy().tobytes())
torch.cuda.synchronize()
assert R.device_status() == 0
print(h.hexdigest())
'''


def digest(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout.strip().splitlines()[-1]


def test_stealing_launch_matches_the_persistent_grid():
    assert torch_cuda_available()
    stealing = digest({})
    persistent = digest({"MOE_ROUTER_STEAL": "0"})
    assert len(stealing) == 64 and stealing == persistent


def torch_cuda_available():
    torch = pytest.importorskip("torch")
    return torch.cuda.is_available()
