"""Seeded synthetic router workloads.

This module only draws inputs: router logits, incoming gradients and the
selection bias, with the shapes and value distributions of the router
benchmarks (8192 tokens, 256/512/2304 experts, fp32 or bf16 logits).  It
holds none of the router's arithmetic, so both the CUDA path's tests and the
CPU oracle can take their inputs from here.

Every array comes from numpy's PCG64 generator:

* logits: i.i.d. normal with standard deviation ``sigma``, drawn in fp32;
  for bf16 workloads the fp32 draws are rounded to bf16 (round to nearest,
  ties to even) and kept as the exact fp32 value of each bf16 number;
* grad_probs: i.i.d. N(0, 1) from stream ``seed + 1`` in the logits dtype;
* expert_bias: U(-bias_range, bias_range) fp32 from stream ``seed + 2``;
* grad_scores (aux-loss backward): i.i.d. N(0, 1) fp32 from ``seed + 3``;
* duplicate rows (tie-break stress): stream ``seed + 4``.
"""
from __future__ import annotations

import dataclasses

import numpy as np

BASE_SEED = 20261202


def config_seed(config_index: int) -> int:
    """Seed of a named workload: a fixed base plus 16 per workload."""
    return BASE_SEED + 16 * config_index


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def round_to_bf16_values(a: np.ndarray) -> np.ndarray:
    """fp32 array -> fp32 array holding the nearest bf16 numbers (RNE).

    Input preparation only: uses torch's own fp32 -> bf16 conversion.
    """
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


@dataclasses.dataclass
class RouterCase:
    """One seeded router problem: inputs for the forward and both backwards."""

    T: int
    E: int
    K: int
    dtype: str  # "f32" or "bf16"
    logits: np.ndarray  # [T, E] fp32 values (bf16-exact when dtype == "bf16")
    grad_probs: np.ndarray  # [T, E] fp32 values, same rounding as logits
    grad_scores: np.ndarray  # [T, E] fp32
    expert_bias: np.ndarray | None  # [E] fp32 or None
    dup_rows: np.ndarray  # indices of rows given exact duplicate values
    seed: int


def make_case(T: int, E: int, K: int, *, dtype: str = "f32", sigma: float = 1.0,
              seed: int = BASE_SEED, with_bias: bool = False,
              bias_range: float = 0.1, dup_frac: float = 0.0,
              all_equal_row: bool = False) -> RouterCase:
    """Draw one router workload.

    ``dup_frac`` > 0 picks that fraction of the rows (seeded permutation) and
    plants exact duplicates around the K-th largest value of each: three other
    positions receive the K-th largest value, so four equal values straddle
    the top-K boundary at mixed indices; every second such row also copies the
    value ranked about E/2 to two more positions.  ``all_equal_row`` makes one
    further row constant.
    """
    if dtype not in ("f32", "bf16"):
        raise ValueError(dtype)
    logits = (_rng(seed).standard_normal((T, E), dtype=np.float32)
              * np.float32(sigma)).astype(np.float32)
    grad = _rng(seed + 1).standard_normal((T, E), dtype=np.float32)
    bias = None
    if with_bias:
        bias = _rng(seed + 2).uniform(-bias_range, bias_range, E).astype(np.float32)
    grad_scores = _rng(seed + 3).standard_normal((T, E), dtype=np.float32)

    dup_rows = np.zeros(0, dtype=np.int64)
    if (dup_frac > 0 or all_equal_row) and T > 0:
        r = _rng(seed + 4)
        perm = r.permutation(T)
        n_dup = int(round(dup_frac * T)) if dup_frac > 0 else 0
        n_dup = min(n_dup, T - (1 if all_equal_row else 0))
        dup_rows = np.sort(perm[:n_dup])
        for j, row in enumerate(perm[:n_dup]):
            x = logits[row]
            order = np.argsort(-x, kind="stable")
            kth = order[min(K, E) - 1]
            others = np.setdiff1d(np.arange(E), [kth])
            pos = r.choice(others, size=min(3, others.size), replace=False)
            x[pos] = x[kth]
            if j % 2 == 1 and E >= 8:
                deep = order[E // 2]
                rest = np.setdiff1d(np.arange(E), np.concatenate([[kth, deep], pos]))
                pos2 = r.choice(rest, size=min(2, rest.size), replace=False)
                x[pos2] = x[deep]
        if all_equal_row:
            row = perm[n_dup]
            logits[row, :] = logits[row, 0]
            dup_rows = np.sort(np.append(dup_rows, row))

    if dtype == "bf16":
        logits = round_to_bf16_values(logits)
        grad = round_to_bf16_values(grad)
    return RouterCase(T=T, E=E, K=K, dtype=dtype, logits=logits, grad_probs=grad,
                      grad_scores=grad_scores, expert_bias=bias, dup_rows=dup_rows,
                      seed=seed)


# Named workloads: the router benchmarks' shapes and distributions.
# Each entry: (config index for the seed, keyword arguments of make_case and of
# the router call).
WORKLOADS = {
    # 1024 tokens, 64 experts, top-4 softmax, fp32 N(0,1)
    "t1024_e64_k4": dict(cfg=0, T=1024, E=64, K=4, sigma=1.0, scaling_factor=1.0),
    # 8192 tokens, 256 experts, top-4 / top-8
    "t8192_e256_k4": dict(cfg=1, T=8192, E=256, K=4, sigma=1.0, scaling_factor=1.0),
    "t8192_e256_k8": dict(cfg=1, T=8192, E=256, K=8, sigma=1.0, scaling_factor=1.0),
    # 8192 tokens, 512 experts, top-22, N(0,2) logits, scaling factor 2.5
    "t8192_e512_k22": dict(cfg=2, T=8192, E=512, K=22, sigma=2.0, scaling_factor=2.5),
    # 8192 tokens, 2304 experts, top-36, 1 % of rows with exact duplicates
    "t8192_e2304_k36": dict(cfg=3, T=8192, E=2304, K=36, sigma=1.0, scaling_factor=1.0,
                            dup_frac=0.01, all_equal_row=True),
    # group-limited sigmoid router: 16384 tokens, 256 experts in 8 groups,
    # keep 4 groups, top-8, bias U(-0.1, 0.1), scaling 2.5, bf16 logits
    "t16384_e256_k8_grouped": dict(cfg=4, T=16384, E=256, K=8, sigma=1.0,
                                   scaling_factor=2.5, num_groups=8, group_topk=4,
                                   with_bias=True, dtype="bf16", score_func="sigmoid"),
}


def make_workload(name: str, *, dtype: str | None = None, T: int | None = None,
                  K: int | None = None) -> tuple[RouterCase, dict]:
    """Build a named workload; returns the inputs and the router arguments.

    ``T`` may shrink the token count (the first T rows of the same draw are
    not kept: a smaller T is a fresh draw of the same recipe and seed).
    """
    w = dict(WORKLOADS[name])
    seed = config_seed(w.pop("cfg"))
    dt = dtype or w.pop("dtype", "f32")
    w.pop("dtype", None)
    TT = T if T is not None else w["T"]
    KK = K if K is not None else w["K"]
    case = make_case(TT, w["E"], KK, dtype=dt, sigma=w["sigma"], seed=seed,
                     with_bias=w.get("with_bias", False),
                     dup_frac=w.get("dup_frac", 0.0),
                     all_equal_row=w.get("all_equal_row", False))
    args = dict(K=KK, scaling_factor=w["scaling_factor"],
                num_groups=w.get("num_groups", 0), group_topk=w.get("group_topk", 0),
                score_func=w.get("score_func", "softmax"))
    return case, args


def make_device_normals(torch, shape, seed: int, device, sigma: float = 1.0):
    """Seeded N(0, sigma) fp32 tensor drawn on the device (torch's generator):
    for batches too large to draw on the host.  Tests hand the oracle the rows
    they check, copied back from this tensor."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sigma
