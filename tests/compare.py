"""Element-by-element comparison of the CUDA router against the CPU oracle.

Tolerances (the router's stated accuracy targets):
* routing_map: bit-exact on every row except near ties (the oracle's K-th and
  (K+1)-th keys, or its group_topk-th and next group scores, distinct but
  within 1e-6 relative).  A mismatch on any other row fails; mismatched rows
  must stay below 1e-4 of all rows.  Exact ties are not exempt.
* fp32 outputs: |gpu - ref| <= 1e-6 against the float64 oracle.
* bf16 outputs: |gpu - ref_bf16| <= 2e-2 |ref_bf16| + 1e-6, with ref_bf16 the
  oracle value rounded to bf16 by the oracle.
Values on rows whose map legitimately differs (near ties) are not compared.
"""
from __future__ import annotations

import dataclasses

import numpy as np

import oracle.router_oracle as O

F32_ABS = 1e-6
BF16_REL = 2e-2
BF16_ABS = 1e-6
MAX_MISMATCH_FRAC = 1e-4


@dataclasses.dataclass
class MapReport:
    rows: int
    near_tie_rows: int
    mismatched_rows: int
    mismatched_non_near: int
    ok_rows: np.ndarray  # bool [T]: maps agree

    def check(self, what=""):
        assert self.mismatched_non_near == 0, \
            f"{what}: {self.mismatched_non_near} rows mismatch outside near ties"
        assert self.mismatched_rows <= MAX_MISMATCH_FRAC * self.rows, \
            f"{what}: {self.mismatched_rows}/{self.rows} rows mismatch"


# Near-tie record of the full-size workloads, printed in the test session's
# terminal summary: label -> [rows, near-tie rows, most mismatched rows over
# the runs, runs].
NEAR_TIE_RECORD: dict[str, list[int]] = {}


def record_near_ties(label: str, rep: MapReport) -> None:
    r = NEAR_TIE_RECORD.setdefault(label, [rep.rows, rep.near_tie_rows, 0, 0])
    r[1] = max(r[1], rep.near_tie_rows)
    r[2] = max(r[2], rep.mismatched_rows)
    r[3] += 1


def near_tie_summary() -> list[str]:
    if not NEAR_TIE_RECORD:
        return []
    lines = ["near-tie record, full-size workloads (rows, near-tie rows, most mismatched "
             "rows over the runs, runs):"]
    worst = 0.0
    total_mis = 0
    for label, (rows, near, mis, runs) in sorted(NEAR_TIE_RECORD.items()):
        lines.append(f"  {label}: {rows} rows, {near} near-tie, {mis} mismatched, {runs} runs")
        worst = max(worst, mis / max(rows, 1))
        total_mis += mis
    lines.append(f"near ties: {len(NEAR_TIE_RECORD)} workloads, mismatched rows {total_mis} "
                 f"in all, largest mismatched fraction {worst:.2e} (bound {MAX_MISMATCH_FRAC:g}), "
                 f"near-tie rows {sum(r[1] for r in NEAR_TIE_RECORD.values())} in all")
    return lines


def compare_map(gpu_map: np.ndarray, ref_map: np.ndarray, near: np.ndarray) -> MapReport:
    gpu_map = np.asarray(gpu_map).astype(bool)
    diff = np.any(gpu_map != ref_map, axis=1)
    return MapReport(rows=int(ref_map.shape[0]), near_tie_rows=int(near.sum()),
                     mismatched_rows=int(diff.sum()),
                     mismatched_non_near=int((diff & ~near).sum()), ok_rows=~diff)


def max_violation(gpu: np.ndarray, ref: np.ndarray, dtype: str, rows=None) -> float:
    """Largest tolerance violation (<= 0 means every element passes)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    if gpu.size == 0:
        return 0.0
    if dtype == "bf16":
        rb = O.round_to_bf16(ref)
        return float(np.max(np.abs(gpu - rb) - (BF16_REL * np.abs(rb) + BF16_ABS)))
    return float(np.max(np.abs(gpu - ref) - F32_ABS))


def assert_close(gpu, ref, dtype, rows=None, what=""):
    v = max_violation(gpu, ref, dtype, rows)
    assert v <= 0.0, f"{what}: tolerance exceeded by {v:.3e}"


def bitwise_equal_fraction(gpu: np.ndarray, ref: np.ndarray) -> float:
    """Share of elements where the GPU value equals the oracle's value rounded
    to the GPU's float32 (reported beside the tolerance)."""
    g = np.asarray(gpu, dtype=np.float32)
    r = np.asarray(ref, dtype=np.float64).astype(np.float32)
    return float(np.mean(g.view(np.uint32) == r.view(np.uint32)))
