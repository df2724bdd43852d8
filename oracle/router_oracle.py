"""CPU oracle of the fused MoE router: plain, slow, float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module; only the test suite, the smoke check and the CPU-baseline leg of
the benchmark use it.  It shares no code with the CUDA library: it takes
float64 copies of the same inputs and recomputes every result from the
definitions, one token row at a time, with a full sort per row.

Sources (titles of the pages the method is read from):

* [TE]  NVIDIA TransformerEngine PR #3012, "[Common] Optimize fused router
  forward/backward kernels": Summary (the two fused ops), Changes/Hardening
  (argument rules), Performance (which tensors the forward reads and writes:
  logits, probs, routing_map and the fp32 intermediate output), the two full
  benchmark tables (softmax and sigmoid score functions), and the review
  summary (the backward's gradient across score function x pre-softmax).
* [ORT] microsoft/onnxruntime PR #33366, "[CUDA] Add fused decode routing,
  single-pass finalize, and PDL overlap for NVFP4 QMoE": Description item 1
  (softmax + top-k per row, one row per warp) and the review's parity request
  (tied logits).
* [AITER] ROCm/aiter PR #5652, "[HIP] [Perf] Fold shared-expert gate GEMV
  into topk_softmax kernel": the review's suggested benchmark (topk_softmax
  writing [T, K] weights, indices and token_expert_indices, with row-strided
  views for the weights and indices) and its note on the token_expert_indices
  width ([T, K]).
* [TRT] NVIDIA TensorRT-LLM PR #14592, "[TRTLLM-12214][perf] DeepGemmFusedMoE:
  fuse masked gather + finalize-scale into one Triton kernel": the
  reverse-permute map (expanded row t + k * num_rows).

Readings where the pages are silent (each one is also listed in the design
notes):

* softmax is taken over all E experts before the top-K choice (the
  pre-softmax order) and the selected probabilities are not renormalised;
* sigmoid probabilities are renormalised over the K selected experts with the
  unbiased scores: p_i = c * s_i / sum_sel s_j, with no epsilon;
* the post-softmax variant ("softmax_post", TransformerEngine's
  use_pre_softmax = false, onnxruntime's normalize_routing_weights) selects
  like softmax and renormalises the softmax over the K selected experts:
  p_i = c * s_i / sum_sel s_j (= c * softmax of the selected logits);
* the selection key is s_i + b_i (b = optional per-expert bias, selection
  only); ties go to the lower expert index, and -0.0 equals +0.0;
* group-limited selection: E splits into num_groups contiguous groups; a
  group's score is the sum of its K/group_topk largest keys; the group_topk
  best groups survive (ties to the lower group index); the top-K is then taken
  over the surviving experts.  num_groups = 0 means no grouping; the oracle
  runs the general grouped algorithm for every num_groups >= 1;
* the aux-loss score is q = softmax(x) for softmax and q = sigmoid(x) /
  sum_E sigmoid(x) for sigmoid; its routing map is the top-K of q with the same
  tie rule, without bias, groups or scaling; the sigmoid variant also saves
  sigmoid(x) for its backward.
"""
from __future__ import annotations

import numpy as np

SOFTMAX = "softmax"
SIGMOID = "sigmoid"
SOFTMAX_POST = "softmax_post"

# A row is a near tie when the keys on either side of its top-K boundary are
# distinct but within this relative distance of each other.
NEAR_TIE_REL = 1e-6


# --------------------------------------------------------------------------
# score function  [TE] Summary; the two benchmark tables (softmax, sigmoid)
# --------------------------------------------------------------------------
def score_row(x: np.ndarray, score_func: str) -> np.ndarray:
    """Per-expert score of one token row, in float64.

    softmax (and softmax_post): s_i = exp(x_i - max x) / sum_j exp(x_j - max x)
    over all E.
    sigmoid: s_i = 1 / (1 + exp(-x_i)).
    """
    x = np.asarray(x, dtype=np.float64)
    if score_func in (SOFTMAX, SOFTMAX_POST):
        e = np.exp(x - x.max())
        return e / e.sum()
    if score_func == SIGMOID:
        return 1.0 / (1.0 + np.exp(-x))
    raise ValueError(score_func)


# --------------------------------------------------------------------------
# ordering with the lower-index tie rule  [ORT] review: tied logits
# --------------------------------------------------------------------------
def order_desc(keys: np.ndarray) -> np.ndarray:
    """Indices of ``keys`` sorted by (key descending, index ascending).

    A stable sort of the negated keys keeps equal keys in ascending index
    order; the comparison is numeric, so -0.0 and +0.0 are equal.
    """
    return np.argsort(-np.asarray(keys, dtype=np.float64), kind="stable")


def group_scores(keys: np.ndarray, num_groups: int, per_group: int) -> np.ndarray:
    """Score of each contiguous expert group: the sum of its ``per_group``
    largest keys (a full sort of each group)."""
    E = keys.size
    eg = E // num_groups
    out = np.empty(num_groups, dtype=np.float64)
    for g in range(num_groups):
        kg = keys[g * eg:(g + 1) * eg]
        out[g] = kg[order_desc(kg)[:per_group]].sum()
    return out


def selectable_experts(keys: np.ndarray, K: int, num_groups: int,
                       group_topk: int) -> tuple[np.ndarray, np.ndarray | None]:
    """Experts the top-K may choose from, after group-limited pre-selection.

    Returns (boolean mask over E, group scores or None).  [TE] Hardening:
    K must be a multiple of group_topk.
    """
    E = keys.size
    if num_groups <= 0:
        return np.ones(E, dtype=bool), None
    per_group = K // group_topk
    gs = group_scores(keys, num_groups, per_group)
    kept = order_desc(gs)[:group_topk]
    eg = E // num_groups
    mask = np.zeros(E, dtype=bool)
    for g in kept:
        mask[g * eg:(g + 1) * eg] = True
    return mask, gs


# --------------------------------------------------------------------------
# near ties: the rows whose selection a float32 computation may legitimately
# decide differently.  Reading of the router's stated accuracy rule: the keys
# on either side of the top-K boundary (the K-th and (K+1)-th in the ranked
# order), or the scores on either side of the group boundary (the
# group_topk-th and (group_topk+1)-th group), are distinct and within 1e-6
# relative of each other.  Exact ties are not near ties: the lower-index rule
# decides them.
# --------------------------------------------------------------------------
def _near(a: float, b: float) -> bool:
    """Distinct, and within NEAR_TIE_REL relative of the larger magnitude."""
    d = abs(a - b)
    return 0.0 < d <= NEAR_TIE_REL * max(abs(a), abs(b))


def boundary_near_tie(ranked_keys: np.ndarray, K: int) -> bool:
    """The top-K boundary of one row: ``ranked_keys`` are the selectable keys
    in selection order (key descending, index ascending); the row is a near
    tie when its K-th and (K+1)-th keys are.  A row with no (K+1)-th
    selectable key has no boundary."""
    if K >= ranked_keys.size:
        return False
    return _near(ranked_keys[K - 1], ranked_keys[K])


def group_near_tie(gs: np.ndarray, group_topk: int) -> bool:
    """The group boundary of one grouped row: its group_topk-th and
    (group_topk+1)-th group scores in group order (score descending, group
    index ascending).  Keeping every group leaves no boundary."""
    if group_topk >= gs.size:
        return False
    ranked = gs[order_desc(gs)]
    return _near(ranked[group_topk - 1], ranked[group_topk])


# --------------------------------------------------------------------------
# router top-K forward  [TE] Summary, Performance
# --------------------------------------------------------------------------
def topk_fwd_row(x, K, score_func, num_groups=0, group_topk=0,
                 scaling_factor=1.0, expert_bias=None, ranked=False):
    """One token row of the top-K router forward.

    Returns (probs, routing_map, scores, near_tie) with probs and scores in
    float64 (not yet rounded to the output dtype); with ranked=True also the
    K selected experts in rank order (key descending, index ascending).
    """
    x = np.asarray(x, dtype=np.float64)
    E = x.size
    s = score_row(x, score_func)                                   # step 1
    b = (np.zeros(E) if expert_bias is None
         else np.asarray(expert_bias, dtype=np.float64))
    key = s + b                                                    # step 2
    allowed, gs = selectable_experts(key, K, num_groups, group_topk)  # step 3
    cand = np.nonzero(allowed)[0]
    order = cand[order_desc(key[cand])]                            # step 4
    sel = order[:K]
    m = np.zeros(E, dtype=bool)
    m[sel] = True

    if score_func == SOFTMAX:                                      # step 5
        probs = np.where(m, scaling_factor * s, 0.0)
    else:  # sigmoid, softmax_post: renormalised over the selected
        probs = np.where(m, scaling_factor * s / s[sel].sum(), 0.0)

    near = boundary_near_tie(key[order], K)                       # near ties
    if gs is not None:
        near = near or group_near_tie(gs, group_topk)
    if ranked:
        return probs, m, s, near, sel
    return probs, m, s, near


def topk_fwd(logits, K, score_func=SOFTMAX, num_groups=0, group_topk=0,
             scaling_factor=1.0, expert_bias=None):
    """Router top-K forward over all rows of ``logits`` [T, E].

    Returns a dict: probs [T,E] f64, routing_map [T,E] bool, scores [T,E] f64,
    near_tie [T] bool.
    """
    logits = np.asarray(logits, dtype=np.float64)
    T, E = logits.shape
    probs = np.zeros((T, E))
    rmap = np.zeros((T, E), dtype=bool)
    scores = np.zeros((T, E))
    near = np.zeros(T, dtype=bool)
    for t in range(T):
        probs[t], rmap[t], scores[t], near[t] = topk_fwd_row(
            logits[t], K, score_func, num_groups, group_topk, scaling_factor,
            expert_bias)
    return dict(probs=probs, routing_map=rmap, scores=scores, near_tie=near)


# --------------------------------------------------------------------------
# compact outputs  [AITER] review of the shared-expert topk_softmax fusion
# (the [T, K] weights / indices / token_expert_indices buffers, row-strided
# weights and indices); [TRT] reverse-permute map (the expanded row of token
# t's k-th choice is t + k * num_rows).  Reading: position k of a row holds
# the expert of rank k in the selection order (key descending, index
# ascending), with its probability as the weight.
# --------------------------------------------------------------------------
def topk_fwd_compact(logits, K, score_func=SOFTMAX, num_groups=0, group_topk=0,
                     scaling_factor=1.0, expert_bias=None):
    """Returns a dict: topk_weights [T,K] f64 (probs of the selected experts,
    not yet rounded), topk_indices [T,K] int64, token_expert_indices [T,K]
    int64 (k * T + t), near_tie [T] bool."""
    logits = np.asarray(logits, dtype=np.float64)
    T, E = logits.shape
    w = np.zeros((T, K))
    idx = np.zeros((T, K), dtype=np.int64)
    tei = np.zeros((T, K), dtype=np.int64)
    near = np.zeros(T, dtype=bool)
    for t in range(T):
        probs, _, _, near[t], sel = topk_fwd_row(
            logits[t], K, score_func, num_groups, group_topk, scaling_factor,
            expert_bias, ranked=True)
        for k in range(K):
            idx[t, k] = sel[k]
            w[t, k] = probs[sel[k]]
            tei[t, k] = k * T + t
    return dict(topk_weights=w, topk_indices=idx, token_expert_indices=tei, near_tie=near)


# --------------------------------------------------------------------------
# expert maps  [ORT] Description item 1 (the (expert, token)-sorted expert
# maps of the top-k choices) and the review's parity request (both row maps,
# the expert ids and the expert offsets); [TRT] reverse-permute map
# (permuted_row = unpermuted_to_permuted[t + k * num_rows]; the expert of a
# permuted row and its column permuted_row - expert_first_token_offset[e]).
# Reading: the T K choices are sorted by (expert ascending, token
# ascending); a token picks an expert at most once, so the order is unique.
# --------------------------------------------------------------------------
def expert_maps(topk_indices, E):
    """Returns a dict of int64 arrays from the [T, K] expert choices:
    expert_first_token_offset [E+1] (first permuted row of each expert; the
    last entry is T K), permuted_to_unpermuted [T K] (the expanded row
    t + k T of each permuted row), unpermuted_to_permuted [T K] (its
    inverse), permuted_experts [T K] (the expert of each permuted row)."""
    idx = np.asarray(topk_indices, dtype=np.int64)
    T, K = idx.shape
    choices = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K))
    n = T * K
    p2u = np.zeros(n, dtype=np.int64)
    u2p = np.zeros(n, dtype=np.int64)
    experts = np.zeros(n, dtype=np.int64)
    for p, (e, t, k) in enumerate(choices):
        p2u[p] = t + k * T
        u2p[t + k * T] = p
        experts[p] = e
    counts = np.zeros(E, dtype=np.int64)
    for e, _, _ in choices:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return dict(expert_first_token_offset=offsets, permuted_to_unpermuted=p2u,
                unpermuted_to_permuted=u2p, permuted_experts=experts)


# --------------------------------------------------------------------------
# router top-K backward  [TE] Backward kernels (two passes: row sums, then
# per-element gradients); review summary (gradient per score function)
# --------------------------------------------------------------------------
def topk_bwd_row(g, m, s, score_func, scaling_factor=1.0):
    """grad_logits of one row, from grad_probs g, the routing map m and the
    saved scores s.  The selection and the bias carry no gradient.

    softmax (p = c m s):       D = c sum_j m_j g_j s_j,  gx_j = s_j (c m_j g_j - D)
    sigmoid (p = c m s / S):   S = sum_j m_j s_j,  D = sum_j m_j g_j s_j,
                               gx_j = m_j (c / S) (g_j - D / S) s_j (1 - s_j)
    softmax_post (p = c m s / S with s the full softmax, i.e. c times the
                  softmax of the selected logits):
                               gx_j = m_j (c / S) (g_j - D / S) s_j
    """
    g = np.asarray(g, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    m = np.asarray(m, dtype=bool).astype(np.float64)
    c = float(scaling_factor)
    if score_func == SOFTMAX:
        D = c * np.sum(m * g * s)              # pass 1
        return s * (c * m * g - D)             # pass 2
    if score_func == SIGMOID:
        S = np.sum(m * s)                      # pass 1
        D = np.sum(m * g * s)
        return m * (c / S) * (g - D / S) * s * (1.0 - s)   # pass 2
    if score_func == SOFTMAX_POST:
        S = np.sum(m * s)                      # pass 1
        D = np.sum(m * g * s)
        return m * (c / S) * (g - D / S) * s               # pass 2
    raise ValueError(score_func)


def topk_bwd(grad_probs, routing_map, scores, score_func=SOFTMAX, scaling_factor=1.0):
    grad_probs = np.asarray(grad_probs, dtype=np.float64)
    out = np.zeros_like(grad_probs)
    for t in range(grad_probs.shape[0]):
        out[t] = topk_bwd_row(grad_probs[t], routing_map[t], scores[t], score_func,
                              scaling_factor)
    return out


# --------------------------------------------------------------------------
# aux-loss scores  [TE] Summary (fused_score_for_moe_aux_loss); the aux_loss
# rows of both benchmark tables
# --------------------------------------------------------------------------
def aux_scores_fwd_row(x, K, score_func):
    """Returns (q, routing_map, saved): q the aux-loss score row, the top-K
    map of q, and what the backward needs (sigmoid(x) for sigmoid, q itself
    for softmax)."""
    x = np.asarray(x, dtype=np.float64)
    if score_func == SOFTMAX:
        q = score_row(x, SOFTMAX)
        saved = q
    elif score_func == SIGMOID:
        sig = score_row(x, SIGMOID)
        q = sig / sig.sum()
        saved = sig
    else:
        raise ValueError(score_func)
    m = np.zeros(x.size, dtype=bool)
    m[order_desc(q)[:K]] = True
    return q, m, saved


def aux_scores_fwd(logits, K, score_func=SOFTMAX):
    logits = np.asarray(logits, dtype=np.float64)
    T, E = logits.shape
    q = np.zeros((T, E))
    m = np.zeros((T, E), dtype=bool)
    saved = np.zeros((T, E))
    near = np.zeros(T, dtype=bool)
    for t in range(T):
        q[t], m[t], saved[t] = aux_scores_fwd_row(logits[t], K, score_func)
        near[t] = boundary_near_tie(q[t][order_desc(q[t])], K)
    return dict(scores=q, routing_map=m, saved=saved, near_tie=near)


def aux_scores_bwd_row(g, saved, score_func):
    """grad_logits of one row from grad_scores g.

    softmax (saved = q):        gx_j = q_j (g_j - sum_i g_i q_i)
    sigmoid (saved = sigma):    Z = sum_i sigma_i, Dq = sum_i g_i sigma_i / Z,
                                gx_j = (g_j - Dq) / Z * sigma_j (1 - sigma_j)
    """
    g = np.asarray(g, dtype=np.float64)
    v = np.asarray(saved, dtype=np.float64)
    if score_func == SOFTMAX:
        return v * (g - np.sum(g * v))
    if score_func == SIGMOID:
        Z = v.sum()
        Dq = np.sum(g * v) / Z
        return (g - Dq) / Z * v * (1.0 - v)
    raise ValueError(score_func)


def aux_scores_bwd(grad_scores, saved, score_func=SOFTMAX):
    grad_scores = np.asarray(grad_scores, dtype=np.float64)
    out = np.zeros_like(grad_scores)
    for t in range(grad_scores.shape[0]):
        out[t] = aux_scores_bwd_row(grad_scores[t], saved[t], score_func)
    return out


# --------------------------------------------------------------------------
# load-balancing aux loss  [TE] Important Files Changed (fused_moe_aux_loss);
# the page names the op only.  Reading: the standard load-balancing loss,
# coeff * E * sum_e f_e * P_e with f_e = tokens_e / (T K) the share of the T K
# assignments routed to expert e and P_e = (1/T) sum_t q_te the mean aux score.
# --------------------------------------------------------------------------
def aux_loss_fwd(aux_scores, routing_map, K, coeff):
    """Returns (loss, tokens_per_expert[E]) from the aux scores q [T,E] and
    the routing map [T,E]: loss = coeff E / (K T^2) sum_e (sum_t q_te) tokens_e."""
    q = np.asarray(aux_scores, dtype=np.float64)
    m = np.asarray(routing_map).astype(bool)
    T, E = q.shape
    tokens = m.sum(axis=0).astype(np.int64)          # tokens routed to each expert
    colsum = q.sum(axis=0)                            # T * P_e
    loss = coeff * E / (K * T * T) * float(np.dot(colsum, tokens))
    return loss, tokens


def aux_loss_bwd(grad_loss, tokens_per_expert, T, K, coeff):
    """grad_scores [T,E]: the loss is linear in q, d loss / d q_te =
    coeff E / (K T^2) tokens_e; the counts carry no gradient."""
    tokens = np.asarray(tokens_per_expert, dtype=np.float64)
    E = tokens.size
    row = float(grad_loss) * coeff * E / (K * T * T) * tokens
    return np.tile(row, (T, 1))


# --------------------------------------------------------------------------
# output rounding
# --------------------------------------------------------------------------
def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 number (8 significant bits,
    ties to even), returned as float64.  Only normal-range values occur in the
    router's outputs; zeros stay zero."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, 0.5 <= |m| < 1
    r = np.round(m * 256.0) / 256.0         # np.round: halves go to even
    return np.ldexp(r, e)


def round_to_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
