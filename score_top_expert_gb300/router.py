"""Python binding of the router's C ABI (include/moe_router.h).

Argument marshalling only: every function checks tensor devices, dtypes and
shapes, allocates missing outputs with torch, passes raw device pointers and
the current torch stream to the library, and raises on a nonzero status.
All router arithmetic runs in the library's CUDA kernels; there is no other
implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MR_SOFTMAX, MR_SIGMOID, MR_SOFTMAX_POST = 0, 1, 2
MR_F32, MR_BF16 = 0, 1
MR_PATH_AUTO, MR_PATH_SEGMENT, MR_PATH_STAGED, MR_PATH_REGISTER = 0, 1, 2, 3
STATUS = {0: "MR_OK", -1: "MR_ERR_INVALID", -2: "MR_ERR_UNSUPPORTED", -3: "MR_ERR_CUDA"}

_SCORE = {"softmax": MR_SOFTMAX, "sigmoid": MR_SIGMOID, "softmax_post": MR_SOFTMAX_POST}
_DTYPE = {torch.float32: MR_F32, torch.bfloat16: MR_BF16}

_lib = None
_fast = None  # the CPython call shim, when built (same C entry points as ctypes)


class RouterError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = lib().moe_router_strerror(code).decode()
        super().__init__(f"{fn}: {STATUS.get(code, code)} ({msg})")


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"router CUDA library not built ({path} missing); run "
                "`python -m score_top_expert_gb300.build`")
        L = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.router_topk_fwd.argtypes = [vp, i, i, i, i, i, i, i, f, vp, vp, vp, vp, vp]
        L.router_topk_fwd_compact.argtypes = [vp, i, i, i, i, i, i, i, f, vp, vp, i, vp, i, vp,
                                              vp, vp, vp, vp]
        L.router_expert_maps_workspace_bytes.argtypes = [i, i]
        L.router_expert_maps_workspace_bytes.restype = ctypes.c_size_t
        L.router_expert_maps.argtypes = [vp, i, i, i, i, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                         vp]
        L.router_topk_fwd_maps.argtypes = [vp, i, i, i, i, i, i, i, f, vp, vp, i, vp, i, vp, vp,
                                           vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.router_topk_bwd.argtypes = [vp, vp, vp, i, i, i, i, i, f, vp, vp]
        L.router_aux_scores_fwd.argtypes = [vp, i, i, i, i, i, vp, vp, vp, vp]
        L.router_aux_scores_bwd.argtypes = [vp, vp, i, i, i, i, i, vp, vp]
        for fn in ("router_topk_fwd", "router_topk_fwd_compact", "router_topk_fwd_maps",
                   "router_expert_maps", "router_topk_bwd",
                   "router_aux_scores_fwd",
                   "router_aux_scores_bwd", "moe_router_force_path",
                   "moe_router_force_fwd_lanes", "moe_router_version",
                   "moe_router_device_status"):
            getattr(L, fn).restype = ctypes.c_int
        L.moe_router_force_path.argtypes = [i]
        L.moe_router_force_fwd_lanes.argtypes = [i]
        L.moe_router_version.argtypes = []
        L.moe_router_device_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
        L.moe_router_selftest_bounded_wait.argtypes = [ctypes.c_uint, vp]
        L.router_aux_loss_workspace_bytes.argtypes = [i, i]
        L.router_aux_loss_workspace_bytes.restype = ctypes.c_size_t
        L.router_aux_loss_fwd.argtypes = [vp, vp, i, i, i, f, vp, vp, vp, ctypes.c_size_t, vp]
        L.router_aux_loss_fwd.restype = ctypes.c_int
        L.router_aux_loss_fwd_noalloc.argtypes = [vp, vp, i, i, i, f, vp, vp, vp]
        L.router_aux_loss_fwd_noalloc.restype = ctypes.c_int
        L.router_aux_loss_bwd.argtypes = [vp, vp, i, i, i, f, vp, vp]
        L.router_aux_loss_bwd.restype = ctypes.c_int
        L.moe_router_selftest_bounded_wait.restype = ctypes.c_int
        L.moe_router_strerror.argtypes = [i]
        L.moe_router_strerror.restype = ctypes.c_char_p
        _lib = L
        _load_fast()
    return _lib


class _CtypesCalls:
    """The hot calls through ctypes (pointers as integers, 0 for NULL), for
    an interpreter without headers to build the CPython shim."""

    def __init__(self, L):
        self.router_topk_fwd = L.router_topk_fwd
        self.router_topk_bwd = L.router_topk_bwd
        self.router_aux_scores_fwd = L.router_aux_scores_fwd
        self.router_aux_scores_bwd = L.router_aux_scores_bwd


def _load_fast():
    """Bind the hot calls: the CPython shim built next to the library, else
    ctypes.  Both call the same exported C entry points."""
    global _fast
    path = _build.PYCALLS
    if os.path.exists(path):
        import importlib.util
        spec = importlib.util.spec_from_file_location("_pycalls", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        _fast = mod
    else:
        _fast = _CtypesCalls(_lib)


def _calls():
    if _fast is None:
        lib()
    return _fast


# The per-call path is kept lean for decode-sized calls, where the host cost
# of a call is most of its latency: pointers go to ctypes as plain integers
# (the argtypes convert them), the stream as the raw handle of torch's current
# stream, and devices as indices.
try:
    _raw_stream = torch._C._cuda_getCurrentRawStream
    _cur_dev = torch._C._cuda_getDevice
except AttributeError:  # pragma: no cover - older torch
    def _raw_stream(i):
        return torch.cuda.current_stream(i).cuda_stream

    _cur_dev = torch.cuda.current_device


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _ptr0(t: torch.Tensor | None) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(device) -> int:
    """Raw handle of torch's current stream on ``device`` (a torch.device or
    an index)."""
    return _raw_stream(device if isinstance(device, int) else device.index)


class _NoSwitch:
    def __enter__(self):
        return None

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _on(device):
    """Make ``device`` (a torch.device or an index) current for the library
    call; no switch (and none of its cost) when it already is."""
    idx = device if isinstance(device, int) else device.index
    if idx is None or idx == _cur_dev():
        return _NO_SWITCH
    return torch.cuda.device(idx)


def _check(fn: str, code: int):
    if code != 0:
        raise RouterError(fn, code)


def _as_input(t: torch.Tensor, name: str, dtypes) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} dtype {t.dtype} not in {dtypes}")
    if t.dim() != 2:
        raise ValueError(f"{name} must be [T, E]")
    return t if t.is_contiguous() else t.contiguous()


def _score(score_func: str) -> int:
    try:
        return _SCORE[score_func]
    except KeyError:
        raise ValueError(f"score_func must be one of {list(_SCORE)}") from None


def _out(t, shape, dtype, device, name):
    """A caller's output tensor, checked (shape, dtype, contiguity, device),
    or a new one.  ``device``: a torch.device with an index."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if t.shape != shape or t.dtype != dtype or not t.is_contiguous() \
            or t.get_device() != device.index:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {shape} on "
                         f"{device}")
    return t


def router_topk_fwd(logits: torch.Tensor, K: int, score_func: str = "softmax",
                    num_groups: int = 0, group_topk: int = 0, scaling_factor: float = 1.0,
                    expert_bias: torch.Tensor | None = None, *, probs=None,
                    routing_map=None, scores=None):
    """Top-K router forward.  Returns (probs [T,E] logits dtype,
    routing_map [T,E] bool, scores [T,E] float32)."""
    logits = _as_input(logits, "logits", _DTYPE)
    shape = logits.shape
    T, E = shape
    dev = logits.device
    dt = logits.dtype
    if expert_bias is not None:
        if expert_bias.dtype != torch.float32 or expert_bias.numel() != E \
                or expert_bias.get_device() != dev.index:
            raise ValueError("expert_bias must be a float32 [E] tensor on the logits' device")
        expert_bias = expert_bias.contiguous()
    probs = _out(probs, shape, dt, dev, "probs")
    routing_map = _out(routing_map, shape, torch.bool, dev, "routing_map")
    scores = _out(scores, shape, torch.float32, dev, "scores")
    with _on(dev):
        rc = _calls().router_topk_fwd(logits.data_ptr(), _DTYPE[dt], T, E, int(K),
                                      _score(score_func), int(num_groups), int(group_topk),
                                      float(scaling_factor), _ptr0(expert_bias),
                                      probs.data_ptr(), routing_map.data_ptr(),
                                      scores.data_ptr(), _stream(dev))
    _check("router_topk_fwd", rc)
    return probs, routing_map, scores


def _rows_out(t, T, K, dtype, device, name):
    """A [T, >= K] output addressed by row stride (unit column stride): a
    column view of a wider buffer is written in place."""
    if t is None:
        return torch.empty((T, K), dtype=dtype, device=device)
    if t.dim() != 2 or t.shape[0] != T or t.shape[1] < K or t.dtype != dtype \
            or t.get_device() != device.index or (T > 1 and t.stride(1) != 1) \
            or t.stride(0) < K:
        raise ValueError(f"{name} must be a {dtype} [T, >= K] tensor with unit column "
                         f"stride and row stride >= K")
    return t


def router_topk_fwd_compact(logits: torch.Tensor, K: int, score_func: str = "softmax",
                            num_groups: int = 0, group_topk: int = 0,
                            scaling_factor: float = 1.0,
                            expert_bias: torch.Tensor | None = None, *, topk_weights=None,
                            topk_indices=None, token_expert_indices=True, dense=False,
                            probs=None, routing_map=None, scores=None):
    """Top-K router forward with compact outputs.  Returns (topk_weights
    [T,K] float32, topk_indices [T,K] int32, token_expert_indices [T,K] int32
    or None, probs, routing_map, scores); row t, column k holds the expert of
    rank k (selection key descending, index ascending).  topk_weights and
    topk_indices may be column views of wider buffers (written in place).
    token_expert_indices: True to allocate, False/None to skip, or a
    contiguous [T,K] int32 tensor.  The dense outputs are None unless
    dense=True or given."""
    logits = _as_input(logits, "logits", _DTYPE)
    T, E = logits.shape
    dev = logits.device
    K = int(K)
    if expert_bias is not None:
        if expert_bias.dtype != torch.float32 or expert_bias.numel() != E \
                or expert_bias.get_device() != dev.index:
            raise ValueError("expert_bias must be a float32 [E] tensor on the logits' device")
        expert_bias = expert_bias.contiguous()
    topk_weights = _rows_out(topk_weights, T, K, torch.float32, dev, "topk_weights")
    topk_indices = _rows_out(topk_indices, T, K, torch.int32, dev, "topk_indices")
    if token_expert_indices is True:
        token_expert_indices = torch.empty((T, K), dtype=torch.int32, device=dev)
    elif token_expert_indices is False:
        token_expert_indices = None
    elif token_expert_indices is not None:
        token_expert_indices = _out(token_expert_indices, (T, K), torch.int32, dev,
                                    "token_expert_indices")
    if dense or probs is not None:
        probs = _out(probs, (T, E), logits.dtype, dev, "probs")
    if dense or routing_map is not None:
        routing_map = _out(routing_map, (T, E), torch.bool, dev, "routing_map")
    if dense or scores is not None:
        scores = _out(scores, (T, E), torch.float32, dev, "scores")
    ld_w = topk_weights.stride(0) if T > 0 else K
    ld_i = topk_indices.stride(0) if T > 0 else K
    with _on(dev):
        rc = lib().router_topk_fwd_compact(
            _ptr(logits), _DTYPE[logits.dtype], T, E, K, _score(score_func), int(num_groups),
            int(group_topk), float(scaling_factor), _ptr(expert_bias), _ptr(topk_weights),
            ld_w, _ptr(topk_indices), ld_i, _ptr(token_expert_indices), _ptr(probs),
            _ptr(routing_map), _ptr(scores), _stream(dev))
    _check("router_topk_fwd_compact", rc)
    return topk_weights, topk_indices, token_expert_indices, probs, routing_map, scores


def _maps_outputs(T, E, K, dev, out):
    n = T * K
    names = ("expert_first_token_offset", "permuted_to_unpermuted", "unpermuted_to_permuted",
             "permuted_experts")
    shapes = ((E + 1,), (n,), (n,), (n,))
    out = out or {}
    return tuple(_out(out.get(nm), sh, torch.int32, dev, nm) for nm, sh in zip(names, shapes))


def _workspace(nbytes, workspace, dev):
    if workspace is None:
        return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    return workspace


def router_expert_maps(topk_indices: torch.Tensor, E: int, *, out=None, workspace=None):
    """(expert, token)-sorted maps of [T, K] expert choices (int32, unit
    column stride; a column view of a wider buffer is fine).  Returns
    (expert_first_token_offset [E+1], permuted_to_unpermuted [T K],
    unpermuted_to_permuted [T K], permuted_experts [T K]), all int32; the
    choice (t, k) is the expanded row t + k T.  ``out`` may hold any of the
    four by name; the workspace is allocated here when not given."""
    if not topk_indices.is_cuda or topk_indices.dtype != torch.int32 or topk_indices.dim() != 2:
        raise ValueError("topk_indices must be a CUDA int32 [T, K] tensor")
    T, K = topk_indices.shape
    if T > 1 and topk_indices.stride(1) != 1:
        raise ValueError("topk_indices needs a unit column stride")
    dev = topk_indices.device
    ld = topk_indices.stride(0) if T > 0 else K
    offsets, p2u, u2p, pexp = _maps_outputs(T, int(E), K, dev, out)
    workspace = _workspace(lib().router_expert_maps_workspace_bytes(T, int(E)), workspace, dev)
    with _on(dev):
        rc = lib().router_expert_maps(_ptr(topk_indices), ld, T, int(E), K, _ptr(offsets),
                                      _ptr(p2u), _ptr(u2p), _ptr(pexp), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(dev))
    _check("router_expert_maps", rc)
    return offsets, p2u, u2p, pexp


def router_topk_fwd_maps(logits: torch.Tensor, K: int, score_func: str = "softmax",
                         num_groups: int = 0, group_topk: int = 0, scaling_factor: float = 1.0,
                         expert_bias: torch.Tensor | None = None, *, topk_weights=None,
                         topk_indices=None, token_expert_indices=True, out=None,
                         workspace=None):
    """Compact router forward plus the expert maps of its choices (one
    launch for up to 8 aligned tokens).  Returns (topk_weights, topk_indices,
    token_expert_indices or None, expert_first_token_offset,
    permuted_to_unpermuted, unpermuted_to_permuted, permuted_experts)."""
    logits = _as_input(logits, "logits", _DTYPE)
    T, E = logits.shape
    dev = logits.device
    K = int(K)
    if expert_bias is not None:
        if expert_bias.dtype != torch.float32 or expert_bias.numel() != E \
                or expert_bias.get_device() != dev.index:
            raise ValueError("expert_bias must be a float32 [E] tensor on the logits' device")
        expert_bias = expert_bias.contiguous()
    topk_weights = _rows_out(topk_weights, T, K, torch.float32, dev, "topk_weights")
    topk_indices = _rows_out(topk_indices, T, K, torch.int32, dev, "topk_indices")
    if token_expert_indices is True:
        token_expert_indices = torch.empty((T, K), dtype=torch.int32, device=dev)
    elif token_expert_indices is False:
        token_expert_indices = None
    elif token_expert_indices is not None:
        token_expert_indices = _out(token_expert_indices, (T, K), torch.int32, dev,
                                    "token_expert_indices")
    offsets, p2u, u2p, pexp = _maps_outputs(T, E, K, dev, out)
    workspace = _workspace(lib().router_expert_maps_workspace_bytes(T, E), workspace, dev)
    ld_w = topk_weights.stride(0) if T > 0 else K
    ld_i = topk_indices.stride(0) if T > 0 else K
    with _on(dev):
        rc = lib().router_topk_fwd_maps(
            _ptr(logits), _DTYPE[logits.dtype], T, E, K, _score(score_func), int(num_groups),
            int(group_topk), float(scaling_factor), _ptr(expert_bias), _ptr(topk_weights), ld_w,
            _ptr(topk_indices), ld_i, _ptr(token_expert_indices), _ptr(offsets), _ptr(p2u),
            _ptr(u2p), _ptr(pexp), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(dev))
    _check("router_topk_fwd_maps", rc)
    return topk_weights, topk_indices, token_expert_indices, offsets, p2u, u2p, pexp


def router_topk_bwd(grad_probs: torch.Tensor, routing_map: torch.Tensor,
                    scores: torch.Tensor, K: int, score_func: str = "softmax",
                    scaling_factor: float = 1.0, *, grad_logits=None):
    """Top-K router backward.  Returns grad_logits [T,E] in grad_probs' dtype."""
    grad_probs = _as_input(grad_probs, "grad_probs", _DTYPE)
    routing_map = _as_input(routing_map, "routing_map", (torch.bool, torch.uint8))
    scores = _as_input(scores, "scores", (torch.float32,))
    T, E = grad_probs.shape
    if routing_map.shape != grad_probs.shape or scores.shape != grad_probs.shape:
        raise ValueError("grad_probs, routing_map and scores must have the same shape")
    dev = grad_probs.device
    grad_logits = _out(grad_logits, (T, E), grad_probs.dtype, dev, "grad_logits")
    with _on(dev):
        rc = _calls().router_topk_bwd(grad_probs.data_ptr(), routing_map.data_ptr(),
                                      scores.data_ptr(), _DTYPE[grad_probs.dtype], T, E, int(K),
                                      _score(score_func), float(scaling_factor),
                                      grad_logits.data_ptr(), _stream(dev))
    _check("router_topk_bwd", rc)
    return grad_logits


def router_aux_scores_fwd(logits: torch.Tensor, K: int, score_func: str = "softmax", *,
                          scores=None, routing_map=None, intermediate=None):
    """Aux-loss scores forward.  Returns (scores q [T,E] float32,
    routing_map [T,E] bool, intermediate [T,E] float32: sigmoid(x) for sigmoid,
    q for softmax)."""
    logits = _as_input(logits, "logits", _DTYPE)
    T, E = logits.shape
    dev = logits.device
    scores = _out(scores, (T, E), torch.float32, dev, "scores")
    routing_map = _out(routing_map, (T, E), torch.bool, dev, "routing_map")
    if score_func == "sigmoid" or intermediate is not None:
        intermediate = _out(intermediate, (T, E), torch.float32, dev, "intermediate")
    with _on(dev):
        rc = _calls().router_aux_scores_fwd(logits.data_ptr(), _DTYPE[logits.dtype], T, E,
                                            int(K), _score(score_func), scores.data_ptr(),
                                            routing_map.data_ptr(), _ptr0(intermediate),
                                            _stream(dev))
    _check("router_aux_scores_fwd", rc)
    return scores, routing_map, (intermediate if intermediate is not None else scores)


def router_aux_scores_bwd(grad_scores: torch.Tensor, saved: torch.Tensor, K: int,
                          score_func: str = "softmax", dtype: torch.dtype = torch.float32,
                          *, grad_logits=None):
    """Aux-loss scores backward.  ``saved`` is the forward's scores (softmax)
    or intermediate (sigmoid).  Returns grad_logits [T,E] in ``dtype``."""
    grad_scores = _as_input(grad_scores, "grad_scores", (torch.float32,))
    saved = _as_input(saved, "saved", (torch.float32,))
    if saved.shape != grad_scores.shape:
        raise ValueError("grad_scores and saved must have the same shape")
    if dtype not in _DTYPE:
        raise ValueError(f"dtype must be one of {list(_DTYPE)}")
    T, E = grad_scores.shape
    dev = grad_scores.device
    grad_logits = _out(grad_logits, (T, E), dtype, dev, "grad_logits")
    with _on(dev):
        rc = _calls().router_aux_scores_bwd(grad_scores.data_ptr(), saved.data_ptr(),
                                            _DTYPE[dtype], T, E, int(K), _score(score_func),
                                            grad_logits.data_ptr(), _stream(dev))
    _check("router_aux_scores_bwd", rc)
    return grad_logits


def force_path(path: str) -> str:
    """Force the forward kernel path: 'auto', 'segment', 'staged' or 'register';
    returns the previous one."""
    names = {"auto": MR_PATH_AUTO, "segment": MR_PATH_SEGMENT, "staged": MR_PATH_STAGED,
             "register": MR_PATH_REGISTER}
    prev = lib().moe_router_force_path(names[path])
    if prev < 0:
        raise RouterError("moe_router_force_path", prev)
    return {v: k for k, v in names.items()}[prev]


def force_fwd_lanes(lanes: int) -> int:
    """Force the lanes per row of the segment forward (0 = automatic)."""
    prev = lib().moe_router_force_fwd_lanes(int(lanes))
    if prev < 0:
        raise RouterError("moe_router_force_fwd_lanes", prev)
    return prev


def device_status() -> int:
    """Read and clear the current device's status word (0 = no kernel gave
    up a bounded wait).  Synchronous."""
    v = ctypes.c_int(0)
    _check("moe_router_device_status", lib().moe_router_device_status(ctypes.byref(v)))
    return v.value


def selftest_bounded_wait(timeout_us: int, device=None) -> None:
    """Enqueue the diagnostic kernel whose bounded wait always runs out (see
    moe_router_selftest_bounded_wait in the header)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with _on(dev):
        _check("moe_router_selftest_bounded_wait",
               lib().moe_router_selftest_bounded_wait(int(timeout_us), _stream(dev)))


def router_aux_loss_fwd(aux_scores: torch.Tensor, routing_map: torch.Tensor, K: int,
                        coeff: float, *, loss=None, tokens_per_expert=None, workspace=None):
    """Load-balancing aux loss.  Returns (loss [1] float32, tokens_per_expert
    [E] int32).  The workspace (a uint8 CUDA tensor) is allocated here when
    not given."""
    aux_scores = _as_input(aux_scores, "aux_scores", (torch.float32,))
    routing_map = _as_input(routing_map, "routing_map", (torch.bool, torch.uint8))
    if routing_map.shape != aux_scores.shape:
        raise ValueError("aux_scores and routing_map must have the same shape")
    T, E = aux_scores.shape
    dev = aux_scores.device
    loss = _out(loss, (1,), torch.float32, dev, "loss")
    tokens_per_expert = _out(tokens_per_expert, (E,), torch.int32, dev, "tokens_per_expert")
    nbytes = lib().router_aux_loss_workspace_bytes(T, E)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    with _on(dev):
        rc = lib().router_aux_loss_fwd(_ptr(aux_scores), _ptr(routing_map), T, E, int(K),
                                       float(coeff), _ptr(loss), _ptr(tokens_per_expert),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(dev))
    _check("router_aux_loss_fwd", rc)
    return loss, tokens_per_expert


def router_aux_loss_fwd_noalloc(aux_scores: torch.Tensor, routing_map: torch.Tensor, K: int,
                                coeff: float, *, loss: torch.Tensor,
                                tokens_per_expert: torch.Tensor):
    """router_aux_loss_fwd for callers that cannot allocate device memory at
    the call: the library keeps its scratch in a fixed device array, and the
    caller passes the outputs (loss [1] float32, tokens_per_expert [E] int32)
    already allocated.  Calls that overlap on the GPU race on that array; the
    first call on a device looks up its address and belongs before any stream
    capture."""
    aux_scores = _as_input(aux_scores, "aux_scores", (torch.float32,))
    routing_map = _as_input(routing_map, "routing_map", (torch.bool, torch.uint8))
    if routing_map.shape != aux_scores.shape:
        raise ValueError("aux_scores and routing_map must have the same shape")
    T, E = aux_scores.shape
    dev = aux_scores.device
    if loss.get_device() != dev.index or loss.dtype != torch.float32 or loss.numel() < 1:
        raise ValueError("loss must be a float32 tensor on the inputs' device")
    if (tokens_per_expert.get_device() != dev.index or tokens_per_expert.dtype != torch.int32
            or tokens_per_expert.numel() != E or not tokens_per_expert.is_contiguous()):
        raise ValueError("tokens_per_expert must be a contiguous int32 [E] tensor on the "
                         "inputs' device")
    with _on(dev):
        rc = lib().router_aux_loss_fwd_noalloc(_ptr(aux_scores), _ptr(routing_map), T, E, int(K),
                                               float(coeff), _ptr(loss),
                                               _ptr(tokens_per_expert), _stream(dev))
    _check("router_aux_loss_fwd_noalloc", rc)
    return loss, tokens_per_expert


def router_aux_loss_bwd(grad_loss: torch.Tensor, tokens_per_expert: torch.Tensor, T: int, K: int,
                        coeff: float, *, grad_aux_scores=None):
    """Gradient of the aux loss with respect to the aux scores, [T, E] float32."""
    if not grad_loss.is_cuda or grad_loss.dtype != torch.float32 or grad_loss.numel() != 1:
        raise ValueError("grad_loss must be a CUDA float32 tensor with one element")
    if not tokens_per_expert.is_cuda or tokens_per_expert.dtype != torch.int32:
        raise ValueError("tokens_per_expert must be a CUDA int32 tensor")
    E = tokens_per_expert.numel()
    dev = tokens_per_expert.device
    grad_loss = grad_loss.contiguous()
    tokens_per_expert = tokens_per_expert.contiguous()
    grad_aux_scores = _out(grad_aux_scores, (T, E), torch.float32, dev, "grad_aux_scores")
    with _on(dev):
        rc = lib().router_aux_loss_bwd(_ptr(grad_loss), _ptr(tokens_per_expert), int(T), E, int(K),
                                       float(coeff), _ptr(grad_aux_scores), _stream(dev))
    _check("router_aux_loss_bwd", rc)
    return grad_aux_scores
