"""Batched verification of speculative-decoding drafts on an NVIDIA GB300.

Thin Python binding over the C ABI of ``libspecverify.so`` (declared in
``include/spec_verify.h``).  Every function here only marshals arguments:
it checks tensor devices, dtypes and layouts, allocates the outputs and the
workspace with PyTorch (device memory only), and calls the library on the
current CUDA stream.  All computation runs in the library's sm_103a
kernels; there is no CPU or PyTorch fallback.  Importing the package does
not load the library; the first call does, and raises if it is missing.

Inputs and outputs may be CUDA tensors or pinned host tensors
(``tensor.pin_memory()``): the kernels read pinned host arrays in place over
the CPU-GPU link, so a call on host-resident logits moves only the rows it
reads (rows past a rejection stay on the host).  Outputs that the call
allocates, and the workspace, are on the current CUDA device.

Functions (same names as the C entry points, without the ``spec_`` prefix):
  verify_chain   chain speculative sampling (accept min(1,p/q), residual, bonus)
  verify_greedy  greedy argmax-match verification
  tree_build     DDTree best-first tree under a node budget
  verify_tree    greedy tree-walk verification
  verify_tree_sample  stochastic tree-walk verification (target draws along the tree)
  kv_compact     keep the accepted path's KV rows
  adaptive_len   DSpark survival, expected advance and verify length
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libspecverify.so")

SPEC_F32, SPEC_BF16 = 0, 1
ST_BAD_ROW, ST_Q_ZERO, ST_R_ZERO, ST_BAD_TOKEN, ST_BAD_K = 1, 2, 4, 8, 16
WS_ERR_WAIT, WS_ERR_QUEUE = 1, 2

_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile libspecverify.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise SpecError(f"{LIB_PATH} is missing: build it with "
                            "speculative_decoding_draft_sampling_gb300.build() first")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.spec_last_error.restype = ctypes.c_char_p
        lib.spec_version.restype = ctypes.c_int
        lib.spec_set_tuning.argtypes = [i32, i32]
        lib.spec_workspace_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.spec_verify_chain_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.spec_verify_chain_workspace_size.restype = sz
        lib.spec_verify_chain.argtypes = [P, i32, i64, i64, P, i64, i64, P, P, i32, i32, i32, f32, i32,
                                          P, P, P, P, P, P, P, P, sz, P]
        lib.spec_verify_greedy_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_verify_greedy_workspace_size.restype = sz
        lib.spec_verify_greedy.argtypes = [P, i32, i64, i64, P, i32, i32, i32, P, P, P, P, P, P, sz, P]
        lib.spec_tree_build_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.spec_tree_build_workspace_size.restype = sz
        lib.spec_tree_build.argtypes = [P, i64, i64, i32, i32, i32, i32, P, P, P, P, P, P, P, P, sz, P]
        lib.spec_eagle_expand_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_eagle_expand_workspace_size.restype = sz
        lib.spec_eagle_expand.argtypes = [P, i64, i64, i32, i32, i32, i32, i32, i32,
                                          P, P, P, P, P, P, P, P, P, P, P, sz, P]
        lib.spec_eagle_rerank.argtypes = [P, P, P, P, P, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.spec_verify_tree_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_verify_tree_workspace_size.restype = sz
        lib.spec_verify_tree.argtypes = [P, i32, i64, i64, P, P, P, i32, i32, i32, i32, P, P, P, P, P, sz, P]
        lib.spec_adaptive_len.argtypes = [P, i32, i32, f32, f32, P, P, P, P, P, P]
        lib.spec_adaptive_len_table.argtypes = [P, i32, i32, P, P, P, P, P, P, P]
        lib.spec_kv_compact.argtypes = [P, i64, i64, i64, P, i64, i64, i64, i32, i32, i32, i64, P, i32, P, P, P]
        lib.spec_kv_compact.restype = ctypes.c_int
        lib.spec_adaptive_len_table.restype = ctypes.c_int
        lib.spec_verify_tree_sample_workspace_size.argtypes = [i32, i32, i32]
        lib.spec_verify_tree_sample_workspace_size.restype = sz
        lib.spec_verify_tree_sample.argtypes = [P, i32, i64, i64, P, P, P, P, i32, i32, i32, i32, f32, i32,
                                                P, P, P, P, P, sz, P]
        for name in ("spec_set_tuning", "spec_workspace_error", "spec_verify_chain", "spec_verify_greedy",
                     "spec_tree_build", "spec_verify_tree", "spec_adaptive_len", "spec_verify_tree_sample"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def lib():
    """The loaded ctypes library (loads it on first use)."""
    return _load()


def _check(rc: int, what: str):
    if rc != 0:
        msg = _load().spec_last_error().decode(errors="replace")
        raise SpecError(f"{what} failed (status {rc}): {msg}")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str, dtype=None):
    """A CUDA tensor, or a pinned host tensor that the kernels read (or write)
    in place through its device mapping."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
        raise SpecError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if dtype is not None and t.dtype != dtype:
        raise SpecError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dev(t: torch.Tensor) -> torch.device:
    """The CUDA device a call on t runs on (the current one for host tensors)."""
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _ldt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise SpecError(f"logits must be float32 or bfloat16, got {t.dtype}")


_ws_cache: dict = {}


def workspace(nbytes: int, device) -> torch.Tensor:
    """A cached device scratch buffer of at least ``nbytes`` bytes (one per
    device); calls on one stream may share it, concurrent calls must not."""
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 12), dtype=torch.uint8, device=torch.device("cuda", key))
        _ws_cache[key] = buf
    return buf


def set_tuning(slices_per_row: int = 0, slots_per_cta: int = 0):
    """CTAs per cluster (one row slice each) and requests in flight per CTA;
    0 = automatic.  For benchmarking sweeps."""
    _check(_load().spec_set_tuning(int(slices_per_row), int(slots_per_cta)), "spec_set_tuning")


def workspace_error(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(_load().spec_workspace_error(_p(ws), _stream(stream), ctypes.byref(v)), "spec_workspace_error")
    return int(v.value)


def version() -> int:
    return int(_load().spec_version())


# ---------------------------------------------------------------------------
# chain speculative sampling
# ---------------------------------------------------------------------------
@dataclass
class ChainResult:
    tokens: torch.Tensor        # [B, K+1] int32
    num_accepted: torch.Tensor  # [B] int32
    status: torch.Tensor        # [B] int32
    diag: Optional[torch.Tensor]
    ws: torch.Tensor


def verify_chain(logits, q, draft, uniforms, temperature: float, top_k: int = 0, *,
                 k_per_req=None, l_row_off=None, q_row_off=None, diag: bool = False,
                 out: Optional[ChainResult] = None, ws: Optional[torch.Tensor] = None,
                 stream=None) -> ChainResult:
    """Chain speculative sampling.

    Dense: logits [B, K+1, V], q [B, K, V] (any batch/row strides, unit
    element stride); with k_per_req alone each request verifies only its
    first k_b positions ("cap-accept").  Packed ("compact", k_per_req with
    l_row_off and q_row_off): logits [rows, V] packed by l_row_off, q
    [rows, V] packed by q_row_off.  draft [B, K] int32, uniforms [B, K+1]
    fp32.
    """
    L = _load()
    _cuda(logits, "logits")
    ldt = _ldt(logits)
    _cuda(q, "q", torch.float32)
    _cuda(draft, "draft", torch.int32)
    _cuda(uniforms, "uniforms", torch.float32)
    if draft.dim() != 2 or not draft.is_contiguous() or not uniforms.is_contiguous():
        raise SpecError("draft [B, K] and uniforms [B, K+1] must be contiguous")
    B, K = draft.shape
    V = logits.shape[-1]
    if uniforms.shape != (B, K + 1):
        raise SpecError("uniforms must be [B, K+1]")
    if logits.stride(-1) != 1 or q.stride(-1) != 1:
        raise SpecError("logits and q need unit element stride")
    packed = l_row_off is not None
    if k_per_req is not None:
        _cuda(k_per_req, "k_per_req", torch.int32)
    if packed:
        if k_per_req is None or q_row_off is None:
            raise SpecError("packed rows need k_per_req, l_row_off and q_row_off")
        for t, n in ((l_row_off, "l_row_off"), (q_row_off, "q_row_off")):
            _cuda(t, n, torch.int32)
        if logits.dim() != 2 or q.dim() != 2:
            raise SpecError("packed ('compact') mode takes packed 2-D logits and q")
        lbs, lrs = 0, logits.stride(0)
        qbs, qrs = 0, q.stride(0)
    else:
        # dense rows: every request verifies K positions, or with k_per_req
        # only its first k_b ("cap-accept")
        if logits.dim() != 3 or logits.shape[:2] != (B, K + 1):
            raise SpecError("dense logits must be [B, K+1, V]")
        if q.dim() != 3 or q.shape[0] != B or q.shape[1] < K or q.shape[2] != V:
            raise SpecError("dense q must be [B, K, V]")
        lbs, lrs = logits.stride(0), logits.stride(1)
        qbs, qrs = q.stride(0), q.stride(1)
    dev = _dev(logits)
    if out is None:
        out = ChainResult(torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                          torch.empty(B, dtype=torch.int32, device=dev),
                          torch.empty(B, dtype=torch.int32, device=dev),
                          torch.full((B, K + 1, 4), float("nan"), dtype=torch.float32, device=dev) if diag else None,
                          None)
    need = L.spec_verify_chain_workspace_size(B, K, V, int(top_k))
    if ws is None and out.ws is not None and out.ws.numel() >= need and out.ws.device == dev:
        ws = out.ws   # a reused result keeps its workspace (and the filter hint kept in it)
    if ws is None:
        ws = workspace(need, dev)
    out.ws = ws
    rc = L.spec_verify_chain(_p(logits), ldt, lbs, lrs, _p(q), qbs, qrs, _p(draft), _p(uniforms),
                             B, K, V, float(temperature), int(top_k),
                             _p(k_per_req), _p(l_row_off), _p(q_row_off),
                             _p(out.tokens), _p(out.num_accepted), _p(out.status), _p(out.diag),
                             _p(ws), ws.numel(), _stream(stream))
    _check(rc, "spec_verify_chain")
    return out


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------
@dataclass
class GreedyResult:
    tokens: torch.Tensor
    num_accepted: torch.Tensor
    status: torch.Tensor
    ws: torch.Tensor


def verify_greedy(logits, draft, *, k_per_req=None, l_row_off=None, out: Optional[GreedyResult] = None,
                  ws: Optional[torch.Tensor] = None, stream=None) -> GreedyResult:
    """Greedy argmax-match verification.  Layouts as in verify_chain."""
    L = _load()
    _cuda(logits, "logits")
    ldt = _ldt(logits)
    _cuda(draft, "draft", torch.int32)
    if draft.dim() != 2 or not draft.is_contiguous():
        raise SpecError("draft must be a contiguous [B, K] tensor")
    B, K = draft.shape
    V = logits.shape[-1]
    if logits.stride(-1) != 1:
        raise SpecError("logits need unit element stride")
    if k_per_req is not None:
        _cuda(k_per_req, "k_per_req", torch.int32)
    if l_row_off is not None:
        if k_per_req is None:
            raise SpecError("l_row_off needs k_per_req")
        _cuda(l_row_off, "l_row_off", torch.int32)
        lbs, lrs = 0, logits.stride(0)
    else:
        if logits.dim() != 3 or logits.shape[:2] != (B, K + 1):
            raise SpecError("dense logits must be [B, K+1, V]")
        lbs, lrs = logits.stride(0), logits.stride(1)
    dev = _dev(logits)
    if out is None:
        out = GreedyResult(torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                           torch.empty(B, dtype=torch.int32, device=dev),
                           torch.empty(B, dtype=torch.int32, device=dev), None)
    need = L.spec_verify_greedy_workspace_size(B, K, V)
    if ws is None:
        ws = workspace(need, dev)
    out.ws = ws
    rc = L.spec_verify_greedy(_p(logits), ldt, lbs, lrs, _p(draft), B, K, V, _p(k_per_req), _p(l_row_off),
                              _p(out.tokens), _p(out.num_accepted), _p(out.status), _p(ws), ws.numel(),
                              _stream(stream))
    _check(rc, "spec_verify_greedy")
    return out


# ---------------------------------------------------------------------------
# DDTree
# ---------------------------------------------------------------------------
@dataclass
class Tree:
    token: torch.Tensor      # [B, N] int32
    parent: torch.Tensor     # [B, N] int32
    depth: torch.Tensor      # [B, N] int32
    score: torch.Tensor      # [B, N] float64
    anc_mask: torch.Tensor   # [B, N, ceil(N/64)] int64 (bit patterns of uint64)
    num_nodes: torch.Tensor  # [B] int32
    status: torch.Tensor     # [B] int32
    ws: torch.Tensor


def tree_build(q, budget: int, *, out: Optional[Tree] = None, ws: Optional[torch.Tensor] = None,
               stream=None) -> Tree:
    """DDTree best-first tree over per-depth marginals q [B, L, V] fp32."""
    Lb = _load()
    _cuda(q, "q", torch.float32)
    if q.dim() != 3 or q.stride(-1) != 1:
        raise SpecError("q must be [B, L, V] with unit element stride")
    B, L, V = q.shape
    N = int(budget)
    W = (N + 63) // 64
    dev = _dev(q)
    if out is None:
        out = Tree(torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.float64, device=dev),
                   torch.empty((B, N, W), dtype=torch.int64, device=dev),
                   torch.empty(B, dtype=torch.int32, device=dev),
                   torch.empty(B, dtype=torch.int32, device=dev), None)
    need = Lb.spec_tree_build_workspace_size(B, L, V, N)
    if need == 0 and B > 0:
        raise SpecError("unsupported tree shape (L <= 16, 1 <= budget <= 256)")
    if ws is None:
        ws = workspace(need, dev)
    out.ws = ws
    rc = Lb.spec_tree_build(_p(q), q.stride(0), q.stride(1), B, L, V, N,
                            _p(out.token), _p(out.parent), _p(out.depth), _p(out.score), _p(out.anc_mask),
                            _p(out.num_nodes), _p(out.status), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "spec_tree_build")
    return out


@dataclass
class EagleState:
    """EAGLE-2 node arrays of capacity G (page §4): the generated candidates."""
    token: torch.Tensor        # [B, G] int32
    parent: torch.Tensor       # [B, G] int32
    depth: torch.Tensor        # [B, G] int32
    score: torch.Tensor        # [B, G] fp64, product of draft probabilities along the path
    num_gen: torch.Tensor      # [B] int32


def eagle_state(B: int, G: int, device) -> EagleState:
    """Node arrays holding only the root (node 0: token -1, depth 0, score 1)."""
    st = EagleState(torch.full((B, G), -1, dtype=torch.int32, device=device),
                    torch.full((B, G), -1, dtype=torch.int32, device=device),
                    torch.full((B, G), -1, dtype=torch.int32, device=device),
                    torch.zeros((B, G), dtype=torch.float64, device=device),
                    torch.ones(B, dtype=torch.int32, device=device))
    st.depth[:, 0] = 0
    st.score[:, 0] = 1.0
    return st


def eagle_expand(q, state: EagleState, front, num_front, K2: int, Fn: int, *, front_out=None,
                 num_front_out=None, status=None, ws: Optional[torch.Tensor] = None, stream=None):
    """One EAGLE-2 expansion step (page §4): q [B, F, V] fp32 holds the draft's
    conditional rows of the frontier nodes front [B, F] (num_front [B] valid).
    Appends the children to `state`; returns (front_out [B, Fn], num_front_out
    [B], status [B])."""
    Lb = _load()
    _cuda(q, "q", torch.float32)
    if q.dim() != 3 or q.stride(-1) != 1:
        raise SpecError("q must be [B, F, V] with unit element stride")
    B, F, V = q.shape
    G = state.token.shape[1]
    _cuda(front, "front", torch.int32)
    _cuda(num_front, "num_front", torch.int32)
    for name in ("token", "parent", "depth", "num_gen"):
        _cuda(getattr(state, name), name, torch.int32)
    _cuda(state.score, "score", torch.float64)
    if tuple(front.shape) != (B, F) or not front.is_contiguous():
        raise SpecError("front must be a contiguous [B, F] tensor")
    dev = _dev(q)
    if front_out is None:
        front_out = torch.empty((B, Fn), dtype=torch.int32, device=dev)
    if num_front_out is None:
        num_front_out = torch.empty(B, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    need = Lb.spec_eagle_expand_workspace_size(B, F, K2)
    if ws is None:
        ws = workspace(need, dev)
    rc = Lb.spec_eagle_expand(_p(q), q.stride(0), q.stride(1), B, F, V, int(K2), int(Fn), G,
                              _p(state.token), _p(state.parent), _p(state.depth), _p(state.score),
                              _p(state.num_gen), _p(front), _p(num_front), _p(front_out), _p(num_front_out),
                              _p(status), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "spec_eagle_expand")
    return front_out, num_front_out, status


def eagle_rerank(state: EagleState, budget: int, *, out: Optional[Tree] = None, stream=None) -> Tree:
    """The EAGLE-2 verification tree (page §4): the root and the budget-1
    best generated nodes, in the layout tree_build returns."""
    Lb = _load()
    B, G = state.token.shape
    N = int(budget)
    W = (N + 63) // 64
    dev = _dev(state.token)
    if out is None:
        out = Tree(torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.int32, device=dev),
                   torch.empty((B, N), dtype=torch.float64, device=dev),
                   torch.empty((B, N, W), dtype=torch.int64, device=dev),
                   torch.empty(B, dtype=torch.int32, device=dev),
                   torch.empty(B, dtype=torch.int32, device=dev), None)
    rc = Lb.spec_eagle_rerank(_p(state.token), _p(state.parent), _p(state.depth), _p(state.score),
                              _p(state.num_gen), B, G, N,
                              _p(out.token), _p(out.parent), _p(out.depth), _p(out.score), _p(out.anc_mask),
                              _p(out.num_nodes), _p(out.status), _stream(stream))
    _check(rc, "spec_eagle_rerank")
    return out


@dataclass
class TreeWalk:
    path_nodes: torch.Tensor   # [B, L+1]
    tokens: torch.Tensor       # [B, L+1]
    num_accepted: torch.Tensor
    status: torch.Tensor
    ws: torch.Tensor


def verify_tree(logits, token, parent, num_nodes, max_depth: int, *, out: Optional[TreeWalk] = None,
                ws: Optional[torch.Tensor] = None, stream=None) -> TreeWalk:
    """Greedy tree walk over target logits [B, N, V] (fp32 or bf16)."""
    Lb = _load()
    _cuda(logits, "logits")
    ldt = _ldt(logits)
    for t, n in ((token, "token"), (parent, "parent"), (num_nodes, "num_nodes")):
        _cuda(t, n, torch.int32)
        if not t.is_contiguous():
            raise SpecError(f"{n} must be contiguous")
    if logits.dim() != 3 or logits.stride(-1) != 1:
        raise SpecError("logits must be [B, N, V] with unit element stride")
    B, N = token.shape
    V = logits.shape[-1]
    Ld = int(max_depth)
    dev = _dev(logits)
    if out is None:
        out = TreeWalk(torch.empty((B, Ld + 1), dtype=torch.int32, device=dev),
                       torch.empty((B, Ld + 1), dtype=torch.int32, device=dev),
                       torch.empty(B, dtype=torch.int32, device=dev),
                       torch.empty(B, dtype=torch.int32, device=dev), None)
    need = Lb.spec_verify_tree_workspace_size(B, N, V)
    if ws is None:
        ws = workspace(need, dev)
    out.ws = ws
    rc = Lb.spec_verify_tree(_p(logits), ldt, logits.stride(0), logits.stride(1), _p(token), _p(parent),
                             _p(num_nodes), B, N, V, Ld, _p(out.path_nodes), _p(out.tokens),
                             _p(out.num_accepted), _p(out.status), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "spec_verify_tree")
    return out


def verify_tree_sample(logits, token, parent, num_nodes, uniforms, max_depth: int, temperature: float,
                       top_k: int = 0, *, out: Optional[TreeWalk] = None, ws: Optional[torch.Tensor] = None,
                       stream=None) -> TreeWalk:
    """Stochastic tree walk over target logits [B, N, V] (fp32 or bf16):
    at depth d the current node's token is drawn from its p (temperature,
    top-k) with uniforms[b, d]; uniforms [B, max_depth+1] fp32."""
    Lb = _load()
    _cuda(logits, "logits")
    ldt = _ldt(logits)
    for t, n in ((token, "token"), (parent, "parent"), (num_nodes, "num_nodes")):
        _cuda(t, n, torch.int32)
        if not t.is_contiguous():
            raise SpecError(f"{n} must be contiguous")
    _cuda(uniforms, "uniforms", torch.float32)
    if logits.dim() != 3 or logits.stride(-1) != 1:
        raise SpecError("logits must be [B, N, V] with unit element stride")
    B, N = token.shape
    V = logits.shape[-1]
    Ld = int(max_depth)
    if uniforms.shape != (B, Ld + 1) or not uniforms.is_contiguous():
        raise SpecError("uniforms must be a contiguous [B, max_depth+1] tensor")
    dev = _dev(logits)
    if out is None:
        out = TreeWalk(torch.empty((B, Ld + 1), dtype=torch.int32, device=dev),
                       torch.empty((B, Ld + 1), dtype=torch.int32, device=dev),
                       torch.empty(B, dtype=torch.int32, device=dev),
                       torch.empty(B, dtype=torch.int32, device=dev), None)
    need = Lb.spec_verify_tree_sample_workspace_size(B, N, V)
    if ws is None:
        ws = workspace(need, dev)
    out.ws = ws
    rc = Lb.spec_verify_tree_sample(_p(logits), ldt, logits.stride(0), logits.stride(1), _p(token), _p(parent),
                                    _p(num_nodes), _p(uniforms), B, N, V, Ld, float(temperature), int(top_k),
                                    _p(out.path_nodes), _p(out.tokens), _p(out.num_accepted), _p(out.status),
                                    _p(ws), ws.numel(), _stream(stream))
    _check(rc, "spec_verify_tree_sample")
    return out


def kv_compact(src, dst, path_nodes, num_accepted, dst_pos=None, stream=None):
    """Keep the accepted path's KV rows (page §5, DDTree): src [P, B, N, ...]
    (one row per tree node), dst [P, B, M, ...] (the cache), same dtype and
    row shape; row dst_pos[b] + j of dst receives src row path_nodes[b, j],
    j = 0..num_accepted[b].  In place on dst."""
    Lb = _load()
    _cuda(src, "src")
    _cuda(dst, "dst", src.dtype)
    _cuda(path_nodes, "path_nodes", torch.int32)
    _cuda(num_accepted, "num_accepted", torch.int32)
    if src.dim() < 4 or dst.dim() != src.dim() or src.shape[3:] != dst.shape[3:]:
        raise SpecError("src [P, B, N, ...] and dst [P, B, M, ...] with the same row shape")
    if src.shape[:2] != dst.shape[:2]:
        raise SpecError("src and dst need the same P and B")
    row = src[0, 0, 0]
    if not (src.stride(-1) == 1 and row.is_contiguous() and dst[0, 0, 0].is_contiguous()):
        raise SpecError("rows must be contiguous")
    es = src.element_size()
    P, B, N = src.shape[:3]
    if not path_nodes.is_contiguous() or path_nodes.dim() != 2 or path_nodes.shape[0] != B:
        raise SpecError("path_nodes must be a contiguous [B, path_width] tensor")
    if dst_pos is not None:
        _cuda(dst_pos, "dst_pos", torch.int32)
    rc = Lb.spec_kv_compact(_p(src), src.stride(0) * es, src.stride(1) * es, src.stride(2) * es,
                            _p(dst), dst.stride(0) * es, dst.stride(1) * es, dst.stride(2) * es,
                            P, B, N, row.numel() * es, _p(path_nodes), path_nodes.shape[1], _p(num_accepted),
                            _p(dst_pos), _stream(stream))
    _check(rc, "spec_kv_compact")
    return dst


# ---------------------------------------------------------------------------
# DSpark
# ---------------------------------------------------------------------------
@dataclass
class AdaptiveLen:
    k: torch.Tensor          # [B] int32
    surv: torch.Tensor       # [B, Kmax] float64
    exp_adv: torch.Tensor    # [B] float64
    l_row_off: torch.Tensor  # [B+1] int32
    q_row_off: torch.Tensor  # [B+1] int32


def adaptive_len(conf, a: float, b: float, *, cost=None, out: Optional[AdaptiveLen] = None,
                 stream=None) -> AdaptiveLen:
    """DSpark verify length from conditional confidences conf [B, Kmax] fp32;
    the cost of k positions is a + b*k, or cost[k] with a profiled table
    (a CUDA float64 tensor of Kmax+1 positive entries)."""
    Lb = _load()
    _cuda(conf, "conf", torch.float32)
    if conf.dim() != 2 or not conf.is_contiguous():
        raise SpecError("conf must be a contiguous [B, Kmax] tensor")
    B, Kmax = conf.shape
    dev = _dev(conf)
    if out is None:
        out = AdaptiveLen(torch.empty(B, dtype=torch.int32, device=dev),
                          torch.empty((B, Kmax), dtype=torch.float64, device=dev),
                          torch.empty(B, dtype=torch.float64, device=dev),
                          torch.empty(B + 1, dtype=torch.int32, device=dev),
                          torch.empty(B + 1, dtype=torch.int32, device=dev))
    if cost is None:
        rc = Lb.spec_adaptive_len(_p(conf), B, Kmax, float(a), float(b), _p(out.k), _p(out.surv), _p(out.exp_adv),
                                  _p(out.l_row_off), _p(out.q_row_off), _stream(stream))
        _check(rc, "spec_adaptive_len")
    else:
        _cuda(cost, "cost", torch.float64)
        if cost.shape != (Kmax + 1,) or not cost.is_contiguous():
            raise SpecError("cost must be a contiguous [Kmax+1] float64 tensor")
        rc = Lb.spec_adaptive_len_table(_p(conf), B, Kmax, _p(cost), _p(out.k), _p(out.surv), _p(out.exp_adv),
                                        _p(out.l_row_off), _p(out.q_row_off), _stream(stream))
        _check(rc, "spec_adaptive_len_table")
    return out
