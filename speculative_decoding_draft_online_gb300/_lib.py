"""ctypes binding of libspecverify.so: argument marshalling only.

Every step of verification runs in the library's CUDA kernels; this module
checks tensor shapes and dtypes, allocates outputs and the workspace with
torch, and passes raw device pointers plus the current torch stream.  If the
library is missing the import fails -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_BF16, SPEC_FP32 = 0, 1
SPEC_OK = 0
STATUS_NAMES = {0: "ok", -1: "arg", -2: "align", -3: "token", -4: "nonfinite", -5: "unsupported",
                -6: "timeout", -7: "cuda", -8: "workspace"}
SPEC_ERR_TOKEN, SPEC_ERR_NONFINITE = -3, -4


class SpecError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({lib.spec_strerror(code).decode()})")
        self.code = code


class _Aux(ctypes.Structure):
    """spec_verify_aux of ABI 1.2."""
    _fields_ = [("p_draft", ctypes.c_void_p), ("q_draft", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("events", ctypes.c_void_p * 4),
                ("sequence_offset", ctypes.c_uint32), ("lenience", ctypes.c_float),
                ("stop_ids", ctypes.c_void_p), ("n_stop", ctypes.c_int32), ("n_committed", ctypes.c_void_p),
                ("match_mask", ctypes.c_void_p), ("n_match", ctypes.c_void_p), ("tail_runs", ctypes.c_void_p),
                ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


ABI_MIN = (1 << 16) | 3


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python __graft_entry__.py build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    L.spec_workspace_size.argtypes = [i32, i32, i32, i32]
    L.spec_workspace_size.restype = sz
    L.spec_workspace_init.argtypes = [vp, sz, vp]
    L.spec_workspace_init.restype = i32
    common = [vp, vp, vp, i32, i32, i32, i32, f32, u64, vp, vp, vp, sz, vp]
    L.spec_verify.argtypes = common
    L.spec_verify.restype = i32
    L.spec_verify_ex.argtypes = common + [ctypes.POINTER(_Aux)]
    L.spec_verify_ex.restype = i32
    L.spec_verify_tree.argtypes = [vp, vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, vp, vp, sz, vp]
    L.spec_verify_tree.restype = i32
    L.spec_verify_guided.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.spec_verify_guided.restype = i32
    L.spec_random.argtypes = [u64, i32, i32, i32, vp, vp, vp, vp]
    L.spec_random.restype = i32
    L.spec_strerror.argtypes = [i32]
    L.spec_strerror.restype = ctypes.c_char_p
    L.spec_abi_version.argtypes = []
    L.spec_abi_version.restype = i32
    L.spec_probe_read.argtypes = [vp, sz, vp, i32, vp]
    L.spec_probe_read.restype = i32
    L.spec_test_force_stage_timeouts.argtypes = [i32]
    L.spec_test_force_stage_timeouts.restype = i32
    if L.spec_abi_version() < ABI_MIN or (L.spec_abi_version() >> 16) != (ABI_MIN >> 16):
        raise ImportError(f"{LIB_PATH} has ABI {L.spec_abi_version():#x}, this binding needs {ABI_MIN:#x}")
    return L


lib = _load()

_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream: Optional[torch.cuda.Stream], device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_FP32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def workspace_size(B: int, k: int, V: int, dtype: int = SPEC_BF16) -> int:
    return int(lib.spec_workspace_size(B, k, V, dtype))


def workspace(B: int, k: int, V: int, dtype: int, device, stream=None) -> torch.Tensor:
    """A zero-filled workspace, cached per (device, stream) and grown on demand.

    Calls that share a cached workspace are ordered on one stream, which the
    library requires; pass your own workspace to run calls concurrently.
    """
    need = workspace_size(B, k, V, dtype)
    if need == 0:
        raise ValueError(f"invalid sizes B={B} k={k} V={V}")
    dev = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    key = (dev.index, s.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(need, dtype=torch.uint8, device=dev)
            _ws_cache[key] = ws
    return ws


def _check(t: torch.Tensor, name: str, shape, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def verify_ex(target: torch.Tensor, draft: Optional[torch.Tensor], tokens: torch.Tensor, temperature: float,
              seed: int = 0, *, out_tokens=None, out_n=None, ws=None, stream=None, aux: bool = False,
              events=None, sequence_offset: int = 0, lenience: float = 1.0,
              stop_ids: Optional[torch.Tensor] = None, committed: bool = False, match: bool = False,
              top_k: int = 0, top_p: float = 0.0):
    """spec_verify_ex on torch tensors.

    target [B][k+1][V] and draft [B][k][V] (bf16 or fp32, same dtype), tokens
    [B][k] int32.  temperature == 0 selects greedy verification (draft may be
    None).  Returns (out_tokens [B][k+1] int32, n_accepted [B] int32), plus a
    dict when any of these is asked for:
      aux=True        p_draft, q_draft, lse, status
      committed=True  n_committed (after truncation at stop_ids)
      match=True      (greedy) match_mask [B][k] uint8, n_match, tail_runs
    sequence_offset is the global index of sequence 0 when the batch is a
    shard of a larger one; lenience >= 1 loosens the stochastic accept test;
    stop_ids is an int32 CUDA tensor of stop ids (the committed tokens end at
    the first one); top_k / top_p filter every target and draft row alike
    before the rule (stochastic mode; 0 = off).
    """
    B, k1, V = target.shape
    k = k1 - 1
    code = dtype_code(target)
    dev = target.device
    _check(target, "target", (B, k + 1, V))
    if temperature != 0.0:
        if draft is None:
            raise ValueError("stochastic verification needs draft logits")
        _check(draft, "draft", (B, k, V), target.dtype)
    _check(tokens, "tokens", (B, k), torch.int32)
    if stop_ids is not None:
        _check(stop_ids, "stop_ids", (stop_ids.numel(),), torch.int32)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(B, k, V, code, dev, stream)
    extra = {}
    a = None
    if (aux or events is not None or sequence_offset or lenience != 1.0 or stop_ids is not None or committed
            or match or top_k or top_p):
        a = _Aux()
        a.sequence_offset = int(sequence_offset)
        a.lenience = float(lenience)
        a.top_k = int(top_k)
        a.top_p = float(top_p)
        if aux:
            extra.update(p_draft=torch.zeros((B, k), dtype=torch.float32, device=dev),
                         q_draft=torch.zeros((B, k), dtype=torch.float32, device=dev),
                         lse=torch.zeros((B, 2 * k), dtype=torch.float32, device=dev),
                         status=torch.zeros((B,), dtype=torch.int32, device=dev))
            a.p_draft, a.q_draft = extra["p_draft"].data_ptr(), extra["q_draft"].data_ptr()
            a.lse, a.status = extra["lse"].data_ptr(), extra["status"].data_ptr()
        if stop_ids is not None and stop_ids.numel() > 0:
            a.stop_ids, a.n_stop = stop_ids.data_ptr(), int(stop_ids.numel())
        if committed:
            extra["n_committed"] = torch.empty((B,), dtype=torch.int32, device=dev)
            a.n_committed = extra["n_committed"].data_ptr()
        if match:
            extra.update(match_mask=torch.empty((B, k), dtype=torch.uint8, device=dev),
                         n_match=torch.empty((B,), dtype=torch.int32, device=dev),
                         tail_runs=torch.empty((B,), dtype=torch.int32, device=dev))
            a.match_mask, a.n_match = extra["match_mask"].data_ptr(), extra["n_match"].data_ptr()
            a.tail_runs = extra["tail_runs"].data_ptr()
        if events is not None:
            for i, e in enumerate(events[:4]):
                a.events[i] = None if e is None else e.cuda_event
    args = (_ptr(target), _ptr(draft) if temperature != 0.0 else None, _ptr(tokens), B, k, V, code,
            float(temperature), ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), _ptr(out_tokens), _ptr(out_n),
            _ptr(ws), ws.numel(), _stream_ptr(stream, dev))
    rc = lib.spec_verify_ex(*args, ctypes.byref(a) if a is not None else None)
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_ex")
    if extra:
        return out_tokens, out_n, extra
    return out_tokens, out_n


def verify(target, draft, tokens, temperature: float, seed: int = 0, **kw):
    """spec_verify on torch tensors: returns (out_tokens, n_accepted)."""
    kw.pop("aux", None)
    return verify_ex(target, draft, tokens, temperature, seed, **kw)


def verify_tree(target: torch.Tensor, node_tokens: torch.Tensor, parents: torch.Tensor, *, ws=None, stream=None,
                temperature: float = 0.0):
    """spec_verify_tree: returns (out_tokens [B][N+1], n_accepted [B], leaf [B], status [B])."""
    B, N1, V = target.shape
    N = N1 - 1
    code = dtype_code(target)
    dev = target.device
    _check(target, "target", (B, N + 1, V))
    _check(node_tokens, "node_tokens", (B, N), torch.int32)
    _check(parents, "parents", (B, N), torch.int32)
    out = torch.empty((B, N + 1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)
    leaf = torch.empty((B,), dtype=torch.int32, device=dev)
    status = torch.empty((B,), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(B, N, V, code, dev, stream)
    rc = lib.spec_verify_tree(_ptr(target), _ptr(node_tokens), _ptr(parents), B, N, V, code, float(temperature),
                              _ptr(out), _ptr(n), _ptr(leaf), _ptr(status), _ptr(ws), ws.numel(),
                              _stream_ptr(stream, dev))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_tree")
    return out, n, leaf, status


def verify_guided(target: torch.Tensor, tokens: torch.Tensor, guide: torch.Tensor, *, ws=None, stream=None):
    """spec_verify_guided (greedy verification, then the target-side guide).

    target [B][k+1][V], tokens [B][k] int32, guide [B][L] int32 (negative =
    past its end).  Returns (out_tokens [B][max(k+1, L)], n_accepted [B],
    n_committed [B], status [B]).
    """
    B, k1, V = target.shape
    k = k1 - 1
    L = guide.shape[1] if guide.dim() == 2 else 0
    code = dtype_code(target)
    dev = target.device
    _check(target, "target", (B, k + 1, V))
    _check(tokens, "tokens", (B, k), torch.int32)
    _check(guide, "guide", (B, L), torch.int32)
    W = max(k + 1, L)
    out = torch.empty((B, W), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)
    nc = torch.empty((B,), dtype=torch.int32, device=dev)
    status = torch.empty((B,), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(B, k, V, code, dev, stream)
    rc = lib.spec_verify_guided(_ptr(target), _ptr(tokens), _ptr(guide) if L > 0 else None, B, k, L, V, code,
                                _ptr(out), _ptr(n), _ptr(nc), _ptr(status), _ptr(ws), ws.numel(),
                                _stream_ptr(stream, dev))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_verify_guided")
    return out, n, nc, status


def random_stream(seed: int, b: int, j: int, V: int, device="cuda", stream=None):
    """spec_random: (Gumbel uniforms [V], Gumbel noise [V], accept uniform of (b, j))."""
    dev = torch.device(device)
    u = torch.empty(V, dtype=torch.float32, device=dev)
    g = torch.empty(V, dtype=torch.float32, device=dev)
    a = torch.empty(1, dtype=torch.float32, device=dev)
    rc = lib.spec_random(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), b, j, V, _ptr(u), _ptr(g), _ptr(a),
                         _stream_ptr(stream, dev))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_random")
    return u, g, a


def force_stage_timeouts(on: bool) -> bool:
    """Test hook: make every bulk-copy stage wait of later calls give up at once
    (spec_test_force_stage_timeouts).  Returns the previous setting."""
    return bool(lib.spec_test_force_stage_timeouts(1 if on else 0))


def probe_read(buf: torch.Tensor, ctas: int = 0, stream=None) -> None:
    """spec_probe_read over a contiguous device tensor (measurement helper)."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("probe_read needs a contiguous CUDA tensor")
    sink = torch.zeros(max(ctas, 4096), dtype=torch.int32, device=buf.device)
    rc = lib.spec_probe_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink), ctas,
                             _stream_ptr(stream, buf.device))
    if rc != SPEC_OK:
        raise SpecError(rc, "spec_probe_read")
