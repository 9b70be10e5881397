"""GB300 (sm_103a) SANTA / S2ANTA decode-step attention.

Thin Python binding over the C ABI in ``include/santa.h`` (``libsanta.so``,
built in-tree by ``stochastic_sparse_decode_split_gb300.build``).  The binding
only marshals arguments: PyTorch tensors supply device memory and the current
CUDA stream, and every step of the operator runs in the library's kernels.
There is no CPU fallback: if the library is missing or a call fails, an
exception is raised.

Operator ("Stochastic Sparse Attention for Memory-Bound Inference", Sec. 2,
Eq. 1 and 4; Sec. 2.1): per query head, exact scores and softmax over the whole
key cache, S draws from the post-softmax distribution (i.i.d., stratified or
systematic; Philox4x32-10 keyed by seed, batch, head, step), and the estimate
(1/S) * sum of the drawn V rows computed as a count-weighted gather-and-add.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import torch

from .build import LIB as _LIB_PATH

__all__ = [
    "SantaError", "Params", "library", "santa_decode", "santa_decode_host_kv", "santa_decode_with_uniforms",
    "santa_dense_decode",
    "workspace_size", "dense_workspace_size", "workspace_layout", "get_error", "Decoder", "exported_symbols",
    "VARIANTS", "DTYPES", "santa_decode_static", "static_warmup", "static_scratch_bytes", "SAMPLERS", "santa_decode_tiled",
    "tiled_workspace_size", "tiled_max_draws", "santa_decode_bernoulli", "bernoulli_workspace_size",
]

VARIANTS = {"iid": 0, "stratified": 1, "systematic": 2}
SAMPLERS = {"prop": 0, "flash": 1}   # SANTA_TILE_PROP, SANTA_TILE_FLASH
DTYPES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "santa.h")

SANTA_OK, SANTA_ERR_DEVICE = 0, 5
# bits of the device error word returned by get_error (SANTA_DEVERR_* in santa.h)
DEVERR_NK_BOUND, DEVERR_S_RANGE, DEVERR_EMPTY, DEVERR_TIMEOUT = 1, 2, 4, 8


class SantaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {library().santa_status_string(status).decode()} (status {status})")


class Params(ctypes.Structure):
    """Mirror of santa_params_t."""
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("kv_offsets", ctypes.c_void_p),
        ("nk", ctypes.c_int64),
        ("S", ctypes.c_int32),
        ("S_per_seq", ctypes.c_void_p),
        ("scale", ctypes.c_float),
        ("seed", ctypes.c_uint64),
        ("step", ctypes.c_uint32),
    ]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("stash", "tile_max", "tile_sum", "prefix", "thresh", "head_max")] + [
        ("chunks", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def library():
    """Loads libsanta.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                                   "`python -m stochastic_sparse_decode_split_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
            P = ctypes.POINTER(Params)
            lib.santa_workspace_size.argtypes = [P]
            lib.santa_workspace_size.restype = sz
            lib.santa_dense_workspace_size.argtypes = [P]
            lib.santa_dense_workspace_size.restype = sz
            lib.santa_workspace_init.argtypes = [vp, sz, vp]
            lib.santa_decode.argtypes = [P, i32, vp, vp, vp, vp, vp, sz, vp, vp]
            lib.santa_decode_host_kv.argtypes = [P, i32, vp, vp, vp, vp, vp, sz, vp, vp]
            lib.santa_decode_profiled.argtypes = [P, i32, vp, vp, vp, vp, vp, sz, vp, vp, vp]
            lib.santa_score_pass.argtypes = [P, vp, vp, vp, sz, vp]
            lib.santa_decode_with_uniforms.argtypes = [P, i32, vp, vp, vp, vp, vp, vp, sz, vp, vp]
            lib.santa_dense_decode.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
            lib.santa_decode_static.argtypes = [P, i32, vp, vp, vp, vp, vp, vp]
            lib.santa_static_warmup.argtypes = []
            lib.santa_workspace_layout.argtypes = [P, ctypes.POINTER(WsLayout)]
            lib.santa_tiled_workspace_size.argtypes = [P, i32, i32]
            lib.santa_tiled_workspace_size.restype = sz
            lib.santa_tiled_max_draws.argtypes = [P, i32, i32]
            lib.santa_tiled_max_draws.restype = i32
            lib.santa_decode_tiled.argtypes = [P, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
            lib.santa_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint64, vp]
            lib.santa_selftest_wait_timeout.restype = i32
            lib.santa_read_probe_sink_words.restype = i32
            lib.santa_read_probe.argtypes = [vp, sz, vp, vp]
            lib.santa_read_probe.restype = i32
            lib.santa_bernoulli_workspace_size.argtypes = [P]
            lib.santa_bernoulli_workspace_size.restype = sz
            lib.santa_decode_bernoulli.argtypes = [P, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp, vp]
            lib.santa_get_error.argtypes = [vp, vp, ctypes.POINTER(i32)]
            lib.santa_status_string.argtypes = [i32]
            lib.santa_status_string.restype = ctypes.c_char_p
            lib.santa_version.restype = i32
            for fn in ("santa_workspace_init", "santa_decode", "santa_decode_host_kv", "santa_decode_profiled",
                       "santa_score_pass",
                       "santa_decode_with_uniforms", "santa_dense_decode", "santa_decode_static",
                       "santa_workspace_layout", "santa_get_error", "santa_decode_tiled", "santa_decode_bernoulli"):
                getattr(lib, fn).restype = i32
            _lib = lib
    return _lib


def exported_symbols():
    """Function names declared in include/santa.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(santa_[a-z_]+)\s*\(", text)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_params(q: torch.Tensor, K: torch.Tensor, S: int, seed: int = 0, step: int = 0, nk: Optional[int] = None,
                kv_offsets: Optional[torch.Tensor] = None, S_per_seq: Optional[torch.Tensor] = None,
                scale: float = 0.0) -> Params:
    if q.dim() != 3 or K.dim() != 3:
        raise ValueError("q must be [B, H, d] and K [rows, H_kv, d]")
    B, H, d = q.shape
    Hkv = K.shape[1]
    if q.dtype not in DTYPES or K.dtype != q.dtype:
        raise ValueError("q, K, V must share one of bf16 / fp16 / fp32")
    if nk is None:
        if kv_offsets is not None:
            raise ValueError("give nk (an upper bound on every sequence length) with kv_offsets")
        if K.shape[0] % B:
            raise ValueError("uniform batch: K rows must be a multiple of the batch")
        nk = K.shape[0] // B
    p = Params()
    p.batch, p.n_q_heads, p.n_kv_heads, p.head_dim = B, H, Hkv, d
    p.dtype = DTYPES[q.dtype]
    p.kv_offsets = None if kv_offsets is None else kv_offsets.data_ptr()
    p.nk = int(nk)
    p.S = int(S)
    p.S_per_seq = None if S_per_seq is None else S_per_seq.data_ptr()
    p.scale = float(scale)
    p.seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    p.step = int(step) & 0xFFFFFFFF
    return p


def workspace_size(p: Params) -> int:
    return int(library().santa_workspace_size(ctypes.byref(p)))


def dense_workspace_size(p: Params) -> int:
    return int(library().santa_dense_workspace_size(ctypes.byref(p)))


def workspace_layout(p: Params) -> dict:
    lay = WsLayout()
    if library().santa_workspace_layout(ctypes.byref(p), ctypes.byref(lay)) != 0:
        raise ValueError("invalid parameters")
    return {n: getattr(lay, n) for n, _ in WsLayout._fields_}


def alloc_workspace(nbytes: int, device) -> torch.Tensor:
    """Device workspace (uint8, 256-byte aligned, control words cleared)."""
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    st = library().santa_workspace_init(_ptr(ws), nbytes, _stream())
    if st != SANTA_OK:
        raise SantaError(st, "santa_workspace_init")
    return ws


def get_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns (then clears) the device error flags."""
    code = ctypes.c_int32(0)
    st = library().santa_get_error(_ptr(workspace), _stream(stream), ctypes.byref(code))
    if st not in (SANTA_OK, SANTA_ERR_DEVICE):
        raise SantaError(st, "santa_get_error")
    return int(code.value)


def _check_tensors(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def santa_decode(q, K, V, S: int, variant: str = "systematic", seed: int = 0, step: int = 0, out=None,
                 nk: Optional[int] = None, kv_offsets=None, S_per_seq=None, scale: float = 0.0, workspace=None,
                 sample_idx=None, stream=None) -> torch.Tensor:
    """One S2ANTA / SANTA decode step; returns out [B, H, d] float32."""
    _check_tensors(q, K, V, out, kv_offsets, S_per_seq, sample_idx)
    p = make_params(q, K, S, seed, step, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(p), q.device)
    st = library().santa_decode(ctypes.byref(p), VARIANTS[variant], _ptr(q), _ptr(K), _ptr(V), _ptr(out),
                                _ptr(workspace), workspace.numel(), _stream(stream), _ptr(sample_idx))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode")
    return out


def santa_decode_host_kv(q, K, V, S: int, variant: str = "systematic", seed: int = 0, step: int = 0, out=None,
                         nk: Optional[int] = None, kv_offsets=None, S_per_seq=None, scale: float = 0.0,
                         workspace=None, sample_idx=None, stream=None) -> torch.Tensor:
    """santa_decode with K and V each either a CUDA tensor or a contiguous
    pinned CPU tensor, read in place by the GPU (of V only the drawn rows).
    q and the optional tensors are CUDA tensors as in santa_decode."""
    _check_tensors(q, out, kv_offsets, S_per_seq, sample_idx)
    for t in (K, V):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("K and V must be contiguous CUDA or pinned CPU tensors")
    p = make_params(q, K, S, seed, step, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(p), q.device)
    st = library().santa_decode_host_kv(ctypes.byref(p), VARIANTS[variant], _ptr(q), _ptr(K), _ptr(V), _ptr(out),
                                        _ptr(workspace), workspace.numel(), _stream(stream), _ptr(sample_idx))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode_host_kv")
    return out


def santa_decode_with_uniforms(q, K, V, uniforms, S: int, variant: str, out=None, nk=None, kv_offsets=None,
                               S_per_seq=None, scale: float = 0.0, workspace=None, sample_idx=None,
                               stream=None) -> torch.Tensor:
    """santa_decode with explicit float64 uniforms [B, H, S] in place of Philox."""
    _check_tensors(q, K, V, uniforms, out, kv_offsets, S_per_seq, sample_idx)
    if uniforms.dtype != torch.float64:
        raise ValueError("uniforms must be float64")
    p = make_params(q, K, S, 0, 0, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(workspace_size(p), q.device)
    st = library().santa_decode_with_uniforms(ctypes.byref(p), VARIANTS[variant], _ptr(q), _ptr(K), _ptr(V),
                                              _ptr(uniforms), _ptr(out), _ptr(workspace), workspace.numel(),
                                              _stream(stream), _ptr(sample_idx))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode_with_uniforms")
    return out


def tiled_workspace_size(p: Params, sampler: str, tile_len: int) -> int:
    return library().santa_tiled_workspace_size(ctypes.byref(p), SAMPLERS[sampler], tile_len)


def tiled_max_draws(p: Params, sampler: str, tile_len: int) -> int:
    return library().santa_tiled_max_draws(ctypes.byref(p), SAMPLERS[sampler], tile_len)


def santa_decode_tiled(q, K, V, S: int, sampler: str = "prop", tile_len: int = 256, seed: int = 0, step: int = 0,
                       out=None, nk: Optional[int] = None, kv_offsets=None, S_per_seq=None, scale: float = 0.0,
                       workspace=None, sample_idx=None, stream=None) -> torch.Tensor:
    """One decode step through S2ANTA-prop or S2ANTA-flash; returns out [B, H, d]
    float32.  sample_idx, if given, is int32 [B, H, tiled_max_draws(...)]."""
    _check_tensors(q, K, V, out, kv_offsets, S_per_seq, sample_idx)
    p = make_params(q, K, S, seed, step, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        n = tiled_workspace_size(p, sampler, tile_len)
        if n == 0:
            raise SantaError(1, "santa_tiled_workspace_size")
        workspace = alloc_workspace(n, q.device)
    st = library().santa_decode_tiled(ctypes.byref(p), SAMPLERS[sampler], tile_len, _ptr(q), _ptr(K), _ptr(V),
                                      _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream),
                                      _ptr(sample_idx))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode_tiled")
    return out


def bernoulli_workspace_size(p: Params) -> int:
    return library().santa_bernoulli_workspace_size(ctypes.byref(p))


def santa_decode_bernoulli(q, K, V, S: int, n_samples: int, stratified: bool = True, variant: str = "systematic",
                           seed: int = 0, step: int = 0, out=None, nk: Optional[int] = None, kv_offsets=None,
                           S_per_seq=None, scale: float = 0.0, workspace=None, sample_idx=None, feature_counts=None,
                           stream=None) -> torch.Tensor:
    """santa_decode on Bernoulli qK^T scores with the mean group query;
    feature_counts, if given, is int32 [B, H_kv, d] (ones per feature)."""
    _check_tensors(q, K, V, out, kv_offsets, S_per_seq, sample_idx, feature_counts)
    p = make_params(q, K, S, seed, step, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(bernoulli_workspace_size(p), q.device)
    st = library().santa_decode_bernoulli(ctypes.byref(p), VARIANTS[variant], n_samples, int(bool(stratified)),
                                          _ptr(q), _ptr(K), _ptr(V), _ptr(out), _ptr(workspace), workspace.numel(),
                                          _stream(stream), _ptr(sample_idx), _ptr(feature_counts))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode_bernoulli")
    return out


def static_scratch_bytes() -> int:
    """SANTA_STATIC_SCRATCH_BYTES from include/santa.h: the largest workspace
    santa_decode_static can serve."""
    m = re.search(r"#define SANTA_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def static_warmup() -> None:
    """Loads santa_decode_static's fixed array on the current device (under
    lazy module loading its one allocation); call at startup."""
    st = library().santa_static_warmup()
    if st != SANTA_OK:
        raise SantaError(st, "santa_static_warmup")


def santa_decode_static(q, K, V, S: int, variant: str = "systematic", seed: int = 0, step: int = 0, out=None,
                        nk: Optional[int] = None, kv_offsets=None, S_per_seq=None, scale: float = 0.0,
                        sample_idx=None, stream=None) -> torch.Tensor:
    """santa_decode through the C entry point that allocates nothing: its
    workspace is the library's fixed device array (for callers that cannot
    allocate device memory; see include/santa.h).  `out` is the caller's; pass
    it to keep this call free of allocation on the Python side as well."""
    _check_tensors(q, K, V, out, kv_offsets, S_per_seq, sample_idx)
    p = make_params(q, K, S, seed, step, nk, kv_offsets, S_per_seq, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    st = library().santa_decode_static(ctypes.byref(p), VARIANTS[variant], _ptr(q), _ptr(K), _ptr(V), _ptr(out),
                                       _stream(stream), _ptr(sample_idx))
    if st != SANTA_OK:
        raise SantaError(st, "santa_decode_static")
    return out


def santa_dense_decode(q, K, V, out=None, nk=None, kv_offsets=None, scale: float = 0.0, workspace=None,
                       stream=None) -> torch.Tensor:
    """Exact decode attention (this library's split-KV comparator)."""
    _check_tensors(q, K, V, out, kv_offsets)
    p = make_params(q, K, 1, 0, 0, nk, kv_offsets, None, scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(dense_workspace_size(p), q.device)
    st = library().santa_dense_decode(ctypes.byref(p), _ptr(q), _ptr(K), _ptr(V), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(stream))
    if st != SANTA_OK:
        raise SantaError(st, "santa_dense_decode")
    return out


class Decoder:
    """Reusable decode call for fixed shapes: holds the parameter block, the
    workspace and the output, so a step is one C-ABI call."""

    def __init__(self, q, K, V, S: int, variant: str = "systematic", seed: int = 0, nk=None, kv_offsets=None,
                 S_per_seq=None, scale: float = 0.0, dense: bool = False, sample_idx=None):
        _check_tensors(q, K, V, kv_offsets, S_per_seq, sample_idx)
        self.q, self.K, self.V = q, K, V
        self.kv_offsets, self.S_per_seq, self.sample_idx = kv_offsets, S_per_seq, sample_idx
        self.dense = dense
        self.variant = VARIANTS[variant]
        self.p = make_params(q, K, S, seed, 0, nk, kv_offsets, S_per_seq, scale)
        n = dense_workspace_size(self.p) if dense else workspace_size(self.p)
        if n == 0:
            raise ValueError("invalid decode parameters")
        self.workspace = alloc_workspace(n, q.device)
        self.out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        self._args = None

    def score_pass(self, stream=None) -> None:
        """Only the score pass (stash and chunk statistics in the workspace)."""
        st = library().santa_score_pass(ctypes.byref(self.p), _ptr(self.q), _ptr(self.K), _ptr(self.workspace),
                                        self.workspace.numel(), _stream(stream))
        if st != SANTA_OK:
            raise SantaError(st, "santa_score_pass")

    def profiled(self, events, step: int = 0, stream=None) -> torch.Tensor:
        """One step recording 4 torch.cuda.Event objects around the three stages
        (each event must have been recorded once so that it exists)."""
        if any(e.cuda_event == 0 for e in events):
            raise ValueError("record each event once before passing it (torch creates events lazily)")
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        self.p.step = step
        st = library().santa_decode_profiled(ctypes.byref(self.p), self.variant, _ptr(self.q), _ptr(self.K),
                                             _ptr(self.V), _ptr(self.out), _ptr(self.workspace),
                                             self.workspace.numel(), _stream(stream), _ptr(self.sample_idx), arr)
        if st != SANTA_OK:
            raise SantaError(st, "santa_decode_profiled")
        return self.out

    def __call__(self, step: int = 0, stream=None) -> torch.Tensor:
        lib = library()
        self.p.step = step
        if self.dense:
            st = lib.santa_dense_decode(ctypes.byref(self.p), _ptr(self.q), _ptr(self.K), _ptr(self.V),
                                        _ptr(self.out), _ptr(self.workspace), self.workspace.numel(),
                                        _stream(stream))
        else:
            st = lib.santa_decode(ctypes.byref(self.p), self.variant, _ptr(self.q), _ptr(self.K), _ptr(self.V),
                                  _ptr(self.out), _ptr(self.workspace), self.workspace.numel(), _stream(stream),
                                  _ptr(self.sample_idx))
        if st != SANTA_OK:
            raise SantaError(st, "santa_dense_decode" if self.dense else "santa_decode")
        return self.out
