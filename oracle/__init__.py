"""CPU oracle for SANTA / S2ANTA decode-step attention.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg are the only users; the product path never imports this
package.  It shares no code with the CUDA library: the arithmetic lives in
``santa_oracle.c`` (plain float64 C, built with gcc) and ``analysis.py``
(closed forms in numpy).  Both follow "Stochastic Sparse Attention for
Memory-Bound Inference" (Sec. 2, Eq. 1 and 4; Sec. 2.1; App. A; App. M; the
tile samplers S2ANTA-prop, App. O, and S2ANTA-flash, App. P).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(worked example, library routines, closed forms, invariants, Philox against
an independent implementation); ``tests/test_oracle_mutants.py`` plants
plausible mistakes in copies of ``santa_oracle.c`` (wrong index, sign,
constant, rounding rule, dropped term) and checks that each one fails a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsanta_oracle.so")
_SRC = os.path.join(_HERE, "santa_oracle.c")
_lock = threading.Lock()
_lib = None

DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp32": 2}
VARIANT_CODE = {"iid": 0, "stratified": 1, "systematic": 2}
SAMPLER_CODE = {"prop": 0, "flash": 1}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed).  Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(os.path.join(_HERE, "santa_oracle.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Problem(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("kv_offsets", ctypes.c_void_p),
        ("q", ctypes.c_void_p),
        ("K", ctypes.c_void_p),
        ("V", ctypes.c_void_p),
        ("scale", ctypes.c_double),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SANTA_ORACLE_LIB names another build of santa_oracle.c (the
            # mutation tests load deliberately broken copies through it)
            lib = ctypes.CDLL(os.environ.get("SANTA_ORACLE_LIB") or build())
            P = ctypes.POINTER(_Problem)
            vp, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64
            lib.santa_oracle_philox4x32_10.argtypes = [vp, vp, vp]
            lib.santa_oracle_philox4x32_10.restype = None
            lib.santa_oracle_uniform.argtypes = [u64, u32, u32, u32, u32]
            lib.santa_oracle_uniform.restype = ctypes.c_double
            lib.santa_oracle_thresholds.argtypes = [i32, i32, u64, u32, u32, u32, vp]
            lib.santa_oracle_thresholds.restype = None
            lib.santa_oracle_scores.argtypes = [P, i32, i32, vp, vp]
            lib.santa_oracle_tile_stats.argtypes = [P, i32, i32, i32, vp, vp]
            lib.santa_oracle_sample_head.argtypes = [P, i32, i32, i32, vp, vp, vp, vp]
            lib.santa_oracle_dense_head.argtypes = [P, i32, i32, vp]
            lib.santa_oracle_gather.argtypes = [P, i32, i32, i32, vp, vp]
            lib.santa_oracle_decode.argtypes = [P, i32, i32, vp, i32, u64, u32, vp, vp, vp, i32]
            lib.santa_oracle_dense.argtypes = [P, vp, i32]
            lib.santa_oracle_prop_budgets.argtypes = [i32, vp, i32, vp]
            lib.santa_oracle_store_elem.argtypes = [i32, ctypes.c_float, vp]
            lib.santa_oracle_store_elem.restype = None
            lib.santa_oracle_bernoulli_group.argtypes = [P, i32, i32, i32, i32, u64, u32, vp, vp]
            lib.santa_oracle_bernoulli_group.restype = ctypes.c_int
            lib.santa_oracle_tiled_head.argtypes = [P, i32, i32, i32, i32, i32, u64, u32, vp, vp, vp, vp, vp]
            lib.santa_oracle_tiled_decode.argtypes = [P, i32, i32, vp, i32, u64, u32, vp, i32]
            for fn in ("santa_oracle_scores", "santa_oracle_tile_stats", "santa_oracle_sample_head",
                       "santa_oracle_dense_head", "santa_oracle_gather", "santa_oracle_decode", "santa_oracle_dense",
                       "santa_oracle_prop_budgets", "santa_oracle_tiled_head", "santa_oracle_tiled_decode"):
                getattr(lib, fn).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class Problem:
    """Holds contiguous host arrays and the C struct that points at them."""

    def __init__(self, q, K, V, kv_offsets, dtype: str, n_kv_heads: int | None = None,
                 scale: float = 0.0):
        self.q = np.ascontiguousarray(q)
        self.K = np.ascontiguousarray(K)
        self.V = np.ascontiguousarray(V)
        self.kv_offsets = np.ascontiguousarray(kv_offsets, dtype=np.int64)
        B, H, d = self.q.shape
        Hkv = n_kv_heads if n_kv_heads is not None else self.K.shape[1]
        self.shape = (B, H, Hkv, d)
        self.c = _Problem(DTYPE_CODE[dtype], B, H, Hkv, d, _ptr(self.kv_offsets).value,
                          _ptr(self.q).value, _ptr(self.K).value, _ptr(self.V).value, float(scale))
        self.dtype = dtype

    @classmethod
    def from_inputs(cls, inp) -> "Problem":
        return cls(inp.q, inp.K, inp.V, inp.kv_offsets, inp.wl.dtype, inp.wl.n_kv_heads)

    def nk(self, b: int) -> int:
        return int(self.kv_offsets[b + 1] - self.kv_offsets[b])


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().santa_oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, h: int, step: int, r: int) -> float:
    return _load().santa_oracle_uniform(seed, b, h, step, r)


def thresholds(variant: str, S: int, seed: int, b: int, h: int, step: int = 0) -> np.ndarray:
    t = np.zeros(S, dtype=np.float64)
    _load().santa_oracle_thresholds(VARIANT_CODE[variant], S, seed, b, h, step, _ptr(t))
    return t


def scores(P: Problem, b: int, h: int):
    """(s, p): scaled scores and softmax probabilities of head (b, h)."""
    nk = P.nk(b)
    s = np.zeros(nk, np.float64)
    p = np.zeros(nk, np.float64)
    if _load().santa_oracle_scores(ctypes.byref(P.c), b, h, _ptr(s), _ptr(p)):
        raise ValueError("oracle scores: bad arguments")
    return s, p


def tile_stats(P: Problem, b: int, h: int, tile_len: int):
    T = -(-P.nk(b) // tile_len)
    m = np.zeros(T, np.float64)
    l = np.zeros(T, np.float64)
    if _load().santa_oracle_tile_stats(ctypes.byref(P.c), b, h, tile_len, _ptr(m), _ptr(l)):
        raise ValueError("oracle tile stats: bad arguments")
    return m, l


def sample_head(P: Problem, b: int, h: int, t: np.ndarray):
    """Inverse-CDF sampling of head (b, h) at explicit thresholds t (in [0, 1)).

    Returns (estimate [d], J [S], delta [S])."""
    t = np.ascontiguousarray(t, dtype=np.float64)
    S = t.shape[0]
    est = np.zeros(P.shape[3], np.float64)
    J = np.zeros(S, np.int32)
    delta = np.zeros(S, np.float64)
    if _load().santa_oracle_sample_head(ctypes.byref(P.c), b, h, S, _ptr(t), _ptr(est), _ptr(J),
                                        _ptr(delta)):
        raise ValueError("oracle sample: bad arguments")
    return est, J, delta


def gather(P: Problem, b: int, h: int, J) -> np.ndarray:
    """Eq. (4) for a given index multiset: (1/S) * sum_j V[J_j]."""
    J = np.ascontiguousarray(J, dtype=np.int32)
    est = np.zeros(P.shape[3], np.float64)
    if _load().santa_oracle_gather(ctypes.byref(P.c), b, h, J.shape[0], _ptr(J), _ptr(est)):
        raise ValueError("oracle gather: bad arguments")
    return est


def dense_head(P: Problem, b: int, h: int) -> np.ndarray:
    out = np.zeros(P.shape[3], np.float64)
    if _load().santa_oracle_dense_head(ctypes.byref(P.c), b, h, _ptr(out)):
        raise ValueError("oracle dense: bad arguments")
    return out


def decode(P: Problem, variant: str, S: int, seed: int, step: int = 0, S_per_seq=None,
           n_threads: int = 0):
    """Whole decode step.  Returns (est [B,H,d], J [B,H,S_stride], delta [B,H,S_stride])."""
    B, H, _, d = P.shape
    Sp = None if S_per_seq is None else np.ascontiguousarray(S_per_seq, dtype=np.int32)
    S_stride = int(Sp.max()) if Sp is not None else S
    est = np.zeros((B, H, d), np.float64)
    J = np.zeros((B, H, S_stride), np.int32)
    delta = np.zeros((B, H, S_stride), np.float64)
    rc = _load().santa_oracle_decode(ctypes.byref(P.c), VARIANT_CODE[variant], S, _ptr(Sp), S_stride,
                                     seed, step, _ptr(est), _ptr(J), _ptr(delta), n_threads)
    if rc:
        raise ValueError("oracle decode: bad arguments")
    return est, J, delta


def dense(P: Problem, n_threads: int = 0) -> np.ndarray:
    B, H, _, d = P.shape
    out = np.zeros((B, H, d), np.float64)
    if _load().santa_oracle_dense(ctypes.byref(P.c), _ptr(out), n_threads):
        raise ValueError("oracle dense: bad arguments")
    return out


def decode_head(P: Problem, variant: str, S: int, seed: int, b: int, h: int, step: int = 0):
    """One head of a decode step (for sampled checks at full size)."""
    return sample_head(P, b, h, thresholds(variant, S, seed, b, h, step))


def prop_budgets(W, S: int) -> np.ndarray:
    """Largest-remainder budgets of App. O, Alg. 4 for tile masses W."""
    W = np.ascontiguousarray(W, dtype=np.float64)
    St = np.zeros(W.shape[0], np.int32)
    if _load().santa_oracle_prop_budgets(W.shape[0], _ptr(W), S, _ptr(St)):
        raise ValueError("oracle prop budgets: bad arguments")
    return St


def tiled_head(P: Problem, b: int, h: int, sampler: str, S: int, tile_len: int, seed: int, step: int = 0,
               a0=None):
    """One head through S2ANTA-prop or S2ANTA-flash.

    Returns (estimate [d], counts [nk_b], delta [nk_b], budgets [T])."""
    nk = P.nk(b)
    T = -(-nk // tile_len)
    a = None if a0 is None else np.ascontiguousarray(a0, dtype=np.float64)
    if a is not None and a.shape[0] < T:
        raise ValueError("a0 needs one offset per tile")
    est = np.zeros(P.shape[3], np.float64)
    counts = np.zeros(nk, np.int32)
    delta = np.zeros(nk, np.float64)
    St = np.zeros(T, np.int32)
    if _load().santa_oracle_tiled_head(ctypes.byref(P.c), b, h, SAMPLER_CODE[sampler], S, tile_len, seed, step,
                                       _ptr(a), _ptr(est), _ptr(counts), _ptr(delta), _ptr(St)):
        raise ValueError("oracle tiled head: bad arguments")
    return est, counts, delta, St


def tiled_decode(P: Problem, sampler: str, S: int, tile_len: int, seed: int, step: int = 0, S_per_seq=None,
                 n_threads: int = 0) -> np.ndarray:
    """Whole step of a tile sampler: estimate [B, H, d]."""
    B, H, _, d = P.shape
    Sp = None if S_per_seq is None else np.ascontiguousarray(S_per_seq, dtype=np.int32)
    est = np.zeros((B, H, d), np.float64)
    if _load().santa_oracle_tiled_decode(ctypes.byref(P.c), SAMPLER_CODE[sampler], S, _ptr(Sp), tile_len, seed,
                                         step, _ptr(est), n_threads):
        raise ValueError("oracle tiled decode: bad arguments")
    return est


_STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32}


def store_elem(dtype: str, x: float):
    """fp32 x rounded to the storage dtype (bits for bf16 / fp16)."""
    out = np.zeros(1, _STORAGE[dtype])
    _load().santa_oracle_store_elem(DTYPE_CODE[dtype], float(x), _ptr(out))
    return out[0]


def bernoulli_group(P: Problem, b: int, kvh: int, nsamp: int, stratified: bool, seed: int, step: int = 0):
    """Bernoulli qK^T, mean group query (App. C.2): (q~ [G, d] in storage
    dtype, counts [d])."""
    B, H, Hkv, d = P.shape
    qt = np.zeros((H // Hkv, d), _STORAGE[P.dtype])
    counts = np.zeros(d, np.int32)
    if _load().santa_oracle_bernoulli_group(ctypes.byref(P.c), b, kvh, nsamp, int(stratified), seed, step,
                                            _ptr(qt), _ptr(counts)):
        raise ValueError("oracle bernoulli: bad arguments")
    return qt, counts


def bernoulli_problem(P: Problem, nsamp: int, stratified: bool, seed: int, step: int = 0):
    """The problem with every query replaced by its Bernoulli effective query
    (App. C.2, Eq. 13), and the per-group feature counts [B, Hkv, d]."""
    B, H, Hkv, d = P.shape
    G = H // Hkv
    q = np.array(P.q, copy=True)
    counts = np.zeros((B, Hkv, d), np.int32)
    for b in range(B):
        for k in range(Hkv):
            qt, c = bernoulli_group(P, b, k, nsamp, stratified, seed, step)
            q[b, k * G:(k + 1) * G] = qt.view(q.dtype).reshape(G, d)
            counts[b, k] = c
    return Problem(q, P.K, P.V, P.kv_offsets, P.dtype, Hkv), counts
