"""Seeded synthetic decode-step workloads.

This module produces the input bytes that both the CUDA path and the CPU
oracle read.  It holds none of the attention method's arithmetic: it draws
Gaussian query/key/value tensors, plants heavy-hitter keys, rounds to the
storage dtype and widens storage bytes back to float64 for reading.

Workload recipe (all draws from one ``numpy.random.PCG64(data_seed)`` stream,
in this order):

1. ``q``    : standard normal, shape ``[B, H, d]`` (float32), rounded to dtype.
2. ragged   : per-sequence key counts ``nk_b`` uniform on the stated range.
3. per sequence ``b`` in order:
   ``K_b``, ``V_b`` standard normal ``[nk_b, H_kv, d]`` (float32), then per KV
   head a set of planted key positions drawn without replacement and their
   noise rows.  A planted key is ``2.5 * q_mean + 0.5 * N(0, 1)`` where
   ``q_mean`` is the mean of the (rounded) query vectors of that KV head's
   query group (the "tiny" workload instead plants ``3 * q / |q| * sqrt(d)``).
4. ``K`` and ``V`` are rounded to the storage dtype (round to nearest even).

The decode geometry follows "Stochastic Sparse Attention for Memory-Bound
Inference", App. Q (sequence-major ``[nk, H_kv, d]`` caches, Gaussian
``randn`` inputs, Llama-3.1-8B GQA shape), with the heavy hitters added so
that the post-softmax distribution is peaked the way real attention is.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

DTYPES = ("bf16", "fp16", "fp32")
VARIANTS = ("iid", "stratified", "systematic")


@dataclasses.dataclass
class Workload:
    """A named decode-step configuration (shapes, dtype, budget, variant)."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    nk: int                     # keys per sequence (uniform) or the maximum (ragged)
    dtype: str
    S: int                      # sample budget (maximum when ``S_rule`` is set)
    variant: str
    plant_frac: float = 0.01
    tiny_plant: int = 0         # >0: plant this many keys at 3*q/|q|*sqrt(d)
    ragged: Optional[tuple] = None   # (lo, hi) inclusive range of nk_b
    S_rule: Optional[str] = None     # "max64_nk_div128" for the ragged batch

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def tiny(variant: str = "systematic") -> Workload:
    return Workload("tiny_b1_h1_d64_nk256_fp32_S16", 1, 1, 1, 64, 256, "fp32", 16,
                    variant, plant_frac=0.0, tiny_plant=4)


def llama32k(nk: int = 32768, S: int = 256, variant: str = "systematic",
             batch: int = 1) -> Workload:
    return Workload(f"llama3.1-8b_b{batch}_h32_kv8_d128_nk{nk}_bf16_S{S}_{variant}", batch, 32, 8,
                    128, nk, "bf16", S, variant)


def qwen_batched(nk: int = 32768, batch: int = 16) -> Workload:
    return Workload(f"qwen2.5-7b_b{batch}_h28_kv4_d128_nk{nk}_fp16_S256_systematic", batch, 28,
                    4, 128, nk, "fp16", 256, "systematic", plant_frac=0.005)


def ragged(batch: int = 64, lo: int = 1024, hi: int = 32768) -> Workload:
    return Workload(f"ragged_b{batch}_h32_kv8_d128_nk{lo}-{hi}_bf16_Smax64nk128_stratified", batch, 32, 8,
                    128, hi, "bf16", max(64, hi // 128), "stratified",
                    ragged=(lo, hi), S_rule="max64_nk_div128")


def sweep_points():
    """nk x S x variant grid on the Llama-3.1-8B layer shape."""
    for nk in (4096, 8192, 16384, 32768, 65536, 131072):
        for S in (64, 256, 1024):
            for variant in ("stratified", "systematic"):
                yield llama32k(nk=nk, S=S, variant=variant)


# ---------------------------------------------------------------------------
# dtype rounding / widening (storage conversions only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> storage array (uint16 bits for bf16, float16, float32)."""
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "fp16":
        return np.asarray(x, dtype=np.float32).astype(np.float16)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float32)
    raise ValueError(dtype)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a).astype(np.float64)


def storage_to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return storage_to_f64(a, dtype).astype(np.float32)


# ---------------------------------------------------------------------------
# generation
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Inputs:
    """Storage-dtype arrays for one decode step (host memory)."""

    wl: Workload
    q: np.ndarray            # [B, H, d]
    K: np.ndarray            # [sum nk_b, H_kv, d]
    V: np.ndarray            # [sum nk_b, H_kv, d]
    kv_offsets: np.ndarray   # int64 [B + 1]
    S_per_seq: Optional[np.ndarray]  # int32 [B] or None
    planted: list            # per (b, kvh): sorted planted positions (int64)

    @property
    def nk_per_seq(self) -> np.ndarray:
        return np.diff(self.kv_offsets)

    @property
    def S_max(self) -> int:
        return int(self.S_per_seq.max()) if self.S_per_seq is not None else self.wl.S

    def S_of(self, b: int) -> int:
        return int(self.S_per_seq[b]) if self.S_per_seq is not None else self.wl.S


def generate(wl: Workload, data_seed: int = 0) -> Inputs:
    rng = np.random.Generator(np.random.PCG64(data_seed))
    B, H, Hkv, d = wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    G = H // Hkv
    q_store = round_to_storage(rng.standard_normal((B, H, d), dtype=np.float32), wl.dtype)
    q32 = storage_to_f32(q_store, wl.dtype)

    if wl.ragged is not None:
        lo, hi = wl.ragged
        nks = rng.integers(lo, hi, size=B, endpoint=True).astype(np.int64)
    else:
        nks = np.full(B, wl.nk, dtype=np.int64)
    offsets = np.zeros(B + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(nks)
    total = int(offsets[-1])

    store_dtype = np.uint16 if wl.dtype == "bf16" else (np.float16 if wl.dtype == "fp16" else np.float32)
    K = np.empty((total, Hkv, d), dtype=store_dtype)
    V = np.empty((total, Hkv, d), dtype=store_dtype)
    planted = []
    for b in range(B):
        nk_b = int(nks[b])
        Kb = rng.standard_normal((nk_b, Hkv, d), dtype=np.float32)
        Vb = rng.standard_normal((nk_b, Hkv, d), dtype=np.float32)
        for kvh in range(Hkv):
            if wl.tiny_plant:
                n_plant = wl.tiny_plant
            else:
                n_plant = int(np.floor(wl.plant_frac * nk_b + 0.5))
            n_plant = min(n_plant, nk_b)
            pos = np.sort(rng.choice(nk_b, size=n_plant, replace=False)) if n_plant else np.zeros(0, np.int64)
            group_q = q32[b, kvh * G:(kvh + 1) * G]
            if wl.tiny_plant:
                qv = group_q.mean(axis=0)
                row = (3.0 * qv / np.linalg.norm(qv) * np.sqrt(d)).astype(np.float32)
                Kb[pos, kvh] = row
            elif n_plant:
                noise = rng.standard_normal((n_plant, d), dtype=np.float32)
                q_mean = group_q.mean(axis=0)
                Kb[pos, kvh] = (np.float32(2.5) * q_mean + np.float32(0.5) * noise).astype(np.float32)
            planted.append(pos.astype(np.int64))
        K[offsets[b]:offsets[b + 1]] = round_to_storage(Kb, wl.dtype)
        V[offsets[b]:offsets[b + 1]] = round_to_storage(Vb, wl.dtype)

    S_per_seq = None
    if wl.S_rule == "max64_nk_div128":
        S_per_seq = np.maximum(64, nks // 128).astype(np.int32)
    return Inputs(wl, q_store, K, V, offsets, S_per_seq, planted)


def thrash_bytes_default() -> int:
    """Size of the buffer written between timed iterations (well above a 129 MB L2)."""
    return 512 * 1024 * 1024


def to_torch(inp: Inputs, device="cuda"):
    """Copies the storage arrays to torch tensors on `device` (bytes unchanged):
    returns dict(q, K, V, kv_offsets, S_per_seq)."""
    import torch
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[inp.wl.dtype]

    def conv(a):
        if inp.wl.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    out = {"q": conv(inp.q), "K": conv(inp.K), "V": conv(inp.V),
           "kv_offsets": torch.from_numpy(inp.kv_offsets.copy()).to(device),
           "S_per_seq": None if inp.S_per_seq is None else torch.from_numpy(inp.S_per_seq.copy()).to(device)}
    return out
