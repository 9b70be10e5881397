"""GPU parity of the dense split-KV comparator (Eq. 1 of "Stochastic Sparse
Attention for Memory-Bound Inference") against the oracle's exact softmax.V."""
import numpy as np
import pytest
import torch

import oracle
import synth
import stochastic_sparse_decode_split_gb300 as santa

pytestmark = pytest.mark.gpu
TOL = 1e-4   # relative L2 per head; fp32 accumulation over <= 2^21 keys


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.library()


def dense_gpu(inp):
    t = synth.to_torch(inp)
    ragged = inp.wl.ragged is not None
    out = santa.santa_dense_decode(t["q"], t["K"], t["V"], nk=int(inp.nk_per_seq.max()) if ragged else None,
                                   kv_offsets=t["kv_offsets"] if ragged else None)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def check(inp, tol=TOL):
    ref = oracle.dense(oracle.Problem.from_inputs(inp))
    out = dense_gpu(inp)
    rel = np.linalg.norm(out - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() <= tol, f"max relative L2 {rel.max():.3e}"
    return rel.max()


@pytest.mark.parametrize("B,H,Hkv,d,nk,dtype", [
    (1, 1, 1, 64, 256, "fp32"),
    (2, 8, 2, 128, 3000, "bf16"),
    (1, 14, 2, 128, 1000, "fp16"),
    (1, 16, 2, 64, 1, "bf16"),
    (1, 6, 2, 128, 2049, "fp32"),
    (2, 10, 2, 64, 777, "bf16"),
    (64, 8, 2, 128, 40, "bf16"),      # many short pieces in every CTA's range
    (3, 32, 8, 128, 16, "fp16"),      # one block per piece
    (1, 8, 1, 128, 20000, "bf16"),    # one piece across many CTAs
])
def test_dense_grid(B, H, Hkv, d, nk, dtype):
    check(synth.generate(synth.Workload("dense", B, H, Hkv, d, nk, dtype, 1, "systematic"), 3))


def test_dense_ragged():
    wl = synth.Workload("dense_ragged", 5, 8, 2, 128, 2000, "bf16", 1, "systematic", ragged=(1, 2000))
    check(synth.generate(wl, 8))
    wl = synth.Workload("dense_ragged_short", 33, 16, 4, 64, 300, "fp16", 1, "systematic", ragged=(1, 300))
    check(synth.generate(wl, 9))


def test_dense_full_size_llama32k():
    print("llama32k dense max rel L2:", check(synth.generate(synth.llama32k(), 0)))


def test_santa_tracks_dense_at_large_budget():
    """With S = 4096 stratified draws the estimate is close to exact attention."""
    inp = synth.generate(synth.Workload("conv", 1, 8, 2, 128, 4096, "bf16", 4096, "stratified"), 2)
    t = synth.to_torch(inp)
    est = santa.santa_decode(t["q"], t["K"], t["V"], S=4096, variant="stratified").double().cpu().numpy()
    ref = dense_gpu(inp)
    rel = np.linalg.norm(est - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert rel.max() < 0.1
