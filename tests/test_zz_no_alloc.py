"""santa_decode_static: the decode entry point that allocates nothing.

Some callers cannot allocate device memory: a plug-in that its host framework
hands only tensors and a stream (the framework's pool owns the device memory),
or code that must not call cudaMalloc mid-run because it synchronises the
device and may fail once the pool has taken the rest of the GPU.  For them the
library keeps a fixed device array of SANTA_STATIC_SCRATCH_BYTES as the
workspace.  These tests check, through the C ABI, that two calls in a row give
the same draws and (within the fp32 reduction-order tolerance of the other
decode tests) the same outputs as santa_decode with a caller workspace, and
that a problem beyond the array is refused before any CUDA call.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import stochastic_sparse_decode_split_gb300 as santa

SANTA_ERR_SCRATCH_LIMIT = 6


def _params(**kw):
    p = santa.Params()
    p.batch, p.n_q_heads, p.n_kv_heads, p.head_dim = 1, 32, 8, 128
    p.dtype, p.nk, p.S, p.scale, p.seed, p.step = 0, 32768, 256, 0.0, 0, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_refuses_problems_beyond_the_array():
    """Host check, no GPU needed: the workspace it would need exceeds the array."""
    lib = santa.library()
    limit = santa.static_scratch_bytes()
    fits, too_big = _params(), _params(batch=2)
    assert 0 < santa.workspace_size(fits) <= limit < santa.workspace_size(too_big)
    vp = ctypes.c_void_p
    st = lib.santa_decode_static(ctypes.byref(too_big), 2, vp(256), vp(256), vp(256), vp(256), None, None)
    assert st == SANTA_ERR_SCRATCH_LIMIT
    assert b"SANTA_STATIC_SCRATCH_BYTES" in lib.santa_status_string(st)
    # invalid parameters keep santa_decode's statuses
    assert lib.santa_decode_static(ctypes.byref(_params(n_kv_heads=3)), 2, vp(256), vp(256), vp(256), vp(256),
                                   None, None) == 1
    # so do a bad variant, null or misaligned buffers: refused before any CUDA
    # call (no GPU in this test)
    assert lib.santa_decode_static(ctypes.byref(fits), 7, vp(256), vp(256), vp(256), vp(256), None, None) == 1
    assert lib.santa_decode_static(ctypes.byref(fits), 2, None, vp(256), vp(256), vp(256), None, None) == 1
    assert lib.santa_decode_static(ctypes.byref(fits), 2, vp(256), vp(264), vp(256), vp(256), None, None) == 1
    assert lib.santa_decode_static(ctypes.byref(fits), 2, vp(256), vp(256), vp(256), vp(256), None, vp(258)) == 1


def _case(name, B, H, Hkv, d, nk, dtype, S, variant, data_seed):
    inp = synth.generate(synth.Workload(name, B, H, Hkv, d, nk, dtype, S, variant), data_seed)
    return inp, synth.to_torch(inp)


@pytest.mark.gpu
def test_two_calls_match_santa_decode():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.static_warmup()
    cases = [  # a second call with another shape, dtype and variant: the array keeps the first call's contents
        (_case("static_a", 2, 8, 2, 128, 3000, "bf16", 64, "systematic", 11), "systematic", 5),
        (_case("static_b", 1, 16, 4, 64, 1500, "fp16", 128, "stratified", 12), "stratified", 6),
        # the motivating size: one Llama-3.1-8B layer at 32K keys, 256 systematic draws
        (_case("static_llama32k", 1, 32, 8, 128, 32768, "bf16", 256, "systematic", 13), "systematic", 7),
    ]
    for (inp, t), variant, seed in cases:
        B, H, d = inp.q.shape
        out_s = torch.full((B, H, d), float("nan"), dtype=torch.float32, device="cuda")
        idx_s = torch.full((B, H, inp.S_max), -7, dtype=torch.int32, device="cuda")
        santa.santa_decode_static(t["q"], t["K"], t["V"], S=inp.S_max, variant=variant, seed=seed, out=out_s,
                                  sample_idx=idx_s)
        idx_r = torch.full((B, H, inp.S_max), -7, dtype=torch.int32, device="cuda")
        out_r = santa.santa_decode(t["q"], t["K"], t["V"], S=inp.S_max, variant=variant, seed=seed,
                                   sample_idx=idx_r)
        torch.cuda.synchronize()
        assert np.array_equal(idx_s.cpu().numpy(), idx_r.cpu().numpy())
        np.testing.assert_allclose(out_s.cpu().numpy(), out_r.cpu().numpy(), rtol=1e-5, atol=1e-6)


@pytest.mark.gpu
def test_calls_after_warmup_allocate_nothing():
    """After santa_static_warmup, a call changes neither the device's free
    memory (cudaMemGetInfo) nor the torch pool."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.static_warmup()
    inp, t = _case("static_alloc", 1, 32, 8, 128, 32768, "bf16", 256, "systematic", 14)
    B, H, d = inp.q.shape
    out = torch.empty((B, H, d), dtype=torch.float32, device="cuda")
    santa.santa_decode_static(t["q"], t["K"], t["V"], S=256, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    pool0 = torch.cuda.memory_reserved()
    for seed in range(3):
        santa.santa_decode_static(t["q"], t["K"], t["V"], S=256, seed=seed, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_reserved() == pool0
    assert abs(free1 - free0) < (1 << 20), (free0, free1)
