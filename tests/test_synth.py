"""The synthetic inputs follow the stated recipe (CPU): the decode geometry of
the paper's measurements (App. Q: sequence-major caches, Gaussian inputs),
planted heavy-hitter keys, ragged lengths and per-sequence budgets, storage
rounding, and determinism in the data seed."""
import numpy as np

import synth


def test_planted_keys_count_and_construction():
    inp = synth.generate(synth.llama32k(32768, 256, "systematic"), 0)
    wl = inp.wl
    G = wl.n_q_heads // wl.n_kv_heads
    q = synth.storage_to_f64(inp.q, wl.dtype)
    for kvh in range(wl.n_kv_heads):
        pos = inp.planted[kvh]
        assert pos.size == 328                      # floor(0.01 * 32768 + 0.5)
        assert np.unique(pos).size == pos.size and pos.min() >= 0 and pos.max() < 32768
        rows = synth.storage_to_f64(inp.K[pos, kvh], wl.dtype)
        resid = rows - 2.5 * q[0, kvh * G:(kvh + 1) * G].mean(axis=0)
        assert abs(resid.mean()) < 0.02 and abs(resid.std() - 0.5) < 0.02   # 0.5 N(0, 1) noise
        others = np.setdiff1d(np.arange(4096), pos)
        plain = synth.storage_to_f64(inp.K[others, kvh], wl.dtype)
        assert abs(plain.mean()) < 0.01 and abs(plain.std() - 1.0) < 0.01


def test_planted_keys_carry_most_of_the_attention():
    inp = synth.generate(synth.llama32k(8192, 256, "systematic"), 0)
    wl = inp.wl
    G = wl.n_q_heads // wl.n_kv_heads
    q = synth.storage_to_f64(inp.q, wl.dtype)[0]
    K = synth.storage_to_f64(inp.K, wl.dtype)
    for h in (0, 13):
        s = K[:, h // G] @ q[h] / np.sqrt(wl.head_dim)
        p = np.exp(s - s.max())
        p /= p.sum()
        assert p[inp.planted[h // G]].sum() > 0.5


def test_qwen_shape_and_plant_rate():
    wl = synth.qwen_batched(nk=4096, batch=2)
    inp = synth.generate(wl, 1)
    assert inp.q.shape == (2, 28, 128) and inp.K.shape == (2 * 4096, 4, 128) and inp.K.dtype == np.float16
    assert all(p.size == 20 for p in inp.planted)   # floor(0.005 * 4096 + 0.5)


def test_ragged_lengths_and_budgets():
    inp = synth.generate(synth.ragged(batch=12, lo=100, hi=3000), 3)
    nk = inp.nk_per_seq
    assert nk.min() >= 100 and nk.max() <= 3000 and np.unique(nk).size > 8
    assert np.array_equal(inp.kv_offsets, np.concatenate([[0], np.cumsum(nk)]))
    assert np.array_equal(inp.S_per_seq, np.maximum(64, nk // 128))
    assert inp.S_max == int(inp.S_per_seq.max())


def test_storage_rounding_is_round_to_nearest_even():
    inp = synth.generate(synth.Workload("r", 1, 2, 1, 64, 300, "bf16", 8, "systematic"), 5)
    x = synth.bf16_bits_to_f64(inp.K.ravel()).astype(np.float32)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(x), inp.K.ravel())   # bf16 values survive a round trip


def test_deterministic_in_the_data_seed():
    wl = synth.Workload("det", 2, 4, 2, 64, 500, "fp16", 16, "systematic")
    a, b, c = synth.generate(wl, 7), synth.generate(wl, 7), synth.generate(wl, 8)
    assert np.array_equal(a.K, b.K) and np.array_equal(a.V, b.V) and np.array_equal(a.q, b.q)
    assert not np.array_equal(a.K, c.K)
