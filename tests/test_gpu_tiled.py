"""GPU parity of the tile samplers S2ANTA-prop and S2ANTA-flash (through the
C ABI) against the CPU oracle ("Stochastic Sparse Attention for
Memory-Bound Inference", App. O, Alg. 2-5; App. P, Alg. 6-8).

Contract: on the same generated inputs and seed, per head and tile,
- prop budgets equal the oracle's, or (where a fractional part is within
  1e-5 of an integer or of another tile's, so float rounding of the tile
  masses decides) form another valid largest-remainder allocation;
- inside tiles with equal budgets every key's count equals the oracle's,
  except draws within 1e-6 (probability units) of an interval end, which
  may move to the neighbouring key;
- outputs agree within 1e-4 relative L2 per head with the oracle's estimate
  (or, where counts differ, with the oracle's weights applied to the GPU's
  own counts).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import stochastic_sparse_decode_split_gb300 as santa

pytestmark = pytest.mark.gpu
BAND = 1e-6
TIE = 1e-5
OUT_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.library()


def run_tiled(inp, sampler, tile_len, seed=0, step=0):
    t = synth.to_torch(inp)
    B, H, _ = inp.q.shape
    ragged = inp.wl.ragged is not None
    nk = int(inp.nk_per_seq.max()) if ragged else None
    p = santa.make_params(t["q"], t["K"], inp.S_max, seed, step, nk, t["kv_offsets"] if ragged else None,
                          t["S_per_seq"])
    nd = santa.tiled_max_draws(p, sampler, tile_len)
    assert nd > 0
    idx = torch.full((B, H, nd), -7, dtype=torch.int32, device="cuda")
    out = santa.santa_decode_tiled(t["q"], t["K"], t["V"], S=inp.S_max, sampler=sampler, tile_len=tile_len,
                                   seed=seed, step=step, nk=nk, kv_offsets=t["kv_offsets"] if ragged else None,
                                   S_per_seq=t["S_per_seq"], sample_idx=idx)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), idx.cpu().numpy()


def tile_weights(P, b, h, tile_len):
    """W_t / Z from the oracle's tile statistics (App. O, Alg. 4)."""
    m, l = oracle.tile_stats(P, b, h, tile_len)
    W = np.exp(m - m.max()) * l
    return W / W.sum()


def values(P, b, h):
    B, H, Hkv, d = P.shape
    off = P.kv_offsets
    return synth.storage_to_f64(P.V[off[b]:off[b + 1], h // (H // Hkv)], P.dtype)


def check_head(P, inp, b, h, sampler, tile_len, seed, out_bh, idx_bh, step=0):
    nk = int(inp.nk_per_seq[b])
    S_b = inp.S_of(b)
    T = -(-nk // tile_len)
    est, c_o, delta, St_o = oracle.tiled_head(P, b, h, sampler, S_b, tile_len, seed, step)
    n_draws = S_b if sampler == "prop" else T * int(St_o[0])
    row = idx_bh
    assert np.all(row[n_draws:] == -1), "unused sample_idx entries are -1"
    drawn = row[:n_draws]
    assert np.all((drawn >= 0) & (drawn < nk))
    # draws come tile by tile, keys increasing inside a tile
    assert np.all(np.diff(drawn) >= 0)
    c_g = np.bincount(drawn, minlength=nk)
    St_g = np.add.reduceat(c_g, np.arange(0, nk, tile_len))
    w = tile_weights(P, b, h, tile_len)
    stats = {"tiles": T, "budget_diff": 0, "count_diff": 0}
    if sampler == "prop":
        assert St_g.sum() == S_b
        q = S_b * w
        fl = np.floor(q)
        diff = np.nonzero(St_g != St_o)[0]
        if diff.size:
            fr = q - fl
            for t in diff:
                assert fl[t] <= St_g[t] <= fl[t] + 1, (t, St_g[t], q[t])
                near = min(fr[t], 1.0 - fr[t]) < TIE or np.any(np.abs(np.delete(fr, t) - fr[t]) < TIE)
                assert near, f"budget of tile {t} differs away from a tie: gpu {St_g[t]} oracle {St_o[t]} q {q[t]}"
            stats["budget_diff"] = int(diff.size)
    else:
        assert np.all(St_g == St_o)
    same = np.repeat(St_g == St_o, tile_len)[:nk]
    bad = np.nonzero(same & (c_g != c_o))[0]
    for n in bad:   # a boundary draw moved to a neighbour: the oracle's draw there lies in the band
        near = [k for k in (n - 1, n, n + 1) if 0 <= k < nk and 0 <= delta[k] < BAND]
        assert near, f"(b={b}, h={h}) key {n}: gpu {c_g[n]} oracle {c_o[n]} away from an interval end"
    stats["count_diff"] = int(bad.size)
    if stats["count_diff"] == 0 and stats["budget_diff"] == 0:
        ref = est
    else:
        V = values(P, b, h)
        tile_of = np.arange(nk) // tile_len
        wt = np.full(nk, 1.0 / S_b) if sampler == "prop" else w[tile_of] / St_o[0]
        ref = (c_g * wt) @ V
    rel = np.linalg.norm(out_bh - ref) / max(np.linalg.norm(ref), 1e-30)
    assert rel <= OUT_TOL, f"(b={b}, h={h}) relative L2 {rel:.3e}"
    return stats


def check_all(inp, sampler, tile_len, seed=0, step=0):
    out, idx = run_tiled(inp, sampler, tile_len, seed, step)
    P = oracle.Problem.from_inputs(inp)
    B, H, _ = inp.q.shape
    tot = {"budget_diff": 0, "count_diff": 0}
    for b in range(B):
        for h in range(H):
            s = check_head(P, inp, b, h, sampler, tile_len, seed, out[b, h], idx[b, h], step)
            for k in tot:
                tot[k] += s[k]
    return tot


def wl(name, B, H, Hkv, d, nk, dtype, S, **kw):
    return synth.Workload(name, B, H, Hkv, d, nk, dtype, S, "systematic", **kw)


@pytest.mark.parametrize("sampler", ["prop", "flash"])
@pytest.mark.parametrize("tile_len", [16, 64])
def test_tiny(sampler, tile_len):
    inp = synth.generate(synth.tiny("systematic"), 0)
    for seed in range(6):
        tot = check_all(inp, sampler, tile_len, seed)
        assert tot["budget_diff"] == 0 and tot["count_diff"] == 0


@pytest.mark.parametrize("sampler", ["prop", "flash"])
@pytest.mark.parametrize("case", [
    ("b2_bf16", 2, 8, 2, 128, 3000, "bf16", 64, 256),
    ("b1_fp16_d64", 1, 16, 4, 64, 1500, "fp16", 128, 64),
    ("fp32_g8", 1, 16, 2, 128, 777, "fp32", 40, 128),
    ("bf16_tile1024", 1, 8, 8, 128, 5000, "bf16", 300, 1024),
    ("few_samples", 1, 4, 1, 64, 4000, "bf16", 8, 32),   # prop: most tiles get no sample
    ("many_tiles", 1, 4, 1, 64, 8192, "bf16", 300, 16),  # 512 tiles: prop sorts the fractional parts
    ("tile48", 1, 4, 1, 64, 3000, "bf16", 100, 48),      # 3 chunks per tile: the general budget and merge
    ("tiles_2048", 1, 4, 1, 64, 32768, "bf16", 600, 16),  # 2048 tiles: past the fast path's 1024
])
def test_parity(sampler, case):
    name, B, H, Hkv, d, nk, dtype, S, L = case
    inp = synth.generate(wl(name, B, H, Hkv, d, nk, dtype, S), 3)
    for seed in (0, 7):
        check_all(inp, sampler, L, seed, step=seed)


@pytest.mark.parametrize("sampler", ["prop", "flash"])
def test_ragged(sampler):
    inp = synth.generate(synth.Workload("ragged_small", 5, 8, 2, 128, 2600, "bf16", 64, "stratified",
                                        ragged=(17, 2600), S_rule="max64_nk_div128"), 4)
    check_all(inp, sampler, 128, seed=2)


def test_deterministic_output_bits():
    inp = synth.generate(wl("det", 1, 8, 2, 128, 4000, "bf16", 256), 5)
    for sampler in ("prop", "flash"):
        o1, i1 = run_tiled(inp, sampler, 256, seed=1)
        o2, i2 = run_tiled(inp, sampler, 256, seed=1)
        assert np.array_equal(o1, o2) and np.array_equal(i1, i2)


@pytest.mark.parametrize("sampler,S", [("prop", 128), ("flash", 2048)])
def test_llama_32k_sampled_heads(sampler, S):
    """The pages' operating points (Sec. 3.4): prop at S = 128, flash at
    S = 2048, Llama-3.1-8B layer at 32K, tiles of 256 keys; four heads checked
    against the oracle."""
    inp = synth.generate(synth.llama32k(32768, S, "systematic"), 0)
    out, idx = run_tiled(inp, sampler, 256, seed=0)
    P = oracle.Problem.from_inputs(inp)
    for h in (0, 5, 18, 31):
        check_head(P, inp, 0, h, sampler, 256, 0, out[0, h], idx[0, h])


def test_invalid_tile_lengths_are_rejected():
    inp = synth.generate(wl("bad", 1, 4, 1, 64, 300, "bf16", 16), 0)
    t = synth.to_torch(inp)
    p = santa.make_params(t["q"], t["K"], 16)
    for L in (0, 8, 24, 2048):
        assert santa.tiled_workspace_size(p, "prop", L) == 0
        with pytest.raises(santa.SantaError):
            santa.santa_decode_tiled(t["q"], t["K"], t["V"], S=16, sampler="prop", tile_len=L)


@pytest.mark.parametrize("sampler", ["prop", "flash"])
def test_device_flags_bad_ragged_metadata(sampler):
    """A sequence longer than the stated bound or a budget out of range is
    flagged in the workspace error word; its heads come out zero with their
    sample_idx rows -1, and the other sequences are unaffected."""
    wl = synth.Workload("flags_t", 3, 4, 2, 128, 600, "bf16", 32, "systematic", ragged=(600, 600))
    inp = synth.generate(wl, 1)
    t = synth.to_torch(inp)
    S_per = torch.tensor([32, 0, 16], dtype=torch.int32, device="cuda")    # S_1 = 0 is out of range
    offs = torch.tensor([0, 600, 1200, 1800], dtype=torch.int64, device="cuda")
    p = santa.make_params(t["q"], t["K"], 32, nk=500, kv_offsets=offs, S_per_seq=S_per)   # bound 500 < 600
    ws = santa.alloc_workspace(santa.tiled_workspace_size(p, sampler, 64), "cuda")
    out = santa.santa_decode_tiled(t["q"], t["K"], t["V"], S=32, sampler=sampler, tile_len=64, nk=500,
                                   kv_offsets=offs, S_per_seq=S_per, workspace=ws)
    code = santa.get_error(ws)
    assert code & 1 and code & 2
    assert torch.count_nonzero(out) == 0
    offs_ok = torch.tensor([0, 600, 1000, 1800], dtype=torch.int64, device="cuda")
    p = santa.make_params(t["q"], t["K"], 32, nk=800, kv_offsets=offs_ok, S_per_seq=S_per)
    nd = santa.tiled_max_draws(p, sampler, 64)
    idx = torch.full((3, 4, nd), -7, dtype=torch.int32, device="cuda")
    out = santa.santa_decode_tiled(t["q"], t["K"], t["V"], S=32, sampler=sampler, tile_len=64, nk=800,
                                   kv_offsets=offs_ok, S_per_seq=S_per, sample_idx=idx)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[0]) > 0 and torch.count_nonzero(out[2]) > 0
    assert bool(torch.all(idx[1] == -1)) and bool(torch.all(idx[0] != -7))
