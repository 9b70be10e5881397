"""GPU parity of Bernoulli qK^T with the mean group query (through the C ABI)
against the CPU oracle ("Stochastic Sparse Attention for Memory-Bound
Inference", Sec. 5.1, App. C.2, Eq. 10-13).

Contract: the per-feature counts and the effective queries (cache dtype bits)
equal the oracle's exactly; the decode that follows matches the oracle's
decode on those queries as santa_decode does on plain ones (index-exact
outside the 1e-6 boundary band, outputs within 1e-3 relative L2).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import stochastic_sparse_decode_split_gb300 as santa

pytestmark = pytest.mark.gpu
BAND = 1e-6
OUT_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.library()


def run(inp, nsamp, stratified, variant, seed=0, step=0):
    t = synth.to_torch(inp)
    B, H, d = inp.q.shape
    Hkv = inp.wl.n_kv_heads
    ragged = inp.wl.ragged is not None
    nk = int(inp.nk_per_seq.max()) if ragged else None
    offs = t["kv_offsets"] if ragged else None
    p = santa.make_params(t["q"], t["K"], inp.S_max, seed, step, nk, offs, t["S_per_seq"])
    ws = santa.alloc_workspace(santa.bernoulli_workspace_size(p), "cuda")
    idx = torch.full((B, H, inp.S_max), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hkv, d), -7, dtype=torch.int32, device="cuda")
    out = santa.santa_decode_bernoulli(t["q"], t["K"], t["V"], S=inp.S_max, n_samples=nsamp, stratified=stratified,
                                       variant=variant, seed=seed, step=step, nk=nk, kv_offsets=offs,
                                       S_per_seq=t["S_per_seq"], workspace=ws, sample_idx=idx, feature_counts=cnt)
    torch.cuda.synchronize()
    off = -(-santa.workspace_size(p) // 256) * 256
    es = 4 if inp.wl.dtype == "fp32" else 2
    qt = ws[off:off + B * H * d * es].cpu().numpy().view(np.float32 if es == 4 else np.uint16).reshape(B, H, d)
    return out.double().cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy(), qt


def check(inp, nsamp, stratified, variant, seed=0, step=0):
    out, idx, cnt, qt = run(inp, nsamp, stratified, variant, seed, step)
    P = oracle.Problem.from_inputs(inp)
    Pb, counts = oracle.bernoulli_problem(P, nsamp, stratified, seed, step)
    np.testing.assert_array_equal(cnt, counts)
    np.testing.assert_array_equal(qt.view(Pb.q.dtype), Pb.q)
    est, J, delta = oracle.decode(Pb, variant, inp.wl.S, seed, step, S_per_seq=inp.S_per_seq)
    B, H, _ = inp.q.shape
    n_diff = 0
    for b in range(B):
        S_b = inp.S_of(b)
        for h in range(H):
            Jg, Jo, dl = idx[b, h, :S_b], J[b, h, :S_b], delta[b, h, :S_b]
            assert not np.any((dl > BAND) & (Jg != Jo)), (b, h)
            n_diff += int((Jg != Jo).sum())
            ref = est[b, h] if np.array_equal(Jg, Jo) else oracle.gather(Pb, b, h, Jg)
            rel = np.linalg.norm(out[b, h] - ref) / max(np.linalg.norm(ref), 1e-30)
            assert rel <= OUT_TOL, (b, h, rel)
    return counts, n_diff


@pytest.mark.parametrize("stratified", [True, False])
@pytest.mark.parametrize("case", [
    ("b2_bf16", 2, 8, 2, 128, 3000, "bf16", 64, "systematic", 4),
    ("fp16_d64", 1, 16, 4, 64, 1500, "fp16", 128, "stratified", 8),
    ("fp32_g8", 1, 16, 2, 128, 700, "fp32", 32, "iid", 2),
])
def test_parity(case, stratified):
    name, B, H, Hkv, d, nk, dtype, S, variant, nsamp = case
    inp = synth.generate(synth.Workload(name, B, H, Hkv, d, nk, dtype, S, variant), 8)
    for seed in (0, 3):
        counts, _ = check(inp, nsamp, stratified, variant, seed, step=seed)
        assert 0 < (counts > 0).mean() <= 1


def test_llama_32k_feature_access():
    """Llama-3.1-8B layer at 32K, B = 8 stratified samples (the pages'
    long-context setting, Sec. 5.2): parity, and the share of key features the
    groups need."""
    inp = synth.generate(synth.llama32k(32768, 256, "systematic"), 0)
    counts, _ = check(inp, 8, True, "systematic", seed=0)
    share = float((counts > 0).mean())
    assert 0.3 < share < 1.0
    print(f"\nkey features needed per KV-head group (B = 8, stratified): {100 * share:.1f}%")


def test_device_flags_bad_ragged_metadata():
    """Bad ragged metadata is flagged as in santa_decode; the other sequences
    are unaffected."""
    wl = synth.Workload("flags_b", 3, 4, 2, 128, 600, "bf16", 32, "systematic", ragged=(600, 600))
    inp = synth.generate(wl, 1)
    t = synth.to_torch(inp)
    S_per = torch.tensor([32, 0, 16], dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, 600, 1200, 1800], dtype=torch.int64, device="cuda")
    p = santa.make_params(t["q"], t["K"], 32, nk=500, kv_offsets=offs, S_per_seq=S_per)
    ws = santa.alloc_workspace(santa.bernoulli_workspace_size(p), "cuda")
    out = santa.santa_decode_bernoulli(t["q"], t["K"], t["V"], S=32, n_samples=4, nk=500, kv_offsets=offs,
                                       S_per_seq=S_per, workspace=ws)
    code = santa.get_error(ws)
    assert code & 1 and code & 2
    assert torch.count_nonzero(out) == 0
    offs_ok = torch.tensor([0, 600, 1000, 1800], dtype=torch.int64, device="cuda")
    out = santa.santa_decode_bernoulli(t["q"], t["K"], t["V"], S=32, n_samples=4, nk=800, kv_offsets=offs_ok,
                                       S_per_seq=S_per)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[0]) > 0


def test_invalid_sample_counts_are_rejected():
    inp = synth.generate(synth.Workload("bad_b", 1, 4, 1, 64, 300, "bf16", 16, "systematic"), 0)
    t = synth.to_torch(inp)
    for n in (0, 1025):
        with pytest.raises(santa.SantaError):
            santa.santa_decode_bernoulli(t["q"], t["K"], t["V"], S=16, n_samples=n)
