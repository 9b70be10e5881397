"""Synthetic measurement pins taken from the CUDA path's own draws.

"Stochastic Sparse Attention for Memory-Bound Inference" measures, on model
attention, how many distinct keys each sampler touches (App. L, Table 17) and
how the estimator variance falls with the budget S (App. D, Fig. 7; App. M).
Here the same statistics come from the GPU's sample indices and outputs over
many Philox seeds, on a synthetic Llama-shaped decode layer (32 query heads,
8 KV heads, d = 128, 8192 bf16 keys with planted high-score keys), and are
held to the closed forms of the oracle's analysis module:

* distinct keys per head: sum_n 1 - (1 - p_n)^S (i.i.d.),
  sum_n 1 - prod_m (1 - w[m, n]) (stratified), sum_n min(1, S p_n)
  (systematic);
* variance traces: tr(Sigma)/S (i.i.d.), the stratified closed form, and the
  exact integral over the systematic offset; and the log-log slope of each
  against S over S = 32 .. 256.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import stochastic_sparse_decode_split_gb300 as santa
from oracle import analysis

pytestmark = pytest.mark.gpu
SS = (32, 64, 128, 256)
VARIANTS = ("iid", "stratified", "systematic")


@pytest.fixture(scope="module")
def layer():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    santa.library()
    inp = synth.generate(synth.llama32k(8192, 256, "systematic"), 0)
    P = oracle.Problem.from_inputs(inp)
    H = inp.q.shape[1]
    heads = []
    for h in range(H):
        _, p = oracle.scores(P, 0, h)
        V = synth.storage_to_f64(inp.V[:, h // inp.wl.group], inp.wl.dtype)
        heads.append((p, V))
    return inp, heads


def _runs(inp, variant, S, R, want_idx):
    """R seeds of one decode: per-seed sample indices (or None) and the
    per-coordinate sum and sum of squares of the outputs (float64)."""
    t = synth.to_torch(inp)
    idx = torch.full((1, inp.q.shape[1], S), -7, dtype=torch.int32, device="cuda") if want_idx else None
    dec = santa.Decoder(t["q"], t["K"], t["V"], S=S, variant=variant, sample_idx=idx)
    s1 = torch.zeros(inp.q.shape, dtype=torch.float64, device="cuda")
    s2 = torch.zeros_like(s1)
    keys = []
    for seed in range(R):
        dec.p.seed = seed
        o = dec(step=0).double()
        s1 += o
        s2 += o * o
        if want_idx:
            keys.append(idx.clone())
    assert santa.get_error(dec.workspace) == 0
    return keys, s1.cpu().numpy()[0], s2.cpu().numpy()[0]


@pytest.mark.parametrize("variant", VARIANTS)
def test_distinct_keys_per_head_match_closed_form(layer, variant):
    """App. L, Table 17 analogue: mean distinct keys per head over 64 seeds,
    against the sampler's closed form averaged over the 32 heads."""
    inp, heads = layer
    f = {"iid": analysis.expected_unique_keys_iid, "stratified": analysis.expected_unique_keys_stratified,
         "systematic": analysis.expected_unique_keys_systematic}[variant]
    R = 64
    for S in SS:
        keys, _, _ = _runs(inp, variant, S, R, True)
        J = torch.stack(keys)[:, 0].cpu().numpy()            # [R, H, S]
        assert J.min() >= 0 and J.max() < 8192
        per_seed = np.array([[np.unique(J[r, h]).size for h in range(J.shape[1])] for r in range(R)]).mean(axis=1)
        want = np.mean([f(p, S) for p, _ in heads])
        se = per_seed.std(ddof=1) / np.sqrt(R)
        assert abs(per_seed.mean() - want) <= 4.0 * se + 0.05, (S, per_seed.mean(), want, se)
        print(f"\n{variant} S={S}: distinct keys per head {per_seed.mean():.2f} (closed form {want:.2f})")


def test_stratified_samplers_touch_more_keys_than_iid(layer):
    """Table 17's ordering on the GPU's draws: at every S the stratified and
    systematic samplers touch more distinct keys than i.i.d. SANTA, and at
    most S."""
    inp, _ = layer
    for S in SS:
        U = {}
        for variant in VARIANTS:
            keys, _, _ = _runs(inp, variant, S, 8, True)
            J = torch.stack(keys)[:, 0].cpu().numpy()
            U[variant] = np.mean([[np.unique(J[r, h]).size for h in range(J.shape[1])] for r in range(len(keys))])
        assert U["iid"] < U["stratified"] <= S and U["iid"] < U["systematic"] <= S, (S, U)


def test_variance_traces_and_slopes_match_closed_forms(layer):
    """App. D, Fig. 7 and App. M analogue: the replicate variance trace of the
    GPU's outputs over 1024 seeds, summed over the 32 heads, within 6 % of
    the closed form at each S, for each sampler; its log-log slope against
    S within 0.05 of the closed form's; stratified and systematic below
    i.i.d. at every S."""
    inp, heads = layer
    R = 1024
    exact = {v: [] for v in VARIANTS}
    gpu = {v: [] for v in VARIANTS}
    for S in SS:
        for variant in VARIANTS:
            _, s1, s2 = _runs(inp, variant, S, R, False)
            var = np.clip((s2 - s1 * s1 / R) / (R - 1), 0.0, None)     # [H, d]
            gpu[variant].append(var.sum())
            if variant == "iid":
                tr = sum(analysis.iid_variance_trace(p, V, S) for p, V in heads)
            elif variant == "stratified":
                tr = sum(analysis.stratified_variance_trace(p, V, S) for p, V in heads)
            else:
                tr = sum(analysis.systematic_coordinate_variance(p, V, S).sum() for p, V in heads)
            exact[variant].append(tr)
            rel = abs(gpu[variant][-1] - tr) / tr
            assert rel < 0.06, (variant, S, gpu[variant][-1], tr)
    slope = lambda v: float(np.polyfit(np.log(SS), np.log(v), 1)[0])
    for variant in VARIANTS:
        sg, se = slope(gpu[variant]), slope(exact[variant])
        print(f"\n{variant}: log-log slope of the variance trace against S: GPU {sg:.3f}, closed form {se:.3f}")
        assert abs(sg - se) < 0.05, (variant, sg, se)
    assert abs(slope(exact["iid"]) + 1.0) < 1e-9
    for i in range(len(SS)):
        assert gpu["stratified"][i] < gpu["iid"][i] and gpu["systematic"][i] < gpu["iid"][i]
