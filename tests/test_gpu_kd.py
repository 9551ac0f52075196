"""GPU parity of the distillation losses (aqfq_kd_loss) against the oracle.

Tolerances, from the arithmetic of the kernel (binary32, hardware base-2
exponentials with relative error about 2^-22, arguments rounded once):
  * per-position KL losses: |d| <= 2^-20 * cond, cond = tau^2 sum_U (p_t + p_s)
    (1 + |log p_t| + |log p_s|) (the oracle's first-order error scale of the
    per-element terms, 4x above the exponential error);
  * mse per position: relative 2^-18 (a sum of exactly formed squares);
  * the means: the sum of the per-position bounds over the valid positions;
  * gradient elements (BF16): |d| <= 2^-8 |ref| (rounding to BF16) + 2^-18 * gmag
    (the oracle's per-element error scale of the binary32 value);
  * the top-K support (integer work): bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from learnable_scale_fake_gb300 import aqfq, synth

pytestmark = pytest.mark.gpu
O = oracle
bits = synth.bf16_bits
DEV = "cuda:0"


def run_gpu(kd_type, s, t, lab, topk=0, tau=1.0, gs=1.0, want_idx=False, want_grad=True):
    T, V = s.shape
    sd, td = s.to(DEV), t.to(DEV)
    labd = torch.as_tensor(lab, dtype=torch.int32).to(DEV)
    losses = torch.full((3,), float("nan"), device=DEV)
    tl = torch.full((T,), float("nan"), device=DEV)
    ds = torch.full((T, V), float("nan"), dtype=torch.bfloat16, device=DEV) if want_grad else None
    idx = torch.full((T, topk), -7, dtype=torch.int32, device=DEV) if want_idx else None
    ws = torch.empty(aqfq.aqfq_kd_workspace_bytes(T), dtype=torch.uint8, device=DEV)
    aqfq.aqfq_kd_loss(kd_type, sd, td, labd, losses, ws, topk=topk, temperature=tau, grad_scale=gs,
                      token_loss=tl, dstudent=ds, topk_idx=idx)
    torch.cuda.synchronize()
    return {"losses": losses.cpu().double().numpy(), "tok": tl.cpu().double().numpy(),
            "ds": None if ds is None else ds.cpu().float().double().numpy(),
            "ds_bits": None if ds is None else bits(ds),
            "idx": None if idx is None else idx.cpu().numpy()}


def check(kd_type, s, t, lab, topk=0, tau=1.0, gs=1.0, want_idx=False, rows=None):
    g = run_gpu(kd_type, s, t, lab, topk, tau, gs, want_idx)
    r = O.kd_loss(kd_type, bits(s), bits(t), lab, topk=topk, temperature=tau, grad_scale=gs)
    valid = (lab >= 0) & (lab < s.shape[1])
    mse = kd_type == O.KD_MSE
    tol_tok = np.where(valid, (2.0 ** -18 * r["cond"][:, 1]) if mse else 2.0 ** -20 * r["cond"][:, 0], 0)
    err = np.abs(g["tok"] - r["tok"][:, 0])
    assert np.all(err <= tol_tok), f"per-position loss: worst {np.max(err - tol_tok)}"
    assert np.all(g["tok"][~valid] == 0)
    n = max(1, valid.sum())
    for k in range(3):
        tk = tol_tok.sum() / n if k == 0 else 2.0 ** -20 * r["cond"][valid, 0].sum() / n
        assert abs(g["losses"][k] - r["losses"][k]) <= tk + 2.0 ** -22 * abs(r["losses"][k]), k
    ds_tol = 2.0 ** -8 * np.abs(r["dstudent"]) + 2.0 ** -18 * r["gmag"]
    derr = np.abs(g["ds"] - r["dstudent"])
    bad = derr > ds_tol
    assert not bad.any(), (f"{bad.sum()} gradient elements off; worst at "
                           f"{np.unravel_index(np.argmax(derr - ds_tol), derr.shape)}")
    assert np.all(g["ds"][~valid] == 0)
    if topk:  # nothing outside the oracle's support
        inside = np.zeros(g["ds"].shape, bool)
        for i in np.nonzero(valid)[0]:
            inside[i, r["topk_idx"][i]] = True
        assert np.all(g["ds"][~inside] == 0)
    if want_idx:
        np.testing.assert_array_equal(g["idx"], r["topk_idx"])
    return g, r


@pytest.mark.parametrize("kd_type", [O.KD_KL, O.KD_RKL, O.KD_CAKLD, O.KD_MSE])
def test_whole_vocabulary_qwen_vocab(kd_type):
    s, t, lab = synth.kd_logits(10, synth.KD_VOCAB, 21)
    check(kd_type, s, t, lab.numpy(), gs=0.5)


@pytest.mark.parametrize("kd_type", [O.KD_KL, O.KD_RKL, O.KD_CAKLD])
@pytest.mark.parametrize("topk", [1, 50, 1000, 4096])
def test_topk_support(kd_type, topk):
    s, t, lab = synth.kd_logits(8, synth.KD_VOCAB, 22)
    check(kd_type, s, t, lab.numpy(), topk=topk, want_idx=True)


@pytest.mark.parametrize("kd_type,topk,tau", [(O.KD_KL, 0, 2.0), (O.KD_CAKLD, 0, 0.7),
                                              (O.KD_RKL, 100, 2.0), (O.KD_CAKLD, 300, 1.5)])
def test_temperature(kd_type, topk, tau):
    s, t, lab = synth.kd_logits(6, 32768, 23)
    check(kd_type, s, t, lab.numpy(), topk=topk, tau=tau, want_idx=topk > 0)


@pytest.mark.parametrize("V", [8, 24, 1000, 4104])
def test_ragged_slices(V):
    """V / 8 not a multiple of 8: the last slices are short or empty."""
    s, t, lab = synth.kd_logits(5, V, 24)
    lab = lab.numpy() % V
    for kd in (O.KD_KL, O.KD_CAKLD, O.KD_MSE):
        check(kd, s, t, lab)
    check(O.KD_RKL, s, t, lab, topk=min(V, 7), want_idx=True)
    check(O.KD_KL, s, t, lab, topk=V, want_idx=True)  # K = V: the whole vocabulary


def test_ties_at_the_threshold_across_slices():
    """Teacher logits from a few levels, so thousands of equal values straddle
    the K-th place and span every slice: the support takes the lower indices."""
    rng = np.random.default_rng(25)
    T, V = 6, 20000
    levels = np.array([-1.0, 0.0, -0.0, 0.5, 1.0, 2.0], np.float32)
    t = torch.from_numpy(levels[rng.integers(0, len(levels), (T, V))]).bfloat16()
    s = torch.from_numpy(rng.normal(size=(T, V)).astype(np.float32)).bfloat16()
    lab = rng.integers(0, V, T)
    for K in (1, 3000, 3333, 9999, 19999):
        check(O.KD_CAKLD, s, t, lab, topk=K, want_idx=True)


def test_many_positions_and_ignored_rows():
    """More positions than resident clusters (the persistent loop), a third
    of them ignored, labels -100 and >= V."""
    s, t, lab = synth.kd_logits(300, 2048, 26, ignore=0.33)
    lab = lab.numpy()
    lab[::17] = 2048
    for kd in (O.KD_KL, O.KD_CAKLD, O.KD_MSE):
        check(kd, s, t, lab, gs=3.0)
    check(O.KD_RKL, s, t, lab, topk=64, want_idx=True)


def test_position_list_over_several_chunks():
    """T = 9001 positions (the count kernel lists them in chunks of 4096, the
    last one ragged), 30 % ignored, handed out by ticket to the clusters: every
    position's loss and gradient row, and zero rows for the ignored ones."""
    s, t, lab = synth.kd_logits(9001, 64, 31, ignore=0.3)
    lab = lab.numpy()
    check(O.KD_CAKLD, s, t, lab)
    check(O.KD_KL, s, t, lab, topk=5, want_idx=True)


def test_largest_vocabulary():
    """V = 262144 with the top-K histogram: the largest shared-memory layout."""
    s, t, lab = synth.kd_logits(3, 262144, 27)
    check(O.KD_CAKLD, s, t, lab.numpy(), topk=2000, want_idx=True)
    check(O.KD_KL, s, t, lab.numpy())


def test_topk_beyond_the_row_kernel():
    """V = 600000 (more than 2^16 vectors of 8): top-K takes the cluster kernel
    (slices of the teacher row over 8 CTAs) instead of one CTA per position."""
    s, t, lab = synth.kd_logits(3, 600000, 32)
    check(O.KD_CAKLD, s, t, lab.numpy(), topk=1000, want_idx=True)
    check(O.KD_KL, s, t, lab.numpy(), topk=7, want_idx=True)


def test_no_valid_position_and_empty():
    s, t, lab = synth.kd_logits(4, 512, 28)
    lab = np.full(4, -100)
    g = run_gpu(O.KD_CAKLD, s, t, lab, topk=10, want_idx=True)
    assert np.all(g["losses"] == 0) and np.all(g["tok"] == 0) and np.all(g["ds"] == 0)
    assert np.all(g["idx"] == -1)
    losses = torch.full((3,), float("nan"), device=DEV)
    ws = torch.empty(aqfq.aqfq_kd_workspace_bytes(0), dtype=torch.uint8, device=DEV)
    e = torch.empty((0, 512), dtype=torch.bfloat16, device=DEV)
    aqfq.aqfq_kd_loss(O.KD_KL, e, e, torch.empty(0, dtype=torch.int32, device=DEV), losses, ws)
    torch.cuda.synchronize()
    assert torch.all(losses == 0)


def test_reproducible_bits():
    s, t, lab = synth.kd_logits(40, 65536, 29)
    a = run_gpu(O.KD_CAKLD, s, t, lab.numpy(), topk=500, want_idx=True)
    b = run_gpu(O.KD_CAKLD, s, t, lab.numpy(), topk=500, want_idx=True)
    np.testing.assert_array_equal(a["ds_bits"], b["ds_bits"])
    np.testing.assert_array_equal(a["tok"], b["tok"])
    np.testing.assert_array_equal(a["losses"], b["losses"])


@pytest.mark.parametrize("name", ["kd_cakld", "kd_topk"])
def test_full_size_bench_workload(name):
    """The bench workloads (4096 positions x 151936 vocabulary, the same call
    and launch configuration): every position's loss and the means against
    the oracle on all rows; the gradient and the top-K support on sampled rows."""
    from learnable_scale_fake_gb300 import workloads

    wl = workloads.BUILDERS[name](torch.device(DEV))
    s, t, lab = wl.inputs["student"], wl.inputs["teacher"], wl.inputs["labels"]
    T, V = s.shape
    kt, topk = (O.KD_CAKLD, 0) if name == "kd_cakld" else (O.KD_KL, 1000)
    tl = torch.empty(T, device=DEV)
    idx = torch.empty((T, topk), dtype=torch.int32, device=DEV) if topk else None
    wl.ops[0].run(torch.cuda.current_stream())  # the bench's call
    ws = torch.empty(aqfq.aqfq_kd_workspace_bytes(T), dtype=torch.uint8, device=DEV)
    losses = torch.empty(3, device=DEV)
    aqfq.aqfq_kd_loss(kt, s, t, lab, losses, ws, topk=topk, token_loss=tl, topk_idx=idx)
    torch.cuda.synchronize()
    labn = lab.cpu().numpy()
    valid = (labn >= 0) & (labn < V)
    r = O.kd_loss(kt, bits(s), bits(t), labn, topk=topk, want_grad=False)
    g_tok = tl.cpu().double().numpy()
    tol = np.where(valid, 2.0 ** -20 * r["cond"][:, 0], 0)
    assert np.all(np.abs(g_tok - r["tok"][:, 0]) <= tol)
    n = valid.sum()
    g_loss = losses.cpu().double().numpy()
    for k in range(3):
        assert abs(g_loss[k] - r["losses"][k]) <= 2.0 ** -20 * r["cond"][valid, 0].sum() / n
    # the bench call's gradient on sampled rows (the oracle on those rows alone,
    # its gradient scale set to the full problem's 1 / n_valid)
    rows = np.array([0, 1, 2, 777, 2048, 3001, T - 2, T - 1])
    sub = O.kd_loss(kt, bits(s[rows]), bits(t[rows]), labn[rows], topk=topk,
                    grad_scale=float(((labn[rows] >= 0) & (labn[rows] < V)).sum()) / n)
    gds = wl.outputs["dstudent"][rows].cpu().float().double().numpy()
    ds_tol = 2.0 ** -8 * np.abs(sub["dstudent"]) + 2.0 ** -18 * sub["gmag"]
    assert np.all(np.abs(gds - sub["dstudent"]) <= ds_tol)
    if topk:
        np.testing.assert_array_equal(idx[rows].cpu().numpy(), sub["topk_idx"])


def test_topk_wide_key_range_two_level_path():
    """Teacher logits spread over 120 octaves (both signs): the keys above the
    vector-max bound span more bins than the exact-key histogram holds, so the
    12-bit + 4-bit path decides the threshold; small and large K."""
    rng = np.random.default_rng(31)
    T, V = 5, 16384
    mag = np.exp2(rng.uniform(-60, 60, (T, V))).astype(np.float32)
    t = torch.from_numpy(mag * rng.choice([-1.0, 1.0], (T, V)).astype(np.float32)).bfloat16()
    s = (t.float() * 0.5 + torch.from_numpy(rng.normal(size=(T, V)).astype(np.float32))).bfloat16()
    lab = rng.integers(0, V, T)
    for K in (5, 50, 700):
        check(O.KD_RKL, s, t, lab, topk=K, want_idx=True)
