"""Pins for the oracle's distillation losses (forward / reverse KL, cakld, mse,
top-K support, temperature) and their gradient with respect to the student
logits.  Each test checks the oracle against something other than itself:
torch's kl_div / log_softmax with autograd in double (library), the closed
form of the KL between two Bernoulli distributions, brute-force selection of
the top-K support, and identities of the definitions (zero divergence of equal
distributions, K = V equals the whole vocabulary, K = 1 gives zero, the
temperature chain rule, the cakld limits, softmax gradients summing to zero).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from learnable_scale_fake_gb300 import synth

O = oracle
bits = synth.bf16_bits


def _case(T=6, V=300, seed=0, **kw):
    s, t, lab = synth.kd_logits(T, V, seed, **kw)
    return s, t, lab.numpy()


def _torch_losses(kd_type, s, t, lab, topk=0, tau=1.0, grad_scale=1.0):
    """The pages' formulas written with torch ops in double, autograd for the
    gradient; the top-K support is chosen here by a stable sort."""
    s64 = s.double().clone().requires_grad_(True)
    t64 = t.double()
    T, V = s64.shape
    valid = [(0 <= int(l) < V) for l in lab]
    n = sum(valid)
    per, fk, rk = [], [], []
    for i in range(T):
        if not valid[i]:
            continue
        a, b = t64[i] / tau, s64[i] / tau
        if topk:
            order = np.lexsort((np.arange(V), -t[i].double().numpy()))  # value desc, index asc
            idx = torch.from_numpy(np.sort(order[:topk]))
            a_k, b_k = a[idx], b[idx]
        else:
            a_k, b_k = a, b
        lpt, lps = F.log_softmax(a_k, -1), F.log_softmax(b_k, -1)
        fkl = F.kl_div(lps, lpt, reduction="sum", log_target=True)   # KL(teacher || student)
        rkl = F.kl_div(lpt, lps, reduction="sum", log_target=True)   # KL(student || teacher)
        conf = torch.softmax(a, -1)[int(lab[i])].detach()
        if kd_type == O.KD_KL:
            loss = tau ** 2 * fkl
        elif kd_type == O.KD_RKL:
            loss = tau ** 2 * rkl
        elif kd_type == O.KD_CAKLD:
            loss = tau ** 2 * (conf * rkl + (1 - conf) * fkl)
        else:
            loss = F.mse_loss(s64[i], t64[i])
        per.append(loss)
        fk.append(tau ** 2 * fkl)
        rk.append(tau ** 2 * rkl)
    total = torch.stack(per).sum() / n
    total.backward()
    return (total.item(), (torch.stack(fk).sum() / n).item(), (torch.stack(rk).sum() / n).item(),
            (s64.grad * grad_scale).numpy())


@pytest.mark.parametrize("kd_type", [O.KD_KL, O.KD_RKL, O.KD_CAKLD, O.KD_MSE])
@pytest.mark.parametrize("topk,tau", [(0, 1.0), (17, 1.0), (0, 2.0), (40, 0.5)])
def test_matches_torch_autograd(kd_type, topk, tau):
    if kd_type == O.KD_MSE and (topk or tau != 1.0):
        pytest.skip("mse has no top-K and no temperature")
    s, t, lab = _case(T=7, V=257, seed=3)
    r = O.kd_loss(kd_type, bits(s), bits(t), lab, topk=topk, temperature=tau, grad_scale=0.75)
    ref_loss, ref_f, ref_r, ref_g = _torch_losses(kd_type, s, t, lab, topk, tau, 0.75)
    assert r["losses"][0] == pytest.approx(ref_loss, rel=1e-12, abs=1e-15)
    assert r["losses"][1] == pytest.approx(ref_f, rel=1e-12, abs=1e-15)
    assert r["losses"][2] == pytest.approx(ref_r, rel=1e-12, abs=1e-15)
    np.testing.assert_allclose(r["dstudent"], ref_g, rtol=1e-10, atol=1e-16)


def test_bernoulli_closed_form():
    """V = 2: softmax of (0, x) is Bernoulli(sigmoid(x)); the KL has the
    textbook closed form p log(p/q) + (1-p) log((1-p)/(1-q)) and its
    derivative with respect to the student logit y is q - p."""
    xs = [0.5, -1.25, 3.0, 0.0]
    ys = [1.0, 2.5, -0.75, 0.0]
    for x, y in zip(xs, ys):
        t = torch.tensor([[0.0, x]]).bfloat16()
        s = torch.tensor([[0.0, y]]).bfloat16()
        p, q = 1 / (1 + math.exp(-x)), 1 / (1 + math.exp(-y))
        kl_pq = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        kl_qp = q * math.log(q / p) + (1 - q) * math.log((1 - q) / (1 - p))
        r = O.kd_loss(O.KD_KL, bits(s), bits(t), np.array([1]))
        assert r["losses"][1] == pytest.approx(kl_pq, rel=1e-12, abs=1e-15)
        assert r["losses"][2] == pytest.approx(kl_qp, rel=1e-12, abs=1e-15)
        assert r["dstudent"][0, 1] == pytest.approx(q - p, rel=1e-12, abs=1e-15)
        assert r["dstudent"][0, 0] == pytest.approx(p - q, rel=1e-12, abs=1e-15)


def test_topk_support_brute_force_with_ties():
    """Teacher logits drawn from a few levels, so the K-th value is tied: the
    support is the K largest values, equal values lower index first, listed
    in ascending index; -0 and +0 count as the same value."""
    rng = np.random.default_rng(4)
    T, V = 9, 64
    levels = np.array([-0.0, 0.0, 1.0, 1.5, 2.0, -3.0], np.float32)
    t = torch.from_numpy(levels[rng.integers(0, len(levels), (T, V))]).bfloat16()
    s = torch.from_numpy(rng.normal(size=(T, V)).astype(np.float32)).bfloat16()
    lab = np.arange(T)
    for K in (1, 5, 13, 31, 63, 64):
        r = O.kd_loss(O.KD_KL, bits(s), bits(t), lab, topk=K)
        for i in range(T):
            vals = t[i].float().numpy()
            order = sorted(range(V), key=lambda j: (-float(vals[j]), j))
            assert list(r["topk_idx"][i]) == sorted(order[:K])


def test_equal_distributions_give_zero():
    s, t, lab = _case(T=5, V=200, seed=8)
    for kd in (O.KD_KL, O.KD_RKL, O.KD_CAKLD, O.KD_MSE):
        r = O.kd_loss(kd, bits(t), bits(t), lab)
        assert np.all(r["tok"] == 0.0) or np.allclose(r["tok"], 0.0, atol=1e-15)
        assert np.allclose(r["dstudent"], 0.0, atol=1e-16)


def test_topk_k_equals_v_is_whole_vocabulary_and_k1_is_zero():
    s, t, lab = _case(T=5, V=128, seed=9)
    full = O.kd_loss(O.KD_CAKLD, bits(s), bits(t), lab)
    allk = O.kd_loss(O.KD_CAKLD, bits(s), bits(t), lab, topk=128)
    np.testing.assert_array_equal(full["tok"], allk["tok"])
    np.testing.assert_array_equal(full["dstudent"], allk["dstudent"])
    one = O.kd_loss(O.KD_CAKLD, bits(s), bits(t), lab, topk=1)
    assert np.all(one["tok"] == 0.0)
    assert np.all(one["dstudent"] == 0.0)


def test_temperature_chain_rule():
    """With logits that halve exactly in BF16: loss at tau = 2 on (s, t) equals
    4 x the loss at tau = 1 on (s/2, t/2), and the gradient is 2 x the tau = 1
    gradient taken at s/2."""
    s, t, lab = _case(T=6, V=160, seed=10)
    s2, t2 = (s.float() / 2).bfloat16(), (t.float() / 2).bfloat16()
    assert torch.equal(s2.float() * 2, s.float()) and torch.equal(t2.float() * 2, t.float())
    for kd in (O.KD_KL, O.KD_RKL, O.KD_CAKLD):
        a = O.kd_loss(kd, bits(s), bits(t), lab, temperature=2.0)
        b = O.kd_loss(kd, bits(s2), bits(t2), lab, temperature=1.0)
        np.testing.assert_allclose(a["tok"], 4 * b["tok"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(a["dstudent"], 2 * b["dstudent"], rtol=1e-10, atol=1e-18)


def test_cakld_limits():
    """conf -> 1 (the label dominates the teacher) gives the reverse KL; a
    label the teacher gives ~0 probability gives the forward KL."""
    s, t, lab = _case(T=4, V=100, seed=11)
    tt = t.float().clone()
    lab = np.array([5, 6, 7, 8])
    for i, l in enumerate(lab):
        tt[i, l] = 80.0       # conf = 1 - O(e^-60)
    t_hi = tt.bfloat16()
    r = O.kd_loss(O.KD_CAKLD, bits(s), bits(t_hi), lab)
    np.testing.assert_allclose(r["tok"][:, 0], r["tok"][:, 2], rtol=1e-12)
    tt = t.float().clone()
    for i, l in enumerate(lab):
        tt[i, l] = -80.0      # conf = O(e^-80)
    r = O.kd_loss(O.KD_CAKLD, bits(s), bits(tt.bfloat16()), lab)
    np.testing.assert_allclose(r["tok"][:, 0], r["tok"][:, 1], rtol=1e-12)


def test_invariants():
    """KL >= 0; the gradient of every KL row sums to zero (softmax); shifting
    a student row by an integer (exact in BF16 for these integer logits)
    changes nothing; ignored positions carry no loss and no gradient."""
    rng = np.random.default_rng(12)
    T, V = 6, 96
    t = torch.from_numpy(rng.integers(-8, 9, (T, V)).astype(np.float32)).bfloat16()
    s = torch.from_numpy(rng.integers(-8, 9, (T, V)).astype(np.float32)).bfloat16()
    lab = np.array([0, -100, 5, 95, 96, 3])  # 96 is outside the vocabulary: ignored
    for kd in (O.KD_KL, O.KD_RKL, O.KD_CAKLD):
        r = O.kd_loss(kd, bits(s), bits(t), lab)
        assert np.all(r["tok"][:, 1:] >= 0)
        gsum = np.abs(r["dstudent"]).sum(axis=1)
        assert np.all(np.abs(r["dstudent"].sum(axis=1)) <= 1e-14 * gsum)
        assert np.all(r["tok"][[1, 4]] == 0) and np.all(r["dstudent"][[1, 4]] == 0)
        sh = O.kd_loss(kd, bits((s.float() + 3).bfloat16()), bits(t), lab)
        np.testing.assert_allclose(sh["tok"], r["tok"], rtol=1e-12, atol=1e-15)
        # the mean is over the 4 valid positions
        assert r["losses"][0] == pytest.approx(r["tok"][:, 0].sum() / 4, rel=1e-14)


def test_mse_matches_numpy():
    s, t, lab = _case(T=5, V=211, seed=13)
    r = O.kd_loss(O.KD_MSE, bits(s), bits(t), lab, grad_scale=2.0)
    d = s.double().numpy() - t.double().numpy()
    valid = (lab >= 0) & (lab < 211)
    np.testing.assert_allclose(r["tok"][valid, 0], (d[valid] ** 2).mean(axis=1), rtol=1e-13)
    np.testing.assert_allclose(r["dstudent"][valid], 2.0 * 2 * d[valid] / 211 / valid.sum(), rtol=1e-13)


def test_rejects_bad_arguments():
    s, t, lab = _case(T=2, V=50, seed=1)
    for kw in ({"topk": 51}, {"temperature": 0.0}, {"temperature": -1.0}):
        with pytest.raises(ValueError):
            O.kd_loss(O.KD_KL, bits(s), bits(t), lab, **kw)
    with pytest.raises(ValueError):
        O.kd_loss(O.KD_MSE, bits(s), bits(t), lab, topk=5)
