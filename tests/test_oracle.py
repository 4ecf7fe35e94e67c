"""Pins for the fp64 oracle: closed forms, invariants, finite differences and an
independent library routine. None of these calls the CUDA library.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import grpo_oracle as orc
import synth


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ----------------------------------------------------------------- logp ----

@pytest.mark.parametrize("V", [4096, 128256, 151936, 201088])
def test_zero_weight_gives_uniform_logp(V):
    # W = 0: every logit is 0, so logp = -log V exactly.
    h = _rand((3, 8), 0)
    W = np.zeros((V, 8))
    ids = np.array([0, V // 2, V - 1])
    logp, lse = oracle.selective_logp(h, W, ids)
    assert np.allclose(logp, -math.log(V), rtol=0, atol=1e-12)
    assert np.allclose(lse, math.log(V), rtol=0, atol=1e-12)


def test_known_uniform_values():
    # -log V for the workloads' vocabularies, to four decimals.
    for V, want in ((4096, 8.3178), (128256, 11.7618), (151936, 11.9312), (201088, 12.2115)):
        lp, _ = oracle.selective_logp(np.ones((1, 4)), np.zeros((V, 4)), [7])
        assert abs(-lp[0] - want) < 5e-5


def test_probabilities_sum_to_one():
    h = _rand((4, 16), 1)
    W = _rand((50, 16), 2, 0.7)
    for t in range(4):
        lp, _ = oracle.selective_logp(np.repeat(h[t:t + 1], 50, 0), W, np.arange(50))
        assert abs(math.fsum(np.exp(lp)) - 1.0) < 1e-13


def test_two_entry_vocab_is_log_sigmoid():
    # V = 2: logp(y=0) = log sigmoid(z0 - z1) = -log1p(exp(z1 - z0)).
    h = _rand((5, 6), 3)
    W = _rand((2, 6), 4)
    lp0, _ = oracle.selective_logp(h, W, np.zeros(5, dtype=int))
    lp1, _ = oracle.selective_logp(h, W, np.ones(5, dtype=int))
    for t in range(5):
        z0 = math.fsum(h[t, d] * W[0, d] for d in range(6))
        z1 = math.fsum(h[t, d] * W[1, d] for d in range(6))
        assert abs(lp0[t] - (-math.log1p(math.exp(z1 - z0)))) < 1e-13
        assert abs(lp1[t] - (-math.log1p(math.exp(z0 - z1)))) < 1e-13


def test_single_entry_vocab_gives_zero():
    lp, _ = oracle.selective_logp(_rand((3, 5), 5), _rand((1, 5), 6), [0, 0, 0])
    assert np.all(np.abs(lp) < 1e-15)


def test_brute_force_tiny():
    # Pure-Python loops with exactly rounded sums.
    N, D, V = 3, 4, 5
    h = _rand((N, D), 7)
    W = _rand((V, D), 8)
    y = [4, 0, 2]
    lp, _ = oracle.selective_logp(h, W, y)
    for t in range(N):
        z = [math.fsum(h[t, d] * W[v, d] for d in range(D)) for v in range(V)]
        lse = math.log(math.fsum(math.exp(x) for x in z))
        assert abs(lp[t] - (z[y[t]] - lse)) < 1e-13


def test_vocab_permutation_invariance():
    h = _rand((6, 12), 9)
    W = _rand((40, 12), 10)
    y = np.random.default_rng(11).integers(0, 40, 6)
    perm = np.random.default_rng(12).permutation(40)
    inv = np.argsort(perm)
    lp, _ = oracle.selective_logp(h, W, y)
    lp2, _ = oracle.selective_logp(h, W[perm], inv[y])
    assert np.allclose(lp, lp2, rtol=0, atol=1e-13)


def test_common_row_shift_invariance():
    # Adding c to every W row shifts every logit of row t by h_t . c.
    h = _rand((6, 12), 13)
    W = _rand((40, 12), 14)
    c = _rand((12,), 15)
    y = np.arange(6) * 5
    lp, _ = oracle.selective_logp(h, W, y)
    lp2, _ = oracle.selective_logp(h, W + c[None, :], y)
    assert np.allclose(lp, lp2, rtol=0, atol=1e-12)


def test_matches_torch_log_softmax_fp64():
    # An independent library routine: torch's float64 log_softmax + gather.
    p = synth.make_problem("tiny", seed=3)
    lp, lse = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    z = p.hidden.double() @ p.weight.double().T
    ref = torch.log_softmax(z, dim=1).gather(1, p.ids.long()[:, None])[:, 0]
    assert np.allclose(lp, ref.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(lse, torch.logsumexp(z, 1).numpy(), rtol=0, atol=1e-12)


def test_row_block_does_not_change_values():
    h = _rand((37, 8), 16)
    W = _rand((33, 8), 17)
    y = np.arange(37) % 33
    a, _ = oracle.selective_logp(h, W, y, row_block=1)
    b, _ = oracle.selective_logp(h, W, y, row_block=64)
    assert np.allclose(a, b, rtol=0, atol=1e-13)  # BLAS kernels differ by row count


# ----------------------------------------------------------------- loss ----

def _loss_case(seed, N=12, T=4, eps=0.2):
    rng = np.random.default_rng(seed)
    logp = -rng.uniform(1, 8, N)
    adv = rng.standard_normal(N // T)
    mask = np.ones(N)
    return logp, adv, mask, T, eps


def test_on_policy_loss_is_minus_mean_advantage():
    # old = logp and beta = 0: ratio 1, L = -sum m A / M, g_t = -A m_t / M
    # (the exp(q - q.detach()) * A identity).
    logp, adv, mask, T, eps = _loss_case(20)
    mask[[2, 3, 9]] = 0
    A_tok = adv[np.arange(12) // T]
    L, g, _, M = oracle.grpo_loss(logp, logp, logp, adv, mask, T, eps, eps, 0.0)
    assert M == 9
    assert abs(L - (-(A_tok * mask).sum() / 9)) < 1e-14
    assert np.allclose(g, -A_tok * mask / 9, rtol=0, atol=1e-15)
    # With ref = logp the KL term vanishes too, for any beta.
    L2, g2, _, _ = oracle.grpo_loss(logp, logp, logp, adv, mask, T, eps, eps, 0.5)
    assert abs(L2 - L) < 1e-14 and np.allclose(g2, g, atol=1e-15)


def test_zero_mean_group_advantage_gives_zero_on_policy_loss():
    p = synth.make_problem("tiny", seed=5)
    lp = -np.ones(p.n_tokens) * 3
    L, _, _, _ = oracle.grpo_loss(lp, lp, lp, p.adv.double(), p.mask, p.seq_len, 0.2, 0.2, 0.0)
    assert abs(L) < 1e-7  # adv was cast to fp32: mean is 0 up to fp32 rounding


@pytest.mark.parametrize("ratio,A,clipped", [
    (2.0, 1.0, True), (0.5, -1.0, True), (2.0, -1.0, False), (0.5, 1.0, False),
    (1.1, 1.0, False), (0.9, -1.0, False)])
def test_clip_branches(ratio, A, clipped):
    eps = 0.2
    logp = np.array([-2.0])
    old = logp - math.log(ratio)
    L, g, lt, M = oracle.grpo_loss(logp, old, logp, np.array([A]), np.ones(1), 1, eps, eps, 0.0)
    c = min(max(ratio, 1 - eps), 1 + eps)
    assert abs(L - (-min(ratio * A, c * A))) < 1e-14
    want_g = 0.0 if clipped else -A * ratio
    assert abs(g[0] - want_g) < 1e-14


def test_asymmetric_clip_bounds():
    logp = np.array([-1.0, -1.0])
    old = logp - np.log([1.25, 0.75])
    L, g, lt, _ = oracle.grpo_loss(logp, old, logp, np.array([1.0, -1.0]), np.ones(2), 1,
                                   eps_low=0.3, eps_high=0.3, beta=0.0)
    assert np.allclose(g, [-1.25 / 2, 0.75 / 2], atol=1e-15)  # inside wider bounds
    L, g, lt, _ = oracle.grpo_loss(logp, old, logp, np.array([1.0, -1.0]), np.ones(2), 1,
                                   eps_low=0.2, eps_high=0.2, beta=0.0)
    assert np.allclose(g, [0.0, 0.0], atol=1e-15)


def test_kl_term_closed_form():
    # A = 0: l = beta * (e^d - d - 1) with d = ref - logp; >= 0, zero iff d = 0.
    logp = np.array([-3.0, -3.0, -3.0])
    ref = logp + np.array([1.0, 0.0, -0.5])
    beta = 0.25
    L, g, lt, _ = oracle.grpo_loss(logp, logp, ref, np.zeros(3), np.ones(3), 1, 0.2, 0.2, beta)
    kl = np.array([math.e - 2.0, 0.0, math.exp(-0.5) + 0.5 - 1.0])
    assert np.allclose(lt, beta * kl, rtol=0, atol=1e-15)
    assert np.all(lt >= 0) and lt[1] == 0
    assert np.allclose(g, beta * (1 - np.exp(ref - logp)) / 3, atol=1e-15)


def test_masked_tokens_are_ignored():
    logp, adv, mask, T, eps = _loss_case(21)
    mask[[0, 5, 11]] = 0
    rng = np.random.default_rng(4)
    old = logp + rng.normal(0, 0.1, 12)
    ref = logp + rng.normal(0, 0.1, 12)
    L, g, _, _ = oracle.grpo_loss(logp, old, ref, adv, mask, T, eps, eps, 0.01)
    old2, ref2, lp2 = old.copy(), ref.copy(), logp.copy()
    old2[[0, 5, 11]] = 1e9
    ref2[[0, 5, 11]] = -1e9
    lp2[[0, 5, 11]] = np.nan
    L2, g2, _, _ = oracle.grpo_loss(lp2, old2, ref2, adv, mask, T, eps, eps, 0.01)
    assert L == L2 and np.array_equal(g, g2)
    assert np.all(g[[0, 5, 11]] == 0)


def test_empty_mask_gives_zero():
    logp, adv, mask, T, eps = _loss_case(22)
    L, g, _, M = oracle.grpo_loss(logp, logp - 0.1, logp, adv, np.zeros(12), T, eps, eps, 0.01)
    assert L == 0.0 and M == 0.0 and np.all(g == 0)


def test_loss_denominator_override():
    logp, adv, mask, T, eps = _loss_case(23)
    L1, g1, _, _ = oracle.grpo_loss(logp, logp - 0.1, logp, adv, mask, T, eps, eps, 0.01)
    L2, g2, _, _ = oracle.grpo_loss(logp, logp - 0.1, logp, adv, mask, T, eps, eps, 0.01,
                                    loss_denominator=48.0)
    assert abs(L2 * 48 - L1 * 12) < 1e-13 and np.allclose(g2 * 48, g1 * 12, atol=1e-15)


def test_loss_gradient_matches_finite_differences():
    logp, adv, mask, T, eps = _loss_case(24)
    mask[3] = 0
    rng = np.random.default_rng(5)
    old = logp + rng.normal(0, 0.15, 12)
    ref = logp + rng.normal(0, 0.15, 12)
    r = np.exp(logp - old)
    assert np.all(np.abs(r - 0.8) > 1e-3) and np.all(np.abs(r - 1.2) > 1e-3)
    L, g, _, _ = oracle.grpo_loss(logp, old, ref, adv, mask, T, eps, eps, 0.05)
    step = 1e-6
    for t in range(12):
        lp_p, lp_m = logp.copy(), logp.copy()
        lp_p[t] += step
        lp_m[t] -= step
        Lp = oracle.grpo_loss(lp_p, old, ref, adv, mask, T, eps, eps, 0.05)[0]
        Lm = oracle.grpo_loss(lp_m, old, ref, adv, mask, T, eps, eps, 0.05)[0]
        assert abs((Lp - Lm) / (2 * step) - g[t]) < 1e-8


# ------------------------------------------------------------- backward ----

def _tiny_full(seed, N=8, D=16, V=64, T=4, eps=0.2, beta=0.05):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.3
    y = rng.integers(0, V, N)
    mask = np.ones(N)
    mask[N - 1] = 0
    lp, _ = oracle.selective_logp(h, W, y)
    old = lp + rng.normal(0, 0.12, N)
    ref = lp + rng.normal(0, 0.12, N)
    r = np.exp(lp - old)
    assert np.all(np.abs(r - (1 - eps)) > 1e-3) and np.all(np.abs(r - (1 + eps)) > 1e-3)
    adv = rng.standard_normal(N // T)
    return h, W, y, mask, old, ref, adv, T, eps, beta


def _L_of_h(h, W, y, mask, old, ref, adv, T, eps, beta):
    lp, _ = oracle.selective_logp(h, W, y)
    return oracle.grpo_loss(lp, old, ref, adv, mask, T, eps, eps, beta)[0]


def test_dH_matches_central_finite_differences():
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(30)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)
    dH = out["dH"]
    fd = np.zeros_like(h)
    step = 1e-6
    for t in range(h.shape[0]):
        for d in range(h.shape[1]):
            hp, hm = h.copy(), h.copy()
            hp[t, d] += step
            hm[t, d] -= step
            fd[t, d] = (_L_of_h(hp, W, y, mask, old, ref, adv, T, eps, beta)
                        - _L_of_h(hm, W, y, mask, old, ref, adv, T, eps, beta)) / (2 * step)
    rel = np.linalg.norm(fd - dH) / np.linalg.norm(dH)
    assert rel < 1e-6
    assert np.all(dH[-1] == 0)  # masked row


def test_grad_hidden_of_single_logp_matches_fd():
    # g = e_t pins d logp_t / d h_t = W[y_t] - E_softmax[W] on its own (sign included).
    rng = np.random.default_rng(31)
    h = rng.standard_normal((3, 5))
    W = rng.standard_normal((7, 5))
    y = np.array([6, 1, 3])
    g = np.array([0.0, 1.0, 0.0])
    dH = oracle.grad_hidden(h, W, y, g)
    step = 1e-6
    for d in range(5):
        hp, hm = h.copy(), h.copy()
        hp[1, d] += step
        hm[1, d] -= step
        fd = (oracle.selective_logp(hp, W, y)[0][1] - oracle.selective_logp(hm, W, y)[0][1]) / (2 * step)
        assert abs(fd - dH[1, d]) < 1e-8
    assert np.all(dH[0] == 0) and np.all(dH[2] == 0)


def test_dH_matches_torch_autograd_fp64():
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(32)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)
    ht = torch.tensor(h, requires_grad=True)
    z = ht @ torch.tensor(W).T
    lp = torch.log_softmax(z, 1).gather(1, torch.tensor(y)[:, None])[:, 0]
    A = torch.tensor(adv)[torch.arange(len(y)) // T]
    r = torch.exp(lp - torch.tensor(old))
    surr = torch.minimum(r * A, torch.clamp(r, 1 - eps, 1 + eps) * A)
    dl = torch.tensor(ref) - lp
    lt = -surr + beta * (torch.exp(dl) - dl - 1)
    m = torch.tensor(mask)
    L = (lt * m).sum() / m.sum()
    L.backward()
    assert abs(L.item() - out["L"]) < 1e-13
    assert np.allclose(ht.grad.numpy(), out["dH"], rtol=1e-10, atol=1e-14)


def test_zero_weight_gives_zero_dH():
    rng = np.random.default_rng(33)
    dH = oracle.grad_hidden(rng.standard_normal((4, 6)), np.zeros((9, 6)), [1, 2, 3, 4],
                            np.array([0.3, -1.0, 2.0, 0.5]))
    assert np.all(dH == 0)


def test_rows_fwd_bwd_matches_full_path():
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(34)
    full = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)
    rows = np.array([0, 3, 5])
    part = oracle.rows_fwd_bwd(h, W, y, rows, old, ref, adv, T, full["M"], eps, eps, beta)
    assert np.allclose(part["logp"], full["logp"][rows], atol=1e-14)
    assert np.allclose(part["g"], full["g"][rows], atol=1e-16)
    assert np.allclose(part["dH"], full["dH"][rows], atol=1e-14)


# ---------------------------------------------- planted mistakes are caught --

def test_planted_sign_error_in_backward_is_caught(monkeypatch):
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(35)
    good = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)["dH"]
    bad = -good  # a flipped sign, as the cross-entropy convention would give
    fd_row = np.zeros(h.shape[1])
    step = 1e-6
    for d in range(h.shape[1]):
        hp, hm = h.copy(), h.copy()
        hp[0, d] += step
        hm[0, d] -= step
        fd_row[d] = (_L_of_h(hp, W, y, mask, old, ref, adv, T, eps, beta)
                     - _L_of_h(hm, W, y, mask, old, ref, adv, T, eps, beta)) / (2 * step)
    assert np.linalg.norm(fd_row - good[0]) < 1e-6 * np.linalg.norm(good[0])
    assert np.linalg.norm(fd_row - bad[0]) > 0.5 * np.linalg.norm(good[0])


def test_planted_clip_mistake_is_caught(monkeypatch):
    # A surrogate that forgets the clip would pass gradient on clipped tokens.
    logp = np.array([-2.0])
    old = logp - math.log(2.0)
    real = orc.token_terms

    def no_clip(lp, od, rf, A, el, eh, b):
        lt, dl, r, kl = real(lp, od, rf, A, 10.0, 10.0, b)
        return lt, dl, r, kl

    monkeypatch.setattr(orc, "token_terms", no_clip)
    _, g_bad, _, _ = orc.grpo_loss(logp, old, logp, np.array([1.0]), np.ones(1), 1, 0.2, 0.2, 0.0)
    monkeypatch.setattr(orc, "token_terms", real)
    _, g_ok, _, _ = orc.grpo_loss(logp, old, logp, np.array([1.0]), np.ones(1), 1, 0.2, 0.2, 0.0)
    assert g_ok[0] == 0.0 and g_bad[0] != 0.0


# ------------------------------------------------------------- generator ---

@pytest.mark.parametrize("name", ["tiny", "qwen2.5-1.5b"])
def test_generator_group_advantages_have_zero_mean(name):
    p = synth.make_problem(name, seed=1, D=64, V=128)
    a64 = synth.group_advantages(p.rewards, p.group).reshape(-1, p.group)
    assert torch.all(a64.mean(1).abs() < 1e-12)


def test_generator_shapes_and_padding():
    p = synth.make_problem("qwen2.5-1.5b", seed=2, D=64, V=128)
    assert p.n_tokens == 8192 and p.seq_len == 1024 and p.n_seqs == 8
    assert p.hidden.dtype == torch.bfloat16 and p.hidden.shape == (8192, 64)
    assert p.ids.dtype == torch.int32 and int(p.ids.max()) < 128
    m = p.mask.reshape(8, 1024)
    for b in range(8):
        L = int(p.lengths[b])
        assert 256 <= L <= 1024
        assert m[b, :L].all() and not m[b, L:].any()
    assert p.n_valid == int(p.mask.sum())


def test_generator_is_deterministic():
    a = synth.make_problem("tiny", seed=9)
    b = synth.make_problem("tiny", seed=9)
    assert torch.equal(a.hidden, b.hidden) and torch.equal(a.weight, b.weight)
    assert torch.equal(a.ids, b.ids) and torch.equal(a.adv, b.adv)


# ------------------------------------------------------ logit transforms ---

def test_temperature_and_scale_equal_rescaled_weights():
    # z / T = h . (W / T) and z * a / b = h . (W * a / b): exact identities.
    h = _rand((7, 12), 40)
    W = _rand((60, 12), 41, 0.5)
    y = np.arange(7) * 8
    lp_t, _ = oracle.selective_logp(h, W, y, xf=oracle.Transform(temperature=0.7))
    lp_w, _ = oracle.selective_logp(h, W / 0.7, y)
    assert np.allclose(lp_t, lp_w, rtol=0, atol=1e-12)
    lp_s, _ = oracle.selective_logp(h, W, y, xf=oracle.Transform(scale_mul=3.0, scale_div=2.0))
    lp_w2, _ = oracle.selective_logp(h, W * 1.5, y)
    assert np.allclose(lp_s, lp_w2, rtol=0, atol=1e-12)


def test_softcap_saturation_closed_form():
    # Two entries with logits far beyond the cap: z' = +-cap / T, so
    # logp(y=0) = -log1p(exp(-2 cap / T)).
    cap, T = 5.0, 0.8
    h = np.array([[1.0, 0.0]])
    W = np.array([[1e4, 0.0], [-1e4, 0.0]])
    lp, _ = oracle.selective_logp(h, W, [0], xf=oracle.Transform(softcap=cap, temperature=T))
    assert abs(lp[0] - (-math.log1p(math.exp(-2 * cap / T)))) < 1e-14


def test_large_softcap_tends_to_identity():
    h = _rand((5, 10), 42)
    W = _rand((30, 10), 43, 0.3)
    y = np.arange(5)
    a, _ = oracle.selective_logp(h, W, y)
    b, _ = oracle.selective_logp(h, W, y, xf=oracle.Transform(softcap=1e7))
    assert np.allclose(a, b, rtol=0, atol=1e-11)


def test_transform_matches_torch_fp64():
    h = _rand((6, 16), 44)
    W = _rand((50, 16), 45, 0.8)
    y = np.random.default_rng(46).integers(0, 50, 6)
    xf = oracle.Transform(scale_mul=1.5, scale_div=2.0, softcap=3.0, temperature=0.6)
    lp, _ = oracle.selective_logp(h, W, y, xf=xf)
    z = torch.tensor(h) @ torch.tensor(W).T
    zt = 3.0 * torch.tanh(z * 0.75 / 3.0) / 0.6
    ref = torch.log_softmax(zt, 1).gather(1, torch.tensor(y)[:, None])[:, 0]
    assert np.allclose(lp, ref.numpy(), rtol=0, atol=1e-12)


def _L_of_h_xf(h, W, y, mask, old, ref, adv, T, eps, beta, xf):
    lp, _ = oracle.selective_logp(h, W, y, xf=xf)
    return oracle.grpo_loss(lp, old, ref, adv, mask, T, eps, eps, beta)[0]


@pytest.mark.parametrize("xf", [
    oracle.Transform(softcap=2.0),
    oracle.Transform(scale_mul=2.0, scale_div=3.0, softcap=1.5, temperature=0.7),
    oracle.Transform(temperature=1.3)])
def test_transformed_dH_matches_finite_differences(xf):
    rng = np.random.default_rng(47)
    N, D, V, T = 6, 8, 40, 3
    h = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.5
    y = rng.integers(0, V, N)
    mask = np.ones(N)
    lp, _ = oracle.selective_logp(h, W, y, xf=xf)
    old = lp + rng.normal(0, 0.1, N)
    ref = lp + rng.normal(0, 0.1, N)
    adv = rng.standard_normal(N // T)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, 0.2, 0.2, 0.05, xf=xf)
    fd = np.zeros_like(h)
    step = 1e-6
    for t in range(N):
        for d in range(D):
            hp, hm = h.copy(), h.copy()
            hp[t, d] += step
            hm[t, d] -= step
            fd[t, d] = (_L_of_h_xf(hp, W, y, mask, old, ref, adv, T, 0.2, 0.05, xf)
                        - _L_of_h_xf(hm, W, y, mask, old, ref, adv, T, 0.2, 0.05, xf)) / (2 * step)
    assert np.linalg.norm(fd - out["dH"]) / np.linalg.norm(out["dH"]) < 1e-6
    # A backward that forgets the transform's derivative is caught.
    no_chain = oracle.grad_hidden(h, W, y, out["g"])
    assert np.linalg.norm(fd - no_chain) / np.linalg.norm(fd) > 1e-2


# ------------------------------------------------- per-sequence aggregation --

def test_sequence_mean_equals_token_mean_without_padding():
    logp, adv, mask, T, eps = _loss_case(50)
    rng = np.random.default_rng(51)
    old = logp + rng.normal(0, 0.1, 12)
    ref = logp + rng.normal(0, 0.1, 12)
    a = oracle.grpo_loss(logp, old, ref, adv, mask, T, eps, eps, 0.02)
    b = oracle.grpo_loss(logp, old, ref, adv, mask, T, eps, eps, 0.02, aggregation="sequence")
    assert abs(a[0] - b[0]) < 1e-15 and np.allclose(a[1], b[1], atol=1e-17)


def test_sequence_mean_hand_case():
    # Two completions of T = 3: lengths 1 and 3, on-policy, beta = 0:
    # l_t = -A_b, so L = (1/2) * (-A_0 + (-A_1)) whatever the lengths.
    logp = np.array([-1.0, -2.0, -3.0, -1.5, -2.5, -0.5])
    mask = np.array([1, 0, 0, 1, 1, 1])
    adv = np.array([0.7, -0.3])
    L, g, _, B = oracle.grpo_loss(logp, logp, logp, adv, mask, 3, 0.2, 0.2, 0.0,
                                  aggregation="sequence")
    assert B == 2.0 and abs(L - (-(0.7 - 0.3) / 2)) < 1e-15
    assert np.allclose(g, [-0.7 / 2, 0, 0, 0.3 / 6, 0.3 / 6, 0.3 / 6], atol=1e-16)
    # Token mean weighs the long completion three times as much.
    Lt, _, _, _ = oracle.grpo_loss(logp, logp, logp, adv, mask, 3, 0.2, 0.2, 0.0)
    assert abs(Lt - (-(0.7 - 3 * 0.3) / 4)) < 1e-15


def test_sequence_mean_empty_completion_and_fd():
    rng = np.random.default_rng(52)
    T = 4
    logp = -rng.uniform(1, 5, 12)
    mask = np.array([1, 1, 0, 0, 0, 0, 0, 0, 1, 1, 1, 0])  # completion 1 is empty
    adv = rng.standard_normal(3)
    old = logp + rng.normal(0, 0.1, 12)
    ref = logp + rng.normal(0, 0.1, 12)
    L, g, _, B = oracle.grpo_loss(logp, old, ref, adv, mask, T, 0.2, 0.2, 0.05,
                                  aggregation="sequence")
    assert B == 2.0
    step = 1e-6
    for t in range(12):
        p_, m_ = logp.copy(), logp.copy()
        p_[t] += step
        m_[t] -= step
        fd = (oracle.grpo_loss(p_, old, ref, adv, mask, T, 0.2, 0.2, 0.05, aggregation="sequence")[0]
              - oracle.grpo_loss(m_, old, ref, adv, mask, T, 0.2, 0.2, 0.05,
                                 aggregation="sequence")[0]) / (2 * step)
        assert abs(fd - g[t]) < 1e-8


# ------------------------------------------------------ lm_head gradient ---

@pytest.mark.parametrize("xf", [oracle.IDENTITY, oracle.Transform(softcap=2.0, temperature=0.8)])
def test_dW_matches_finite_differences(xf):
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(70, N=8, D=5, V=12)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta, xf=xf)
    dW = oracle.grad_weight(h, W, y, out["g"], xf=xf)
    step = 1e-6
    fd = np.zeros_like(W)
    for v in range(W.shape[0]):
        for d in range(W.shape[1]):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, d] += step
            Wm[v, d] -= step
            fd[v, d] = (_L_of_h_xf(h, Wp, y, mask, old, ref, adv, T, eps, beta, xf)
                        - _L_of_h_xf(h, Wm, y, mask, old, ref, adv, T, eps, beta, xf)) / (2 * step)
    assert np.linalg.norm(fd - dW) / np.linalg.norm(fd) < 1e-6


def test_dW_columns_sum_to_zero():
    # sum_v (onehot - softmax)_v = 0 for every token, so sum_v dW_v = 0.
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(71)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)
    dW = oracle.grad_weight(h, W, y, out["g"])
    assert np.abs(dW.sum(axis=0)).max() < 1e-14 * max(1.0, np.abs(dW).max()) * W.shape[0]
    assert np.abs(dW).max() > 1e-6


def test_dW_matches_torch_autograd():
    h, W, y, mask, old, ref, adv, T, eps, beta = _tiny_full(72)
    out = oracle.loss_fwd_bwd(h, W, y, mask, old, ref, adv, T, eps, eps, beta)
    dW = oracle.grad_weight(h, W, y, out["g"])
    Wt = torch.tensor(W, requires_grad=True)
    lp = torch.log_softmax(torch.tensor(h) @ Wt.T, 1).gather(1, torch.tensor(y)[:, None])[:, 0]
    A = torch.tensor(adv)[torch.arange(len(y)) // T]
    r = torch.exp(lp - torch.tensor(old))
    surr = torch.minimum(r * A, torch.clamp(r, 1 - eps, 1 + eps) * A)
    dl = torch.tensor(ref) - lp
    m = torch.tensor(mask)
    L = ((-surr + beta * (torch.exp(dl) - dl - 1)) * m).sum() / m.sum()
    L.backward()
    assert np.allclose(Wt.grad.numpy(), dW, rtol=1e-10, atol=1e-14)
