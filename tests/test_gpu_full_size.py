"""Full-size GPU parity on the four large workloads, for both backward forms
(flags 1 = stored fp16 logits, the form the library chooses by default when
no workspace budget is set and the form bench.py times; flags 32 = the single
pass over vocabulary blocks; flags 16 = recomputed logit tiles), each with its
automatic plan as bench.py launches it.

The oracle cannot afford all N x V logits in fp64 at these sizes, so:
  * logp and dH are compared on a seeded sample of rows. Given the loss
    denominator M, a row's logp, g and dH depend on that row alone, so the
    oracle's values for sampled rows are exact, not estimates.
  * the loss is compared exactly in a second call whose mask keeps only the
    sampled rows (M = sample size), same shapes and hidden states;
  * for the Llama-3.1-8B shape (the bench workload) the oracle also computes
    every row's logp, so the loss of the full call is compared exactly.
Masked rows in the sample must have logp = 0 and dH exactly 0.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LOGP_TOL = 1e-2
LOSS_RTOL = 1e-3
DH_RTOL = 2e-2
DEV = "cuda:0"
N_SAMPLE = 192
N_SAMPLE_MASKED = 32


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def _sample_rows(p, seed):
    rng = np.random.default_rng(seed)
    m = p.mask.numpy().astype(bool)
    valid = np.nonzero(m)[0]
    masked = np.nonzero(~m)[0]
    rows = rng.choice(valid, size=min(N_SAMPLE, len(valid)), replace=False)
    mrows = rng.choice(masked, size=min(N_SAMPLE_MASKED, len(masked)), replace=False)
    # Always include the first and last valid rows (tile and chunk edges).
    rows = np.unique(np.concatenate([rows, valid[:1], valid[-1:]]))
    return np.sort(rows), np.sort(mrows)


def _run(clp, p, mask, old, ref, flags=16):
    dev = torch.device(DEV)
    args = [t.to(dev) for t in (p.hidden, p.weight, p.ids, mask, old, ref, p.adv)]
    params = clp.make_params(flags=flags)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws)
    st = clp.grpo_read_device_status(ws)
    return loss.item(), logp.cpu(), dH, st


@pytest.mark.parametrize("flags", [16, 1, 32], ids=["recompute", "stored", "single_pass"])
@pytest.mark.parametrize("name", ["qwen2.5-1.5b", "llama-3.1-8b", "qwen3-8b-long",
                                  "gpt-oss-20b-long"])
def test_full_size_sampled_rows(clp, name, flags):
    p = synth.make_problem(name, seed=1)
    rows, mrows = _sample_rows(p, seed=2)
    W64 = p.weight.float().numpy().astype(np.float64)
    lp_rows, _ = oracle.selective_logp(p.hidden[rows], W64, p.ids.numpy()[rows])
    base = torch.full((p.n_tokens,), -math.log(p.vocab), dtype=torch.float64)
    base[rows] = torch.from_numpy(lp_rows)
    old, ref = p.old_ref(base)
    M = float(p.mask.sum())

    # (1) the workload itself: sampled rows of logp and dH.
    L, logp, dH, st = _run(clp, p, p.mask, old, ref, flags)
    assert st == 0
    want = oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), rows, old, ref, p.adv,
                               p.seq_len, M, p.eps_low, p.eps_high, p.beta)
    got_lp = logp.double().numpy()[rows]
    got_dh = dH[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    dl = np.abs(got_lp - want["logp"]).max()
    rel_dh = np.linalg.norm(got_dh - want["dH"]) / np.linalg.norm(want["dH"])
    print(f"{name}: rows={len(rows)} max|dlogp|={dl:.3e} rel_dH={rel_dh:.3e}")
    assert dl <= LOGP_TOL and rel_dh <= DH_RTOL
    if len(mrows):
        assert torch.all(logp[mrows] == 0)
        assert torch.all(dH[torch.from_numpy(mrows).to(DEV)] == 0)
    assert math.isfinite(L)

    # (2) same shapes, mask = sampled rows only: the loss is exact.
    mask2 = torch.zeros_like(p.mask)
    mask2[rows] = 1
    L2, logp2, dH2, st2 = _run(clp, p, mask2, old, ref, flags)
    assert st2 == 0
    lp_full = np.zeros(p.n_tokens)
    lp_full[rows] = lp_rows
    L_want, _, _, M2 = oracle.grpo_loss(lp_full, old, ref, p.adv, mask2, p.seq_len,
                                        p.eps_low, p.eps_high, p.beta)
    rel_loss = abs(L2 - L_want) / abs(L_want)
    got_dh2 = dH2[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    want_dh2 = want["dH"] * (M / M2)  # dH is linear in g, and g scales as 1/M
    rel_dh2 = np.linalg.norm(got_dh2 - want_dh2) / np.linalg.norm(want_dh2)
    print(f"{name}: sampled-mask loss={L2:.6e} want={L_want:.6e} rel={rel_loss:.3e} "
          f"rel_dH={rel_dh2:.3e}")
    assert rel_loss <= LOSS_RTOL and rel_dh2 <= DH_RTOL
    other = torch.ones(p.n_tokens, dtype=torch.bool)
    other[rows] = False
    assert torch.all(logp2[other] == 0)
    assert int((dH2[other.to(DEV)] != 0).sum()) == 0


@pytest.fixture(scope="module")
def llama_full_oracle():
    # Every row through the oracle (about 1.7e13 fp64 flops), once for both forms.
    p = synth.make_problem("llama-3.1-8b", seed=3)
    W64 = p.weight.float().numpy().astype(np.float64)
    lp, _ = oracle.selective_logp(p.hidden, W64, p.ids.numpy(), row_block=256)
    return p, lp


@pytest.mark.parametrize("flags", [1, 16, 32], ids=["stored", "recompute", "single_pass"])
def test_llama_full_loss_exact(clp, llama_full_oracle, flags):
    # The loss of the bench's own workload, exactly, with old/ref = oracle logp
    # + noise: every row's logp enters it.
    p, lp = llama_full_oracle
    old, ref = p.old_ref(torch.from_numpy(lp))
    L, logp, dH, st = _run(clp, p, p.mask, old, ref, flags)
    assert st == 0
    L_want, g, _, _ = oracle.grpo_loss(lp, old, ref, p.adv, p.mask, p.seq_len,
                                       p.eps_low, p.eps_high, p.beta)
    d = np.abs(logp.double().numpy() - lp)
    rel = abs(L - L_want) / abs(L_want)
    print(f"llama full (flags {flags}): max|dlogp|={d.max():.3e} rms={np.sqrt((d ** 2).mean()):.3e} "
          f"loss={L:.6e} want={L_want:.6e} rel={rel:.3e}")
    assert d.max() <= LOGP_TOL and rel <= LOSS_RTOL


def test_llama_lm_head_gradient_column_sums(clp):
    # sum_v (onehot - softmax)_v = 0 per token, so the columns of dW sum to ~0 at
    # any size: a full-size property check of the dW GEMM (both backward modes).
    p = synth.make_problem("llama-3.1-8b", seed=4)
    old = torch.full((p.n_tokens,), -12.0)
    dev = torch.device(DEV)
    args = [t.to(dev) for t in (p.hidden, p.weight, p.ids, p.mask, old, old, p.adv)]
    for flags in (16, 1):
        params = clp.make_params(flags=flags)
        _, _, _, dW = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, want_dW=True)
        colsum = dW.double().sum(dim=0).abs().max().item()
        scale = dW.double().abs().sum(dim=0).max().item()
        print(f"llama dW flags={flags}: max|col sum|={colsum:.3e} vs col |.| sum {scale:.3e}")
        assert torch.isfinite(dW).all() and colsum <= 2e-2 * scale


@pytest.mark.parametrize("flags", [1, 16, 32], ids=["stored", "recompute", "single_pass"])
def test_qwen3_head_chunk_sweep(clp, flags):
    # The Qwen3-8B long-context head (D = 4096, V = 151936) with the workload's
    # chunk sweep of 1K, 4K and 16K rows, on a reduced batch (3 completions in
    # 3 x 12288 slots, lengths U[1024, 12288]) that still gives several chunks
    # of 16K rows, so the stored form's double-buffered blocks and side-stream
    # G pass are used at every chunk size.
    p = synth.make_problem("qwen3-8b-long", seed=5, prompts=1, G=3, T=12288,
                           lengths=(1024, 12288))
    rows, mrows = _sample_rows(p, seed=6)
    W64 = p.weight.float().numpy().astype(np.float64)
    lp_rows, _ = oracle.selective_logp(p.hidden[rows], W64, p.ids.numpy()[rows])
    base = torch.full((p.n_tokens,), -math.log(p.vocab), dtype=torch.float64)
    base[rows] = torch.from_numpy(lp_rows)
    old, ref = p.old_ref(base)
    M = float(p.mask.sum())
    want = oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), rows, old, ref, p.adv,
                               p.seq_len, M, p.eps_low, p.eps_high, p.beta)
    dev = torch.device(DEV)
    args = [t.to(dev) for t in (p.hidden, p.weight, p.ids, p.mask, old, ref, p.adv)]
    idx = torch.from_numpy(rows).to(dev)
    out = {}
    for chunk in (1024, 4096, 16384):
        params = clp.make_params(chunk_tokens=chunk, flags=flags)
        plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
        ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
        loss, logp, dH = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws)
        assert clp.grpo_read_device_status(ws) == 0
        got_lp = logp.cpu().double().numpy()[rows]
        got_dh = dH[idx].double().cpu().numpy()
        dl = np.abs(got_lp - want["logp"]).max()
        rel_dh = np.linalg.norm(got_dh - want["dH"]) / np.linalg.norm(want["dH"])
        active_chunks = -(-int(p.mask.view(-1, 128).amax(1).sum()) * 128 // plan["chunk_rows"])
        print(f"chunk {chunk} ({active_chunks} active chunks of {plan['chunk_rows']} rows): "
              f"loss={loss.item():.8e} max|dlogp|={dl:.3e} rel_dH={rel_dh:.3e}")
        assert dl <= LOGP_TOL and rel_dh <= DH_RTOL
        assert torch.all(logp[torch.from_numpy(mrows).to(dev)] == 0)
        out[chunk] = (loss.clone(), logp.clone(), dH.clone(), active_chunks)
        del ws
    assert out[16384][3] >= 2  # several chunks even at the largest size
    L0, lp0, dh0, _ = out[1024]
    for chunk in (4096, 16384):
        L1, lp1, dh1, _ = out[chunk]
        # Every form's forward splits the vocabulary to fill whole rounds of SM
        # pairs at its chunk size, so the fp32 sums run in a chunk-dependent
        # order: the results agree to rounding, not bit for bit.
        assert (lp0 - lp1).abs().max().item() <= 1e-4
        assert abs(L0.item() - L1.item()) <= 1e-5 * abs(L0.item())
