"""GPU parity of the tail split of the stored-logit backward's dH launches.

A dH launch runs units (row unit x hidden tile, each a K loop over the whole
vocabulary) one per SM pair and round. When its last round has fewer units
than pairs, each of those units runs on its own pair up to a balance point
(its main piece) and idle pairs share the units' tails, cut at K-stage
boundaries; cut pieces leave fp32 partial tiles that a fixup pass adds in a
fixed order. (The split applies when no G pass runs beside the dH GEMM: the
fused form, or a single chunk.) These cases make the device cut units in
every way the split can: fewer units than pairs, a ragged last hidden tile
(cheaper stages: those units keep no tail), the fused dH GEMM that forms G on
chip, the single-CTA variant, whole rounds followed by a split last round,
several chunks, and padding that leaves fewer active row blocks than the host
planned for. Each is compared with the fp64 oracle (all rows, or a seeded
sample of rows where the oracle would be slow), and repeated calls must give
bitwise identical results: the sum of a unit's pieces never depends on which
pair finishes first.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

LOGP_TOL = 1e-2
LOSS_RTOL = 1e-3
DH_RTOL = 2e-2
DEV = "cuda:0"
STORED = 1       # GRPO_FLAG_STORED_LOGITS
SINGLE_CTA = 2   # GRPO_FLAG_SINGLE_CTA


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def _call(clp, p, old, ref, flags, chunk=0, mask="p"):
    mask = p.mask if isinstance(mask, str) else mask
    dev = torch.device(DEV)
    params = clp.make_params(flags=flags, chunk_tokens=chunk)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        p.hidden.to(dev), p.weight.to(dev), p.ids.to(dev),
        mask.to(dev) if mask is not None else None, old.to(dev), ref.to(dev), p.adv.to(dev),
        p.seq_len, params=params, workspace=ws)
    st = clp.grpo_read_device_status(ws)
    return loss.item(), logp.cpu(), dH, st


# name, prompts, G, T, D, V, lengths, flags, chunk tokens
# (units of the dH launch on GB300's 76 SM pairs / 152 SMs in the comments)
FULL_ORACLE = [
    # 2 row units x 6 hidden tiles (the last 320 of 512 columns): 12 units on
    # 12 pairs plus 25 tail pairs, several tail pieces per unit; the narrow
    # units keep no tail. G formed by its own pass (one chunk: not overlapped).
    ("ragged_tile_many_pieces", 1, 4, 128, 2880, 20000, None, STORED, 0),
    # the fused dH GEMM (G on chip); trailing padding: the device sees fewer
    # active row blocks than the 4 row units x 3 tiles the host planned.
    ("fused_padded", 1, 4, 256, 1536, 16384, (40, 256), STORED, 0),
    # single-CTA GEMMs: 128-row x 256-column units, 4 x 6 = 24 on 152 slots.
    ("single_cta", 1, 4, 128, 1536, 12000, None, STORED | SINGLE_CTA, 0),
    # two chunks of at most 3 row units (fused form): each launch cuts its units.
    ("two_chunks", 1, 4, 256, 2048, 9000, (100, 256), STORED, 768),
]


@pytest.mark.parametrize("name,prompts,G,T,D,V,lengths,flags,chunk", FULL_ORACLE,
                         ids=[c[0] for c in FULL_ORACLE])
def test_tail_split_against_oracle(clp, name, prompts, G, T, D, V, lengths, flags, chunk):
    p = synth.make_problem("tiny", seed=D + V, prompts=prompts, G=G, T=T, D=D, V=V,
                           lengths=lengths)
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(np.asarray(base)))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta)
    L, logp, dH, st = _call(clp, p, old, ref, flags, chunk)
    assert st == 0
    m = p.mask.numpy().astype(bool)
    lp = logp.double().numpy()
    dh = dH.double().cpu().numpy()
    dl = np.abs(lp - want["logp"]).max()
    rel_loss = abs(L - want["L"]) / abs(want["L"])
    rel_dh = np.linalg.norm(dh[m] - want["dH"][m]) / np.linalg.norm(want["dH"][m])
    print(f"{name}: max|dlogp|={dl:.3e} rel_loss={rel_loss:.3e} rel_dH={rel_dh:.3e}")
    assert dl <= LOGP_TOL and rel_loss <= LOSS_RTOL and rel_dh <= DH_RTOL
    assert np.all(lp[~m] == 0.0) and np.all(dh[~m] == 0.0)
    # Every row, not only in aggregate: no unit's pieces were dropped or doubled.
    row_err = np.linalg.norm(dh[m] - want["dH"][m], axis=1)
    row_ref = np.linalg.norm(want["dH"][m], axis=1)
    assert np.all(row_err <= 0.05 * row_ref + 1e-6)
    # Repeated calls: bitwise the same.
    L2, logp2, dH2, st2 = _call(clp, p, old, ref, flags, chunk)
    assert st2 == 0 and L2 == L
    assert torch.equal(logp2, logp) and torch.equal(dH2, dH)


def test_tail_split_whole_rounds_then_a_split_round(clp):
    # 20 row units x 8 hidden tiles = 160 units on 76 pairs: units 0..151 run
    # whole in two rounds, the last 8 are split with 9 tail pairs. The oracle
    # checks a seeded sample of rows (each row's dH depends on that row alone,
    # given the loss denominator), among them the first and last rows.
    p = synth.make_problem("tiny", seed=7, prompts=1, G=4, T=1280, D=4096, V=9000,
                           lengths=None)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([rng.choice(p.n_tokens, 96, replace=False),
                                     [0, 2559, 2560, 5119]]))
    W64 = p.weight.float().numpy().astype(np.float64)
    lp_rows, _ = oracle.selective_logp(p.hidden[rows], W64, p.ids.numpy()[rows])
    base = torch.full((p.n_tokens,), -math.log(p.vocab), dtype=torch.float64)
    base[rows] = torch.from_numpy(lp_rows)
    old, ref = p.old_ref(base)
    M = float(p.mask.sum())
    L, logp, dH, st = _call(clp, p, old, ref, STORED, chunk=5120)
    assert st == 0 and math.isfinite(L)
    want = oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), rows, old, ref, p.adv,
                               p.seq_len, M, p.eps_low, p.eps_high, p.beta)
    got_lp = logp.double().numpy()[rows]
    got_dh = dH[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    dl = np.abs(got_lp - want["logp"]).max()
    rel_dh = np.linalg.norm(got_dh - want["dH"]) / np.linalg.norm(want["dH"])
    print(f"whole rounds + split round: rows={len(rows)} max|dlogp|={dl:.3e} rel_dH={rel_dh:.3e}")
    assert dl <= LOGP_TOL and rel_dh <= DH_RTOL
    row_err = np.linalg.norm(got_dh - want["dH"], axis=1)
    assert np.all(row_err <= 0.05 * np.linalg.norm(want["dH"], axis=1) + 1e-6)
    # Without a mask the host knows every row block is active; the result is
    # the same as with an all-ones mask, bit for bit.
    L0, logp0, dH0, st0 = _call(clp, p, old, ref, STORED, chunk=5120, mask=None)
    assert st0 == 0 and L0 == L
    assert torch.equal(logp0, logp) and torch.equal(dH0, dH)


def test_tail_split_whole_rounds_without_a_mask(clp):
    # 19 row units x 4 hidden tiles = 76 units: one whole round, no unit cut.
    # With and without a mask (the host then skips the fixup pass) the dH
    # rows agree bit for bit, and with the oracle on sampled rows.
    p = synth.make_problem("tiny", seed=9, prompts=1, G=4, T=1216, D=2048, V=8448,
                           lengths=None)
    rows = np.array([0, 255, 256, 2431, 2432, 4863])
    W64 = p.weight.float().numpy().astype(np.float64)
    lp_rows, _ = oracle.selective_logp(p.hidden[rows], W64, p.ids.numpy()[rows])
    base = torch.full((p.n_tokens,), -math.log(p.vocab), dtype=torch.float64)
    base[rows] = torch.from_numpy(lp_rows)
    old, ref = p.old_ref(base)
    L, logp, dH, st = _call(clp, p, old, ref, STORED, chunk=4864)
    L0, logp0, dH0, st0 = _call(clp, p, old, ref, STORED, chunk=4864, mask=None)
    assert st == 0 and st0 == 0 and L0 == L
    assert torch.equal(logp0, logp) and torch.equal(dH0, dH)
    want = oracle.rows_fwd_bwd(p.hidden, W64, p.ids.numpy(), rows, old, ref, p.adv,
                               p.seq_len, float(p.mask.sum()), p.eps_low, p.eps_high, p.beta)
    got_dh = dH[torch.from_numpy(rows).to(DEV)].double().cpu().numpy()
    rel_dh = np.linalg.norm(got_dh - want["dH"]) / np.linalg.norm(want["dH"])
    assert rel_dh <= DH_RTOL


def test_tail_split_with_the_lm_head_gradient(clp):
    # With dW the stored form forms G in a pass of its own and the dW GEMM reads
    # the same G block after the dH launch, its tail split and the fixup (one
    # chunk: the unoverlapped schedule). 2 pair row units x 3 hidden tiles = 6
    # units, cut with 11 tail pairs (tail shares of at least 64 full stages).
    p = synth.make_problem("tiny", seed=11, prompts=1, G=4, T=128, D=1536, V=12000,
                           lengths=(40, 128))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(np.asarray(base)))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta)
    want_dW = oracle.grad_weight(p.hidden, p.weight, p.ids.numpy(), want["g"])
    dev = torch.device(DEV)
    params = clp.make_params(flags=STORED)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
    outs = []
    for _ in range(2):
        dW = torch.full((p.vocab, p.hidden_size), float("nan"), device=dev)
        loss, logp, dH, dW = clp.grpo_loss_fwd_bwd(
            p.hidden.to(dev), p.weight.to(dev), p.ids.to(dev), p.mask.to(dev), old.to(dev),
            ref.to(dev), p.adv.to(dev), p.seq_len, params=params, workspace=ws, dW=dW)
        assert clp.grpo_read_device_status(ws) == 0
        outs.append((loss.item(), logp.cpu(), dH.cpu(), dW.cpu()))
    L, logp, dH, dW = outs[0]
    m = p.mask.numpy().astype(bool)
    dh = dH.double().numpy()
    rel_dh = np.linalg.norm(dh[m] - want["dH"][m]) / np.linalg.norm(want["dH"][m])
    rel_dw = np.linalg.norm(dW.double().numpy() - want_dW) / np.linalg.norm(want_dW)
    print(f"with dW: rel_dH={rel_dh:.3e} rel_dW={rel_dw:.3e}")
    assert np.abs(logp.double().numpy() - want["logp"]).max() <= LOGP_TOL
    assert abs(L - want["L"]) / abs(want["L"]) <= LOSS_RTOL
    assert rel_dh <= DH_RTOL and rel_dw <= DH_RTOL and np.all(dh[~m] == 0.0)
    L2, logp2, dH2, dW2 = outs[1]
    assert L2 == L and torch.equal(dH2, dH) and torch.equal(logp2, logp)


SINGLE_PASS = 32  # GRPO_FLAG_SINGLE_PASS

# name, prompts, G, T, D, V, lengths, chunk tokens, vocab block
SINGLE_PASS_CASES = [
    # 4 pair row units x 3 hidden tiles per U GEMM launch, 4 vocabulary blocks
    # (the first, middle and last U updates all go through the fixup when cut).
    ("sp_blocks", 1, 4, 256, 1536, 40000, (40, 256), 0, 12800),
    # two chunks, ragged last block, a hidden size with a narrow last tile
    ("sp_chunks", 1, 4, 256, 1280, 30000, (100, 256), 512, 9728),
]


@pytest.mark.parametrize("name,prompts,G,T,D,V,lengths,chunk,vblock", SINGLE_PASS_CASES,
                         ids=[c[0] for c in SINGLE_PASS_CASES])
def test_tail_split_single_pass(clp, name, prompts, G, T, D, V, lengths, chunk, vblock):
    # The single pass with P formed on chip: its U GEMM launches split like the
    # stored form's dH launches, and the fixup applies the U update (the
    # rescale by the running maximum, and dH on the last block) to the sum of
    # a cut unit's pieces.
    p = synth.make_problem("tiny", seed=D + V + 1, prompts=prompts, G=G, T=T, D=D, V=V,
                           lengths=lengths)
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(np.asarray(base)))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta)
    dev = torch.device(DEV)
    params = clp.make_params(flags=SINGLE_PASS, chunk_tokens=chunk, vocab_block=vblock)
    plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
    assert plan["single_pass"] == 1 and plan["g_in_dh_gemm"] == 1 and plan["n_vocab_blocks"] > 2
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
    args = [t.to(dev) for t in (p.hidden, p.weight, p.ids, p.mask)] + [old.to(dev), ref.to(dev),
                                                                       p.adv.to(dev)]
    outs = []
    clp.grpo_launch_timing_enable(True)
    try:
        for _ in range(2):
            loss, logp, dH = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws)
            assert clp.grpo_read_device_status(ws) == 0
            outs.append((loss.item(), logp.cpu(), dH.cpu()))
    finally:
        clp.grpo_launch_timing_enable(False)
    times = {k["name"]: k["launches"] for k in clp.grpo_launch_timing_read()}
    assert times.get("tail_fixup_kernel", 0) == 2 * plan["n_chunks"] * plan["n_vocab_blocks"]
    assert sum(times.values()) == 2 * plan["launches_loss"]
    L, logp, dH = outs[0]
    m = p.mask.numpy().astype(bool)
    dh = dH.double().numpy()
    dl = np.abs(logp.double().numpy() - want["logp"]).max()
    rel_loss = abs(L - want["L"]) / abs(want["L"])
    rel_dh = np.linalg.norm(dh[m] - want["dH"][m]) / np.linalg.norm(want["dH"][m])
    print(f"{name}: max|dlogp|={dl:.3e} rel_loss={rel_loss:.3e} rel_dH={rel_dh:.3e}")
    assert dl <= LOGP_TOL and rel_loss <= LOSS_RTOL and rel_dh <= DH_RTOL
    assert np.all(dh[~m] == 0.0)
    row_err = np.linalg.norm(dh[m] - want["dH"][m], axis=1)
    assert np.all(row_err <= 0.05 * np.linalg.norm(want["dH"][m], axis=1) + 1e-6)
    L2, logp2, dH2 = outs[1]
    assert L2 == L and torch.equal(logp2, logp) and torch.equal(dH2, dH)


def test_tail_split_overlapped_schedule_last_chunk(clp):
    # D > 2048 with several chunks: each chunk's G pass runs on a side stream
    # beside the previous chunk's dH launch, which therefore keeps whole units;
    # only the last chunk's dH launch, with nothing beside it, is split.
    # Lengths over 128 keep both row blocks of every completion active, so the
    # last chunk has units to split (trailing padding inside them).
    p = synth.make_problem("tiny", seed=13, prompts=1, G=4, T=256, D=2304, V=9000,
                           lengths=(200, 256))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(np.asarray(base)))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta)
    dev = torch.device(DEV)
    params = clp.make_params(flags=STORED, chunk_tokens=256)
    plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
    assert plan["g_in_dh_gemm"] == 0 and plan["n_chunks"] >= 3
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, dev)
    args = [t.to(dev) for t in (p.hidden, p.weight, p.ids, p.mask)] + [old.to(dev), ref.to(dev),
                                                                       p.adv.to(dev)]
    outs = []
    clp.grpo_launch_timing_enable(True)
    try:
        for _ in range(2):
            loss, logp, dH = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws)
            assert clp.grpo_read_device_status(ws) == 0
            outs.append((loss.item(), logp.cpu(), dH.cpu()))
    finally:
        clp.grpo_launch_timing_enable(False)
    times = {k["name"]: k["launches"] for k in clp.grpo_launch_timing_read()}
    assert times.get("tail_fixup_kernel", 0) == 2
    assert sum(times.values()) == 2 * plan["launches_loss"]
    L, logp, dH = outs[0]
    m = p.mask.numpy().astype(bool)
    dh = dH.double().numpy()
    rel_dh = np.linalg.norm(dh[m] - want["dH"][m]) / np.linalg.norm(want["dH"][m])
    print(f"overlapped, last chunk split: rel_dH={rel_dh:.3e}")
    assert np.abs(logp.double().numpy() - want["logp"]).max() <= LOGP_TOL
    assert abs(L - want["L"]) / abs(want["L"]) <= LOSS_RTOL and rel_dh <= DH_RTOL
    row_err = np.linalg.norm(dh[m] - want["dH"][m], axis=1)
    assert np.all(row_err <= 0.05 * np.linalg.norm(want["dH"][m], axis=1) + 1e-6)
    assert np.all(dh[~m] == 0.0)
    L2, logp2, dH2 = outs[1]
    assert L2 == L and torch.equal(logp2, logp) and torch.equal(dH2, dH)
