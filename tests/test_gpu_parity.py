"""GPU parity: the CUDA library (called through the C ABI) against the fp64
oracle on identical seeded bf16 inputs.

Gates: |d logp| <= 1e-2 absolute, relative loss error <= 1e-3, relative
Frobenius error of dH over unmasked rows <= 2e-2. Masked rows: logp = 0 and
dH exactly 0.
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
# Backward forms (grpo_params.flags): without either bit the call chooses.
STORED = 1        # GRPO_FLAG_STORED_LOGITS
RECOMPUTE = 16    # GRPO_FLAG_RECOMPUTE_LOGITS
SINGLE_PASS = 32  # GRPO_FLAG_SINGLE_PASS


@pytest.fixture(scope="module")
def clp():
    import __graft_entry__

    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


DEV = "cuda:0"


def _to(t):
    return t.to(DEV) if t is not None else None


def gpu_loss(clp, p, old, ref, params=None, mask=None, ids=None, hidden=None, weight=None):
    mask = p.mask if mask is None else mask
    ids = p.ids if ids is None else ids
    hidden = p.hidden if hidden is None else hidden
    weight = p.weight if weight is None else weight
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        _to(hidden), _to(weight), _to(ids), _to(mask), _to(old), _to(ref), _to(p.adv),
        p.seq_len, params=params, workspace=ws)
    st = clp.grpo_read_device_status(ws)
    return (loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st)


def oracle_case(p, mask=None, base=None, eps=None, beta=None):
    mask = p.mask if mask is None else mask
    if base is None:
        base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(np.asarray(base)))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), mask.numpy(), old, ref, p.adv,
                               p.seq_len, p.eps_low if eps is None else eps,
                               p.eps_high if eps is None else eps,
                               p.beta if beta is None else beta)
    return old, ref, want


def check(got, want, mask, tag=""):
    L, logp, dH, st = got
    m = mask.numpy().astype(bool)
    assert st == 0, f"{tag} device status {st}"
    dl = np.abs(logp - want["logp"])
    rel_loss = abs(L - want["L"]) / max(abs(want["L"]), 1e-30)
    num = np.linalg.norm(dH[m] - want["dH"][m])
    den = np.linalg.norm(want["dH"][m])
    rel_dh = num / den if den > 0 else num
    print(f"{tag}: max|dlogp|={dl.max():.3e} rms={np.sqrt((dl ** 2).mean()):.3e} "
          f"rel_loss={rel_loss:.3e} (L={want['L']:.6e}) rel_dH={rel_dh:.3e}")
    assert dl.max() <= LOGP_TOL
    assert rel_loss <= LOSS_RTOL
    assert rel_dh <= DH_RTOL
    assert np.all(logp[~m] == 0.0)
    assert np.all(dH[~m] == 0.0)


def test_logp_fwd_tiny(clp):
    p = synth.make_problem("tiny", seed=0)
    logp, lse = clp.grpo_logp_fwd(_to(p.hidden), _to(p.weight), _to(p.ids), want_lse=True)
    want, want_lse = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    d = np.abs(logp.cpu().double().numpy() - want)
    dl = np.abs(lse.cpu().double().numpy() - want_lse)
    print(f"logp tiny: max={d.max():.3e} rms={np.sqrt((d ** 2).mean()):.3e} lse max={dl.max():.3e}")
    assert d.max() <= LOGP_TOL and dl.max() <= LOGP_TOL


def test_loss_fwd_bwd_tiny(clp):
    p = synth.make_problem("tiny", seed=0)
    old, ref, want = oracle_case(p)
    check(gpu_loss(clp, p, old, ref), want, p.mask, "tiny")


# N, T, D, V, chunk_tokens, vocab_block, padded
RAGGED = [
    (300, 75, 200, 1000, 128, 512, True),     # tails in every dim; 3 chunks x 2 vocab blocks
    (129, 129, 64, 257, 0, 0, False),         # one row past a tile, one column past a tile
    (1000, 250, 136, 3000, 256, 1024, True),  # D not a multiple of 64
    (256, 64, 2880, 2000, 0, 0, True),        # gpt-oss hidden size
    (512, 128, 1536, 5000, 0, 768, True),     # Qwen2.5-1.5B hidden size, 7 vocab blocks
    (640, 640, 4096, 777, 0, 0, False),       # Llama hidden size, vocab < 1K
]


@pytest.mark.parametrize("N,T,D,V,chunk,vblock,padded", RAGGED)
def test_ragged_shapes(clp, N, T, D, V, chunk, vblock, padded):
    G = 4 if (N // T) % 4 == 0 else 1
    p = synth.make_problem("tiny", seed=N + D + V, prompts=(N // T) // G, G=G, T=T, D=D, V=V,
                           lengths=(max(1, T // 3), T) if padded else None)
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, vocab_block=vblock, flags=RECOMPUTE)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"ragged {N}x{D}x{V}")


# D = 2880: an odd number of 64-wide K slices (the pair GEMMs' last stage is half empty).
@pytest.mark.parametrize("D,V", [(200, 1000), (2880, 1300)])
def test_logp_fwd_ragged(clp, D, V):
    p = synth.make_problem("tiny", seed=3, T=75, prompts=1, G=4, D=D, V=V)
    logp, _ = clp.grpo_logp_fwd(_to(p.hidden), _to(p.weight), _to(p.ids))
    want, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    assert np.abs(logp.cpu().double().numpy() - want).max() <= LOGP_TOL


def test_chunking_does_not_change_results(clp):
    # "No loss of accuracy" from chunking. At this vocabulary (12 tiles) every
    # forward launch splits it into single tiles, whatever its chunk, so the
    # forward does not depend on the chunking (with more tiles the splits
    # follow each chunk's row units and results agree to rounding, as the
    # Qwen3-8B head's chunk sweep checks); dH rows depend on the chunk size
    # not at all, and on the vocab block only through fp32 accumulation
    # order.
    p = synth.make_problem("tiny", seed=11, T=128, prompts=1, G=4, D=256, V=3000,
                           lengths=(40, 128))
    old, ref, _ = oracle_case(p)
    runs = {}
    for chunk, vb in ((128, 0), (256, 0), (512, 0), (0, 256), (0, 1024), (128, 512)):
        runs[(chunk, vb)] = gpu_loss(clp, p, old, ref, clp.make_params(chunk_tokens=chunk,
                                                                      vocab_block=vb,
                                                                      flags=RECOMPUTE))
    L0, lp0, dH0, _ = runs[(128, 0)]
    for key, (L, lp, dH, st) in runs.items():
        assert st == 0
        assert L == L0 and np.array_equal(lp, lp0), key
        if key[1] == 0:
            assert np.array_equal(dH, dH0), key
        else:
            assert np.linalg.norm(dH - dH0) <= 1e-2 * np.linalg.norm(dH0), key


def test_all_masked_gives_zero(clp):
    p = synth.make_problem("tiny", seed=4)
    mask = torch.zeros_like(p.mask)
    old = torch.zeros(p.n_tokens)
    L, logp, dH, st = gpu_loss(clp, p, old, old, mask=mask)
    assert st == 0 and L == 0.0
    assert np.all(logp == 0) and np.all(dH == 0)


def test_masked_ids_are_never_read(clp):
    p = synth.make_problem("tiny", seed=5, lengths=(10, 64))
    ids = p.ids.clone()
    ids[p.mask == 0] = -12345  # would be out of range if read
    old, ref, want = oracle_case(p)
    check(gpu_loss(clp, p, old, ref, ids=ids), want, p.mask, "masked ids")


def test_bad_token_id_sets_status(clp):
    p = synth.make_problem("tiny", seed=6)
    ids = p.ids.clone()
    ids[7] = p.vocab  # unmasked and out of range
    old = torch.full((p.n_tokens,), -8.0)
    L, logp, dH, st = gpu_loss(clp, p, old, old, ids=ids)
    assert st == -8  # GRPO_ERR_BAD_TOKEN_ID
    assert math.isnan(logp[7]) and math.isnan(L)


def test_zero_weight_gives_uniform(clp):
    p = synth.make_problem("tiny", seed=7)
    W = torch.zeros_like(p.weight)
    logp, lse = clp.grpo_logp_fwd(_to(p.hidden), _to(W), _to(p.ids), want_lse=True)
    assert np.abs(logp.cpu().double().numpy() + math.log(p.vocab)).max() < 1e-5
    old = torch.full((p.n_tokens,), -math.log(p.vocab)) + 0.01
    L, lp, dH, st = gpu_loss(clp, p, old, old, weight=W)
    assert st == 0 and np.all(dH == 0)


def test_on_policy_identity(clp):
    # old = ref = logp: ratio 1 and zero KL, so loss = -mean masked advantage.
    p = synth.make_problem("tiny", seed=8, lengths=(20, 64))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    lp = torch.from_numpy(base).float()
    L, _, _, st = gpu_loss(clp, p, lp, lp)
    A = p.adv.double().numpy()[np.arange(p.n_tokens) // p.seq_len]
    m = p.mask.double().numpy()
    want = -(A * m).sum() / m.sum()
    assert st == 0 and abs(L - want) <= 1e-4 * max(1.0, abs(want))


def test_vocab_of_one(clp):
    p = synth.make_problem("tiny", seed=9, V=1)
    p.ids.zero_()
    logp, _ = clp.grpo_logp_fwd(_to(p.hidden), _to(p.weight), _to(p.ids))
    assert np.abs(logp.cpu().numpy()).max() < 1e-6


def test_empty_batch(clp):
    h = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(100, 64, device=DEV).to(torch.bfloat16)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    f = torch.empty(0, dtype=torch.float32, device=DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(h, W, e, torch.empty(0, dtype=torch.uint8, device=DEV),
                                           f, f, torch.empty(0, dtype=torch.float32, device=DEV),
                                           1)
    assert loss.item() == 0.0 and dH.numel() == 0


@pytest.mark.parametrize("chunk", [256, 0])
def test_padding_blocks_are_skipped_and_zeroed(clp, chunk):
    # Completions of 512 slots with 1..512 valid tokens: most 128-row blocks are
    # pure padding, skipped by every GEMM; their dH rows must still come out 0.
    p = synth.make_problem("tiny", seed=21 + chunk, prompts=2, G=4, T=512, D=256, V=3000,
                           lengths=(1, 512))
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, vocab_block=1024, flags=RECOMPUTE)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    dH = torch.full((p.n_tokens, p.hidden_size), float("nan"), dtype=torch.bfloat16, device=DEV)
    logp = torch.full((p.n_tokens,), float("nan"), device=DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        _to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old), _to(ref), _to(p.adv),
        p.seq_len, params=params, workspace=ws, dH=dH, logp=logp)
    st = clp.grpo_read_device_status(ws)
    got = (loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st)
    check(got, want, p.mask, f"padding chunk={chunk}")


@pytest.mark.parametrize("flags", [STORED, RECOMPUTE], ids=["stored", "recompute"])
@pytest.mark.parametrize("D", [256, 2304])
def test_splits_chosen_from_the_active_rows(clp, flags, D):
    # 16 row units of slots, about 2 of them active after padding: the logit
    # GEMM picks its vocab splits on the device from the active ones (not the
    # count the host plans for), and the row finish reads all 32 partial
    # slots of a row, the unused ones filled with (-inf, 0) by split 0.
    # Results match the oracle and repeat bit for bit.
    p = synth.make_problem("tiny", seed=71 + D, prompts=1, G=4, T=1024, D=D, V=9000,
                           lengths=(1, 150))
    old, ref, want = oracle_case(p)
    params = clp.make_params(flags=flags)
    plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
    assert plan["n_chunks"] >= 1
    got = gpu_loss(clp, p, old, ref, params)
    check(got, want, p.mask, f"active-row splits flags={flags} D={D}")
    again = gpu_loss(clp, p, old, ref, params)
    assert got[0] == again[0]
    assert np.array_equal(got[1], again[1]) and np.array_equal(got[2], again[2])


XFORMS = [
    dict(temperature=0.7),
    dict(logit_softcapping=30.0),
    dict(logit_softcapping=2.0),
    dict(logit_scale_multiply=1.5, logit_scale_divide=2.0, logit_softcapping=3.0,
         temperature=0.9),
    dict(logit_scale_multiply=0.5),
]


@pytest.mark.parametrize("kw", XFORMS)
def test_logit_transforms(clp, kw):
    # Logit std ~2.8 (W ~ N(0, 0.2^2), D = 200) so that softcaps of 2-3 saturate.
    p = synth.make_problem("tiny", seed=31, T=75, prompts=1, G=4, D=200, V=3000,
                           lengths=(20, 75), weight_std=0.2)
    xf = oracle.Transform(scale_mul=kw.get("logit_scale_multiply", 1.0),
                          scale_div=kw.get("logit_scale_divide", 1.0),
                          softcap=kw.get("logit_softcapping", 0.0),
                          temperature=kw.get("temperature", 1.0))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy(), xf=xf)
    old, ref = p.old_ref(torch.from_numpy(base))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta, xf=xf)
    params = clp.make_params(chunk_tokens=128, vocab_block=1024, flags=RECOMPUTE, **kw)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"transform {kw}")
    lp, _ = clp.grpo_logp_fwd(_to(p.hidden), _to(p.weight), _to(p.ids), params=params)
    assert np.abs(lp.cpu().double().numpy() - base).max() <= LOGP_TOL


# ---------------------------------------------- stored-logit backward ------



@pytest.mark.parametrize("N,T,D,V,chunk,vblock,padded", RAGGED)
def test_stored_logits_ragged(clp, N, T, D, V, chunk, vblock, padded):
    G = 4 if (N // T) % 4 == 0 else 1
    p = synth.make_problem("tiny", seed=N + D + V + 1, prompts=(N // T) // G, G=G, T=T, D=D,
                           V=V, lengths=(max(1, T // 3), T) if padded else None)
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, flags=STORED)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"stored {N}x{D}x{V}")


# Hidden sizes on either side of the switch between G formed inside the dH
# GEMM (D <= 2048) and G formed in a pass of its own over the logit block.
@pytest.mark.parametrize("D", [200, 2176])
@pytest.mark.parametrize("kw", XFORMS)
def test_stored_logits_transforms(clp, kw, D):
    p = synth.make_problem("tiny", seed=32, T=75, prompts=1, G=4, D=D, V=3000,
                           lengths=(20, 75), weight_std=0.2 if D < 1000 else 0.06)
    xf = oracle.Transform(scale_mul=kw.get("logit_scale_multiply", 1.0),
                          scale_div=kw.get("logit_scale_divide", 1.0),
                          softcap=kw.get("logit_softcapping", 0.0),
                          temperature=kw.get("temperature", 1.0))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy(), xf=xf)
    old, ref = p.old_ref(torch.from_numpy(base))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta, xf=xf)
    params = clp.make_params(chunk_tokens=128, flags=STORED, **kw)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"stored transform {kw}")


@pytest.mark.parametrize("chunk", [256, 0])
def test_stored_logits_padding_blocks(clp, chunk):
    p = synth.make_problem("tiny", seed=41 + chunk, prompts=2, G=4, T=512, D=256, V=3000,
                           lengths=(1, 512))
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, flags=STORED)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    dH = torch.full((p.n_tokens, p.hidden_size), float("nan"), dtype=torch.bfloat16, device=DEV)
    logp = torch.full((p.n_tokens,), float("nan"), device=DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        _to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old), _to(ref), _to(p.adv),
        p.seq_len, params=params, workspace=ws, dH=dH, logp=logp)
    st = clp.grpo_read_device_status(ws)
    got = (loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st)
    check(got, want, p.mask, f"stored padding chunk={chunk}")


# ------------------------------------------------ single-pass backward -----

# vocab_block: the vocabulary in several blocks (their logits, partial slots
# and the rescaled U accumulator), with a ragged last block.
@pytest.mark.parametrize("N,T,D,V,chunk,vblock,padded", RAGGED)
def test_single_pass_ragged(clp, N, T, D, V, chunk, vblock, padded):
    G = 4 if (N // T) % 4 == 0 else 1
    p = synth.make_problem("tiny", seed=N + D + V + 5, prompts=(N // T) // G, G=G, T=T, D=D,
                           V=V, lengths=(max(1, T // 3), T) if padded else None)
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, vocab_block=vblock, flags=SINGLE_PASS)
    plan = clp.grpo_get_plan(p.n_tokens, D, V, T, params)
    assert plan["single_pass"] == 1 and plan["stored_logits"] == 0
    check(gpu_loss(clp, p, old, ref, params), want, p.mask,
          f"single pass {N}x{D}x{V} ({plan['n_vocab_blocks']} blocks)")


# D = 200: P formed on chip; D = 2176: by a pass of its own, double-buffered
# beside the next block's logit GEMM (12 or 4 blocks) or not (1 block).
@pytest.mark.parametrize("D", [200, 2176])
@pytest.mark.parametrize("vblock", [256, 768, 0])
@pytest.mark.parametrize("kw", XFORMS)
def test_single_pass_transforms(clp, kw, vblock, D):
    # Logit std ~2.8 so that softcaps of 2-3 saturate.
    p = synth.make_problem("tiny", seed=33, T=75, prompts=1, G=4, D=D, V=3000,
                           lengths=(20, 75), weight_std=0.2 if D < 1000 else 0.06)
    xf = oracle.Transform(scale_mul=kw.get("logit_scale_multiply", 1.0),
                          scale_div=kw.get("logit_scale_divide", 1.0),
                          softcap=kw.get("logit_softcapping", 0.0),
                          temperature=kw.get("temperature", 1.0))
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy(), xf=xf)
    old, ref = p.old_ref(torch.from_numpy(base))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta, xf=xf)
    params = clp.make_params(chunk_tokens=128, vocab_block=vblock, flags=SINGLE_PASS, **kw)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"single pass transform {kw}")


@pytest.mark.parametrize("chunk", [256, 0])
def test_single_pass_padding_blocks(clp, chunk):
    p = synth.make_problem("tiny", seed=42 + chunk, prompts=2, G=4, T=512, D=256, V=3000,
                           lengths=(1, 512))
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, vocab_block=1024, flags=SINGLE_PASS)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    dH = torch.full((p.n_tokens, p.hidden_size), float("nan"), dtype=torch.bfloat16, device=DEV)
    logp = torch.full((p.n_tokens,), float("nan"), device=DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(
        _to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old), _to(ref), _to(p.adv),
        p.seq_len, params=params, workspace=ws, dH=dH, logp=logp)
    st = clp.grpo_read_device_status(ws)
    got = (loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st)
    check(got, want, p.mask, f"single pass padding chunk={chunk}")


@pytest.mark.parametrize("D", [320, 2304])
def test_single_pass_many_chunks_and_blocks(clp, D):
    # 4 chunks x 3 vocab blocks, padded: at D = 2304 the P pass of each
    # (chunk, block) runs on the side stream beside the next one's logit GEMM,
    # alternating two blocks, across chunk boundaries.
    p = synth.make_problem("tiny", seed=57 + D, T=256, prompts=1, G=4, D=D, V=3000,
                           lengths=(60, 256))
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=256, vocab_block=1024, flags=SINGLE_PASS)
    plan = clp.grpo_get_plan(p.n_tokens, D, p.vocab, p.seq_len, params)
    assert plan["n_chunks"] == 4 and plan["n_vocab_blocks"] == 3
    assert plan["g_in_dh_gemm"] == (1 if D <= 2048 else 0)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"single pass D={D} 4x3 steps")


def test_single_pass_both_placements_above_2048(clp):
    # Above D = 2048 the planner places the single pass's P conversion on chip
    # (one logit block) or in a pass of its own (two blocks), whichever is
    # modelled faster within the budget: a range of budgets reaches both, and
    # each gives the oracle's results.
    p = synth.make_problem("tiny", seed=58, T=512, prompts=1, G=4, D=2304, V=6000,
                           lengths=(100, 512))
    old, ref, want = oracle_case(p)
    full = clp.grpo_workspace_size(p.n_tokens, p.hidden_size, p.vocab, p.seq_len,
                                   clp.make_params(flags=SINGLE_PASS, vocab_block=2048))
    seen = {}
    for frac in (0, 1.0, 0.8, 0.6, 0.5, 0.4, 0.3):
        params = clp.make_params(flags=SINGLE_PASS, vocab_block=2048,
                                 workspace_limit_bytes=int(full * frac))
        plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
        assert plan["single_pass"] == 1
        seen.setdefault(plan["g_in_dh_gemm"], params)
    assert set(seen) == {0, 1}, seen
    for on_chip, params in seen.items():
        check(gpu_loss(clp, p, old, ref, params), want, p.mask,
              f"single pass D=2304, P {'on chip' if on_chip else 'in its own pass'}")


def test_three_backward_forms_agree(clp):
    # Same inputs through the three forms: same forward values up to fp32
    # summation order, dH within bf16 rounding of G (or P) of each other.
    p = synth.make_problem("tiny", seed=53, T=500, prompts=1, G=4, D=320, V=5000,
                           lengths=(100, 500))
    old, ref, want = oracle_case(p)
    runs = {f: gpu_loss(clp, p, old, ref, clp.make_params(chunk_tokens=512, vocab_block=1280,
                                                          flags=f))
            for f in (STORED, SINGLE_PASS, RECOMPUTE)}
    for f, got in runs.items():
        check(got, want, p.mask, f"form {f}")
    L0, lp0, dH0, _ = runs[RECOMPUTE]
    for f in (STORED, SINGLE_PASS):
        L1, lp1, dH1, _ = runs[f]
        assert np.abs(lp1 - lp0).max() <= 1e-5 and abs(L1 - L0) <= 1e-5 * abs(L0)
        assert np.linalg.norm(dH1 - dH0) <= 1e-2 * np.linalg.norm(dH0)


def test_single_pass_bad_id_and_all_masked(clp):
    p = synth.make_problem("tiny", seed=17)
    params = clp.make_params(flags=SINGLE_PASS, vocab_block=1024)
    ids = p.ids.clone()
    ids[9] = p.vocab + 5
    old = torch.full((p.n_tokens,), -8.0)
    L, logp, dH, st = gpu_loss(clp, p, old, old, params, ids=ids)
    assert st == -8 and math.isnan(logp[9]) and math.isnan(L)
    L, logp, dH, st = gpu_loss(clp, p, old, old, params, mask=torch.zeros_like(p.mask))
    assert st == 0 and L == 0.0 and np.all(logp == 0) and np.all(dH == 0)


def test_stored_and_recomputed_backward_agree(clp):
    p = synth.make_problem("tiny", seed=12, T=128, prompts=2, G=4, D=256, V=5000,
                           lengths=(30, 128))
    old, ref, _ = oracle_case(p)
    L1, lp1, dH1, s1 = gpu_loss(clp, p, old, ref, clp.make_params(flags=RECOMPUTE))
    L2, lp2, dH2, s2 = gpu_loss(clp, p, old, ref, clp.make_params(flags=STORED))
    assert s1 == 0 and s2 == 0
    assert np.abs(lp1 - lp2).max() <= 1e-5
    assert abs(L1 - L2) <= 1e-5 * abs(L1)
    assert np.linalg.norm(dH1 - dH2) <= 1e-2 * np.linalg.norm(dH1)


@pytest.mark.parametrize("chunk", [0, 128])
def test_g_in_dh_gemm_matches_separate_pass(clp, chunk):
    # D <= 2048: without dW the dH GEMM turns the stored logits into G itself;
    # asking for dW makes the same call form G in a pass of its own (both GEMMs
    # read it). Same inputs, same row values: logp and loss bit-identical, dH
    # equal up to the rounding of the target column's G value.
    p = synth.make_problem("tiny", seed=17, prompts=2, G=4, T=96, D=512, V=3001,
                           lengths=(10, 96))
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, flags=STORED)
    plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params)
    assert plan["g_in_dh_gemm"] == 1
    args = [_to(x) for x in (p.hidden, p.weight, p.ids, p.mask, old, ref, p.adv)]
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    L1, lp1, dH1 = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws)
    st = clp.grpo_read_device_status(ws)
    L2, lp2, dH2, dW = clp.grpo_loss_fwd_bwd(*args, p.seq_len, params=params, workspace=ws,
                                             want_dW=True)
    assert st == 0 and clp.grpo_read_device_status(ws) == 0
    assert torch.equal(L1, L2) and torch.equal(lp1, lp2)
    d1, d2 = dH1.double().cpu().numpy(), dH2.double().cpu().numpy()
    assert np.linalg.norm(d1 - d2) <= 1e-2 * np.linalg.norm(d1)
    m = p.mask.numpy().astype(bool)
    assert np.all(d1[~m] == 0) and np.all(d2[~m] == 0)
    check((L1.item(), lp1.cpu().double().numpy(), d1, st), want, p.mask,
          f"fused G chunk={chunk}")


@pytest.mark.parametrize("flags", [STORED, SINGLE_PASS])
@pytest.mark.parametrize("n", [2048, 4096, 8192])
def test_device_plan_fits_host_sized_workspace(clp, n, flags):
    # grpo_workspace_size plans without a device; the call plans with the SM
    # count (and may split a batch that fits one logit block into
    # double-buffered chunks). The host-sized workspace must always suffice,
    # and both backward variants must agree.
    D, V = 2304, 3000
    p = synth.make_problem("tiny", seed=n, prompts=n // 1024, G=4, T=256, D=D, V=V,
                           lengths=(128, 256))
    base, _ = oracle.selective_logp(p.hidden[:4], p.weight, p.ids.numpy()[:4])
    old = torch.full((n,), float(base.mean()))
    params = clp.make_params(flags=flags)
    plan = clp.grpo_get_plan(n, D, V, p.seq_len, params)
    assert plan["workspace_bytes"] <= clp.grpo_workspace_size(n, D, V, p.seq_len, params)
    L1, lp1, dH1, s1 = gpu_loss(clp, p, old, old, params)
    L2, lp2, dH2, s2 = gpu_loss(clp, p, old, old, clp.make_params(flags=RECOMPUTE))
    assert s1 == 0 and s2 == 0
    assert np.abs(lp1 - lp2).max() <= 1e-5 and abs(L1 - L2) <= 1e-5 * abs(L2)
    assert np.linalg.norm(dH1 - dH2) <= 1e-2 * np.linalg.norm(dH2)


def test_stored_logits_bad_id_and_all_masked(clp):
    p = synth.make_problem("tiny", seed=13)
    params = clp.make_params(flags=STORED)
    ids = p.ids.clone()
    ids[9] = -3
    old = torch.full((p.n_tokens,), -8.0)
    L, logp, dH, st = gpu_loss(clp, p, old, old, params, ids=ids)
    assert st == -8 and math.isnan(logp[9]) and math.isnan(L)
    L, logp, dH, st = gpu_loss(clp, p, old, old, params, mask=torch.zeros_like(p.mask))
    assert st == 0 and L == 0.0 and np.all(logp == 0) and np.all(dH == 0)


# -------------------------------------- single-CTA GEMMs (flag) vs pairs ---

SINGLE = 2  # GRPO_FLAG_SINGLE_CTA


@pytest.mark.parametrize("flags", [SINGLE | RECOMPUTE, SINGLE | STORED, SINGLE | SINGLE_PASS])
@pytest.mark.parametrize("N,T,D,V,chunk,vblock,padded", RAGGED[:4])
def test_single_cta_gemms(clp, flags, N, T, D, V, chunk, vblock, padded):
    G = 4 if (N // T) % 4 == 0 else 1
    p = synth.make_problem("tiny", seed=N + D + V + 2, prompts=(N // T) // G, G=G, T=T, D=D,
                           V=V, lengths=(max(1, T // 3), T) if padded else None)
    old, ref, want = oracle_case(p)
    params = clp.make_params(chunk_tokens=chunk, vocab_block=vblock, flags=flags)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"single {flags} {N}x{D}x{V}")


def test_pair_and_single_cta_agree(clp):
    # Odd number of 128-row blocks: the last CTA pair has one real row block.
    p = synth.make_problem("tiny", seed=14, T=640, prompts=1, G=1, D=256, V=3000)
    old, ref, _ = oracle_case(p)
    for extra in (RECOMPUTE, STORED, SINGLE_PASS):
        L1, lp1, dH1, s1 = gpu_loss(clp, p, old, ref, clp.make_params(flags=extra))
        L2, lp2, dH2, s2 = gpu_loss(clp, p, old, ref, clp.make_params(flags=extra | SINGLE))
        assert s1 == 0 and s2 == 0
        assert np.abs(lp1 - lp2).max() <= 1e-5 and abs(L1 - L2) <= 1e-5 * abs(L1)
        assert np.linalg.norm(dH1 - dH2) <= 1e-2 * np.linalg.norm(dH1)


# ------------------------------------- aggregation and workspace budgets ---

SEQMEAN = 4  # GRPO_FLAG_SEQUENCE_MEAN
FITFREE = 8  # GRPO_FLAG_FIT_FREE_MEMORY


@pytest.mark.parametrize("flags", [SEQMEAN | RECOMPUTE, SEQMEAN | STORED,
                                   SEQMEAN | SINGLE | RECOMPUTE, SEQMEAN,
                                   SEQMEAN | SINGLE_PASS])
def test_sequence_mean_aggregation(clp, flags):
    p = synth.make_problem("tiny", seed=60, T=100, prompts=2, G=4, D=256, V=3000,
                           lengths=(5, 100))
    p.mask[300:400] = 0  # completion 3 has no token at all
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
    old, ref = p.old_ref(torch.from_numpy(base))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta,
                               aggregation="sequence")
    check(gpu_loss(clp, p, old, ref, clp.make_params(flags=flags)), want, p.mask,
          f"sequence mean {flags}")


@pytest.mark.parametrize("flags,limit", [(FITFREE, 0), (STORED | FITFREE, 0),
                                         (STORED, 24 << 20), (RECOMPUTE, 24 << 20),
                                         (RECOMPUTE | FITFREE, 0), (0, 24 << 20),
                                         (SINGLE_PASS, 24 << 20), (SINGLE_PASS | FITFREE, 0)])
def test_workspace_budget_plans_give_same_results(clp, flags, limit):
    p = synth.make_problem("tiny", seed=61, T=512, prompts=2, G=4, D=512, V=6000,
                           lengths=(100, 512))
    old, ref, want = oracle_case(p)
    params = clp.make_params(flags=flags, workspace_limit_bytes=limit)
    if limit:
        assert clp.grpo_workspace_size(p.n_tokens, p.hidden_size, p.vocab, p.seq_len,
                                       params) <= limit
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"budget {flags} {limit}")


# ----------------------------------------------------- lm_head gradient dW --

DW_CASES = [
    # N, T, D, V, chunk, vblock, padded, flags
    (256, 64, 256, 4096, 0, 0, False, RECOMPUTE),
    (256, 64, 256, 4096, 0, 0, False, STORED),
    (300, 75, 200, 1000, 128, 512, True, RECOMPUTE),
    (300, 75, 200, 1000, 128, 512, True, STORED),
    (300, 75, 200, 1000, 128, 512, True, SINGLE | RECOMPUTE),
    (300, 75, 200, 1000, 128, 512, True, SINGLE | STORED),
    (4096, 512, 256, 3000, 256, 1024, True, STORED),   # many skipped blocks, empty chunks
    (4096, 512, 256, 3000, 256, 1024, True, RECOMPUTE),
    # dW with the single pass: the call recomputes the logit tiles instead.
    (300, 75, 200, 1000, 128, 512, True, SINGLE_PASS),
]


@pytest.mark.parametrize("N,T,D,V,chunk,vblock,padded,flags", DW_CASES)
def test_lm_head_gradient(clp, N, T, D, V, chunk, vblock, padded, flags):
    G = 4 if (N // T) % 4 == 0 else 1
    p = synth.make_problem("tiny", seed=N + V + flags, prompts=(N // T) // G, G=G, T=T, D=D,
                           V=V, lengths=(1 if N >= 4096 else T // 3, T) if padded else None)
    old, ref, want = oracle_case(p)
    want_dW = oracle.grad_weight(p.hidden, p.weight, p.ids.numpy(), want["g"])
    params = clp.make_params(chunk_tokens=chunk, vocab_block=vblock, flags=flags)
    ws = clp.alloc_workspace(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, params, DEV)
    dW = torch.full((V, D), float("nan"), device=DEV)
    loss, logp, dH, dW = clp.grpo_loss_fwd_bwd(
        _to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old), _to(ref), _to(p.adv),
        p.seq_len, params=params, workspace=ws, dW=dW)
    st = clp.grpo_read_device_status(ws)
    check((loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st), want,
          p.mask, f"dW case {N}x{D}x{V} flags={flags}")
    got = dW.cpu().double().numpy()
    rel = np.linalg.norm(got - want_dW) / np.linalg.norm(want_dW)
    print(f"   dW rel={rel:.3e}")
    assert np.all(np.isfinite(got)) and rel <= DH_RTOL


def test_lm_head_gradient_all_masked_is_zero(clp):
    p = synth.make_problem("tiny", seed=62)
    dW = torch.full((p.vocab, p.hidden_size), float("nan"), device=DEV)
    for flags in (RECOMPUTE, STORED):
        _, _, _, dW = clp.grpo_loss_fwd_bwd(
            _to(p.hidden), _to(p.weight), _to(p.ids), _to(torch.zeros_like(p.mask)),
            _to(torch.zeros(p.n_tokens)), _to(torch.zeros(p.n_tokens)), _to(p.adv), p.seq_len,
            params=clp.make_params(flags=flags), dW=dW)
        assert torch.all(dW == 0)


def test_lm_head_gradient_with_transform(clp):
    p = synth.make_problem("tiny", seed=63, T=75, prompts=1, G=4, D=200, V=3000,
                           lengths=(20, 75), weight_std=0.2)
    xf = oracle.Transform(softcap=2.0, temperature=0.8)
    base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy(), xf=xf)
    old, ref = p.old_ref(torch.from_numpy(base))
    want = oracle.loss_fwd_bwd(p.hidden, p.weight, p.ids.numpy(), p.mask.numpy(), old, ref,
                               p.adv, p.seq_len, p.eps_low, p.eps_high, p.beta, xf=xf)
    want_dW = oracle.grad_weight(p.hidden, p.weight, p.ids.numpy(), want["g"], xf=xf)
    for flags in (RECOMPUTE, STORED):
        params = clp.make_params(chunk_tokens=128, flags=flags, logit_softcapping=2.0,
                                 temperature=0.8)
        _, _, _, dW = clp.grpo_loss_fwd_bwd(
            _to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old), _to(ref),
            _to(p.adv), p.seq_len, params=params, want_dW=True)
        rel = np.linalg.norm(dW.cpu().double().numpy() - want_dW) / np.linalg.norm(want_dW)
        assert rel <= DH_RTOL, (flags, rel)


def _side_stream_params(clp, flags, n, D, V, T):
    """Params under which a call of this shape runs its G (stored form) or P
    (single pass) pass on the side stream, in more than one step."""
    for chunk, vb in ((512, 1024), (256, 1024), (512, 0), (1024, 1024)):
        params = clp.make_params(chunk_tokens=chunk, vocab_block=vb, flags=flags)
        plan = clp.grpo_get_plan(n, D, V, T, params)
        steps = plan["n_chunks"] * (plan["n_vocab_blocks"] if flags == SINGLE_PASS else 1)
        if plan["g_in_dh_gemm"] == 0 and steps > 1:
            return params
    raise AssertionError("no plan with a side-stream pass")


@pytest.mark.parametrize("flags", [STORED, SINGLE_PASS])
def test_concurrent_calls_from_two_threads(clp, flags):
    # Separate workspaces and streams, several chunks (and vocabulary blocks)
    # with G or P formed in a pass of their own (D > 2048), so the shared side
    # stream is used: results equal the same calls made serially.
    import threading

    D = 2304
    probs = [synth.make_problem("tiny", seed=90 + i, prompts=2, G=4, T=256, D=D, V=3000,
                                lengths=(64, 256)) for i in range(2)]
    params = _side_stream_params(clp, flags, probs[0].n_tokens, D, 3000, probs[0].seq_len)

    def args_of(p):
        base, _ = oracle.selective_logp(p.hidden, p.weight, p.ids.numpy())
        old, ref = p.old_ref(torch.from_numpy(base))
        return [_to(x) for x in (p.hidden, p.weight, p.ids, p.mask, old, ref, p.adv)]

    inputs = [args_of(p) for p in probs]
    serial = []
    for p, a in zip(probs, inputs):
        loss, logp, dH = clp.grpo_loss_fwd_bwd(*a, p.seq_len, params=params)
        torch.cuda.synchronize()
        serial.append((loss.clone(), logp.clone(), dH.clone()))

    out = [None, None]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ws = clp.alloc_workspace(probs[i].n_tokens, D, 3000, probs[i].seq_len, params,
                                         DEV)
                for _ in range(3):
                    r = clp.grpo_loss_fwd_bwd(*inputs[i], probs[i].seq_len, params=params,
                                              workspace=ws)
                s.synchronize()
                out[i] = r
        except Exception as e:  # surfaced below
            errors.append(e)

    th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors
    for (l0, lp0, d0), (l1, lp1, d1) in zip(serial, out):
        assert torch.equal(l0, l1) and torch.equal(lp0, lp1) and torch.equal(d0, d1)


@pytest.mark.parametrize("flags", [RECOMPUTE, STORED, SINGLE_PASS])
def test_device_memory_is_the_workspace_only(clp, flags):
    # The memory claim ("GRPO with 7x longer context", section "Flattened
    # sequence length chunking", Eq. 1-3): at a fixed chunk the memory a call
    # needs grows with N only by a few words per row, never with N x V. Checked
    # on the device: with inputs, outputs and workspace allocated beforehand,
    # a call changes the free device memory by nothing (the library allocates
    # nothing), and the workspace over an N sweep grows by O(N) only.
    D, V, T, chunk = 1024, 32000, 1024, 2048
    dev = torch.device(DEV)
    params = clp.make_params(chunk_tokens=chunk, flags=flags)
    sizes = {}
    for n in (4096, 16384, 65536):
        g = torch.Generator(device="cpu").manual_seed(n)
        hidden = torch.randn(n, D, generator=g).to(torch.bfloat16).to(dev)
        W = (0.02 * torch.randn(V, D, generator=g)).to(torch.bfloat16).to(dev)
        ids = torch.randint(0, V, (n,), generator=g, dtype=torch.int32).to(dev)
        mask = torch.ones(n, dtype=torch.uint8, device=dev)
        old = torch.full((n,), -10.0, device=dev)
        adv = torch.randn(n // T, generator=g).to(dev)
        ws = clp.alloc_workspace(n, D, V, T, params, dev)
        loss = torch.empty(1, device=dev)
        logp = torch.empty(n, device=dev)
        dH = torch.empty(n, D, dtype=torch.bfloat16, device=dev)
        clp.grpo_loss_fwd_bwd(hidden, W, ids, mask, old, old, adv, T, params=params,
                              workspace=ws, loss=loss, logp=logp, dH=dH)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info(dev)
        for _ in range(2):
            clp.grpo_loss_fwd_bwd(hidden, W, ids, mask, old, old, adv, T, params=params,
                                  workspace=ws, loss=loss, logp=logp, dH=dH)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info(dev)
        assert free1 == free0, (n, free0 - free1)
        assert clp.grpo_read_device_status(ws) == 0 and math.isfinite(loss.item())
        sizes[n] = ws.numel()
        print(f"flags={flags} N={n}: workspace {ws.numel() / 2**20:.1f} MiB, "
              f"fp32 N x V logits would be {n * V * 4 / 2**20:.0f} MiB")
        del hidden, W, ids, mask, old, adv, ws, loss, logp, dH
    per_row = (sizes[65536] - sizes[4096]) / (65536 - 4096)
    assert per_row < 1024  # a few fp32 / fp64 words and the split partials per row
    assert sizes[65536] < 65536 * V * 4 / 20


# Vocabulary edges through every backward form: V = 1 (logp = 0, G = 0),
# V = 7 (a stored row narrower than one 16-byte chunk), V = 65 (one column
# past a 64-wide K slice); D = 256 forms G in the dH GEMM, D = 2304 in its own
# pass; RECOMPUTE is the recomputed backward.
@pytest.mark.parametrize("flags", [RECOMPUTE, STORED, SINGLE_PASS])
@pytest.mark.parametrize("D", [256, 2304])
@pytest.mark.parametrize("V", [1, 7, 65])
def test_small_vocab_edges(clp, flags, D, V):
    p = synth.make_problem("tiny", seed=V * 7 + D, prompts=1, G=4, T=32, D=D, V=V,
                           lengths=(5, 32), weight_std=0.3)
    old, ref, want = oracle_case(p)
    params = clp.make_params(flags=flags)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"V={V} D={D} flags={flags}")


@pytest.mark.parametrize("flags", [STORED, STORED | SINGLE])
def test_empty_batch_stored(clp, flags):
    h = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(100, 64, device=DEV).to(torch.bfloat16)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    f = torch.empty(0, dtype=torch.float32, device=DEV)
    loss, logp, dH = clp.grpo_loss_fwd_bwd(h, W, e, torch.empty(0, dtype=torch.uint8, device=DEV),
                                           f, f, torch.empty(0, dtype=torch.float32, device=DEV),
                                           1, params=clp.make_params(flags=flags))
    assert loss.item() == 0.0 and dH.numel() == 0


# Smallest legal shapes: hidden sizes far below one 64-wide K slice (D = 8,
# 24), a single token, and D = 2056 (just past the size up to which G is
# formed in the dH GEMM, and not a multiple of 64); every backward form.
@pytest.mark.parametrize("flags", [RECOMPUTE, STORED, STORED | SINGLE, SINGLE_PASS,
                                   SINGLE_PASS | SINGLE])
@pytest.mark.parametrize("N,D", [(1, 8), (3, 24), (130, 8), (70, 2056)])
def test_tiny_hidden_and_single_token(clp, flags, N, D):
    p = synth.make_problem("tiny", seed=N * 31 + D, prompts=1, G=1, T=N, D=D, V=300,
                           weight_std=0.5 if D < 64 else 0.05)
    old, ref, want = oracle_case(p)
    params = clp.make_params(flags=flags)
    check(gpu_loss(clp, p, old, ref, params), want, p.mask, f"N={N} D={D} flags={flags}")
    lp, _ = clp.grpo_logp_fwd(_to(p.hidden), _to(p.weight), _to(p.ids), params=params)
    assert np.abs(lp.cpu().double().numpy() - want["logp"]).max() <= LOGP_TOL


def _guarded(n, dtype, fill, guard):
    # A tensor of n elements inside a buffer of guard elements on each side,
    # everything set to `fill` (so writes outside the view can be detected).
    buf = torch.full((n + 2 * guard,), fill, dtype=dtype, device=DEV)
    return buf, buf[guard:guard + n]


# No write outside the output buffers and no read of uninitialised workspace:
# every output is a view inside a buffer of sentinels, and the workspace is
# prefilled with 0xFF bytes (NaN in every float format) inside its own guard
# band. Results must still match the oracle and every sentinel must survive.
@pytest.mark.parametrize("flags", [RECOMPUTE, STORED, STORED | SINGLE, SINGLE_PASS,
                                   SINGLE_PASS | SINGLE])
@pytest.mark.parametrize("D", [256, 2304])
@pytest.mark.parametrize("with_dw", [False, True])
def test_guard_bands_and_poisoned_workspace(clp, flags, D, with_dw):
    p = synth.make_problem("tiny", seed=D + flags, prompts=1, G=4, T=75, D=D, V=1000,
                           lengths=(20, 75))
    old, ref, want = oracle_case(p)
    N, V = p.n_tokens, p.vocab
    params = clp.make_params(chunk_tokens=128, flags=flags)
    g = 4096
    lb, loss = _guarded(1, torch.float32, 7.0, g)
    pb, logp = _guarded(N, torch.float32, 7.0, g)
    hb, dH = _guarded(N * D, torch.bfloat16, 7.0, g)
    dH = dH.view(N, D)
    wb, dW = _guarded(V * D, torch.float32, 7.0, g) if with_dw else (None, None)
    if dW is not None:
        dW = dW.view(V, D)
    size = clp.grpo_workspace_size(N, D, V, p.seq_len, params)
    wsb = torch.full((size + 2 * g,), 0xFF, dtype=torch.uint8, device=DEV)
    ws = wsb[g:g + size]
    out = clp.grpo_loss_fwd_bwd(_to(p.hidden), _to(p.weight), _to(p.ids), _to(p.mask), _to(old),
                                _to(ref), _to(p.adv), p.seq_len, params=params, workspace=ws,
                                loss=loss, logp=logp, dH=dH, dW=dW)
    st = clp.grpo_read_device_status(ws)
    check((loss.item(), logp.cpu().double().numpy(), dH.cpu().double().numpy(), st), want,
          p.mask, f"guarded D={D} flags={flags} dW={with_dw}")
    for name, buf, n in (("loss", lb, 1), ("logp", pb, N), ("dH", hb, N * D)) + (
            (("dW", wb, V * D),) if with_dw else ()):
        assert torch.all(buf[:g] == 7.0) and torch.all(buf[g + n:] == 7.0), name
    assert torch.all(wsb[:g] == 0xFF) and torch.all(wsb[g + size:] == 0xFF)
    if with_dw:
        want_dW = oracle.grad_weight(p.hidden, p.weight, p.ids.numpy(), want["g"])
        got = out[3].cpu().double().numpy()
        assert np.linalg.norm(got - want_dW) <= DH_RTOL * np.linalg.norm(want_dW)


# --------------------------------------------- automatic backward form -----

def test_automatic_backward_form_is_the_forced_one(clp):
    # Flags 0: without a budget the call takes the stored form; under a budget
    # too small for one stored chunk of 256 rows (32000 fp16 logits each) it
    # takes the recomputed one, with vocab blocks of 4096. Either way its
    # results are bitwise those of the form forced by its flag.
    p = synth.make_problem("tiny", seed=71, T=1024, prompts=2, G=4, D=1024, V=32000,
                           lengths=(256, 1024))
    old, ref, want = oracle_case(p)
    for limit, form in ((0, STORED), (12 << 20, RECOMPUTE)):
        auto = clp.make_params(workspace_limit_bytes=limit, vocab_block=4096)
        plan = clp.grpo_get_plan(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, auto)
        assert plan["stored_logits"] == (1 if form == STORED else 0), (limit, plan)
        forced = clp.make_params(flags=form, workspace_limit_bytes=limit, vocab_block=4096)
        assert clp.grpo_workspace_size(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, auto) == \
            clp.grpo_workspace_size(p.n_tokens, p.hidden_size, p.vocab, p.seq_len, forced)
        got = gpu_loss(clp, p, old, ref, auto)
        check(got, want, p.mask, f"automatic, budget {limit}")
        ref_run = gpu_loss(clp, p, old, ref, forced)
        assert got[0] == ref_run[0] and np.array_equal(got[1], ref_run[1])
        assert np.array_equal(got[2], ref_run[2])
