"""fp64 CPU oracle for the chunked selective log-softmax and the GRPO token loss.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only
the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it. It shares no code with the CUDA library and imports
nothing from the package.

What it computes, and where each step comes from (the pages are cited by
title and section):

* "GRPO with 7x longer context" (Unsloth docs), section "Flattened sequence
  length chunking", the ``chunked_hidden_states_selective_log_softmax`` call
  and its notes: the log-probability of the sampled completion token is taken
  straight from the final hidden states and the lm_head weight, with the
  logits upcast to float32 "to keep accuracy". The oracle goes further and
  works in float64 throughout:  logp_t = h_t . W[y_t] - logsumexp_v(h_t . W_v).
  Chunking never changes that value, so the oracle does not chunk: it
  materialises whole logit rows (a loop over blocks of rows only bounds the
  memory a row block needs; each row is computed on its own).
* Same page, section "Offloading activations for log-softmax": the backward
  pass re-runs the forward under autograd and back-propagates the incoming
  gradient. Here the gradient of logp_t with respect to h_t is written out:
  d logp_t / d h_t = W[y_t] - sum_v softmax_v W_v.
* "Unsloth internals" (ai.trevor-barnes.com), section "The relationship to
  TRL": GRPO forms a clipped surrogate objective with a KL-to-reference term
  over group-relative advantages.
* "Train reasoning models with 5GB VRAM" (digialps.com), section "Under the
  Hood": the KL is the reverse KL, and the per-token objective is
  exp(q - q.detach()) * advantages.unsqueeze(1): a ratio equal to one in value
  whose gradient is the advantage, broadcast over the tokens of a sequence.
* "How does Unsloth implement GRPO" (instagit.com), section "Corrected
  hyperparameters": beta = 0.001.

Readings taken where the pages are silent (each one is listed in the design
notes of the repository):

* ratio r_t = exp(logp_t - old_t); surrogate = min(r A, clamp(r, 1-eps_low,
  1+eps_high) A); at r exactly on a clip bound the unclipped branch is taken.
* KL is the k3 estimator of the reverse KL to the reference policy:
  kl_t = exp(ref_t - logp_t) - (ref_t - logp_t) - 1.
* token loss l_t = -surrogate_t + beta kl_t; the batch loss is the masked
  token mean  L = sum_t m_t l_t / M  with  M = sum_t m_t  (or a caller-given
  denominator when it is > 0); M = 0 gives L = 0 and a zero gradient.
* sequence b of token t is t // T (completions of length T laid end to end);
  the advantage of the sequence is broadcast over its tokens.
* masked rows get logp = 0 and a zero gradient row.
* per-sequence aggregation (optional, a reading of the GRPO objective's
  per-completion normalisation; the pages name no aggregation at all):
  L = (1/B') sum_b (1/len_b) sum_{t in b} m_t l_t with len_b = sum_{t in b} m_t
  and B' the number of completions with len_b > 0 (or a caller-given
  denominator > 0 in place of B').
* logit transforms ("GRPO with 7x longer context", notes under the
  chunked_hidden_states_selective_log_softmax call: softcapping, temperature
  and the logit scale multiply/divide): applied to the raw logit z in the
  order the call lists them, z' = f(z) = s(z * mult / div) / temperature with
  s(x) = cap * tanh(x / cap) when a softcap is set, else s(x) = x. logp is the
  log-softmax of z'; the chain rule adds f'(z_v) to every vocab term of dH.
"""

from __future__ import annotations

import numpy as np

# Rows per block when whole logit rows are materialised; bounds the float64
# temporary to ROW_BLOCK * V * 8 bytes.
ROW_BLOCK = 64


class Transform:
    """Logit transform z' = s(z * mult / div) / temperature (identity by default)."""

    def __init__(self, scale_mul=1.0, scale_div=1.0, softcap=0.0, temperature=1.0):
        self.scale_mul = float(scale_mul)
        self.scale_div = float(scale_div)
        self.softcap = float(softcap)
        self.temperature = float(temperature)

    @property
    def identity(self):
        return (self.scale_mul == 1.0 and self.scale_div == 1.0 and self.softcap == 0.0
                and self.temperature == 1.0)

    def apply(self, z):
        """Returns (z', dz'/dz), both float64 arrays shaped like z."""
        x = z * self.scale_mul / self.scale_div
        dx = self.scale_mul / self.scale_div
        if self.softcap > 0.0:
            u = np.tanh(x / self.softcap)
            x = self.softcap * u
            d = dx * (1.0 - u * u)
        else:
            d = np.full_like(z, dx)
        return x / self.temperature, d / self.temperature


IDENTITY = Transform()


def _f64(x) -> np.ndarray:
    """Widen a numpy array or a CPU torch tensor (bf16 included) to float64."""
    if hasattr(x, "detach"):  # torch tensor: widen on the torch side first
        import torch  # local import: the oracle itself does not need torch

        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def logits_rows(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Full logit rows z_{t,v} = sum_d h_{t,d} W_{v,d} (float64 matmul)."""
    return h @ W.T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse_t = mx_t + log sum_v exp(z_{t,v} - mx_t), mx_t = max_v z_{t,v}."""
    mx = z.max(axis=1)
    return mx + np.log(np.exp(z - mx[:, None]).sum(axis=1))


def selective_logp(hidden, W, ids, row_block: int = ROW_BLOCK, xf: Transform = IDENTITY):
    """Selective log-softmax of the sampled tokens, from hidden states.

    ("GRPO with 7x longer context", section "Flattened sequence length
    chunking": chunked_hidden_states_selective_log_softmax.)

    hidden: [N, D]; W: [V, D] (lm_head weight, one row per vocabulary entry);
    ids: [N] integer token ids in [0, V).
    Returns (logp [N], lse [N]) in float64.
    """
    h = _f64(hidden)
    Wd = _f64(W)
    y = np.asarray(ids, dtype=np.int64)
    n = h.shape[0]
    logp = np.empty(n, dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        z = logits_rows(h[r0:r1], Wd)
        if not xf.identity:
            z = xf.apply(z)[0]
        l = logsumexp_rows(z)
        lse[r0:r1] = l
        logp[r0:r1] = z[np.arange(r1 - r0), y[r0:r1]] - l
    return logp, lse


def token_terms(logp, old, ref, adv_tok, eps_low, eps_high, beta):
    """Per-token GRPO loss l_t and its derivative dl_t/dlogp_t (float64).

    ("Unsloth internals", section "The relationship to TRL": clipped surrogate
    plus a KL-to-reference term; "Train reasoning models with 5GB VRAM",
    section "Under the Hood": reverse KL and the exp(q - q.detach()) * A
    identity.)
    """
    logp = _f64(logp)
    old = _f64(old)
    ref = _f64(ref)
    A = _f64(adv_tok)
    r = np.exp(logp - old)
    c = np.clip(r, 1.0 - eps_low, 1.0 + eps_high)
    surr = np.minimum(r * A, c * A)
    delta = ref - logp
    kl = np.exp(delta) - delta - 1.0
    loss_tok = -surr + beta * kl
    # d surr / d logp: the unclipped branch passes A r; a clipped branch that
    # min() selects strictly passes nothing.
    clipped = ((A > 0) & (r > 1.0 + eps_high)) | ((A < 0) & (r < 1.0 - eps_low))
    dsurr = np.where(clipped, 0.0, A * r)
    dloss_tok = -dsurr + beta * (1.0 - np.exp(delta))
    return loss_tok, dloss_tok, r, kl


def broadcast_advantage(adv_per_seq, n_tokens: int, seq_len: int) -> np.ndarray:
    """advantages.unsqueeze(1): token t takes the advantage of sequence t // T."""
    a = _f64(adv_per_seq)
    return a[np.arange(n_tokens) // seq_len]


def token_weights(mask, seq_len, aggregation="token", loss_denominator=0.0):
    """w_t with L = sum_t w_t l_t: m_t / M (token mean) or m_t / (len_b B')
    (mean over completions of the per-completion token mean)."""
    m = _f64(mask)
    n = m.shape[0]
    if aggregation == "token":
        M = float(loss_denominator) if loss_denominator > 0 else float(m.sum())
        return (m / M if M != 0.0 else np.zeros(n)), M
    lens = m.reshape(-1, seq_len).sum(axis=1)
    B = float(loss_denominator) if loss_denominator > 0 else float((lens > 0).sum())
    if B == 0.0:
        return np.zeros(n), B
    len_tok = np.repeat(lens, seq_len)
    w = np.where(m > 0, m / np.where(len_tok > 0, len_tok, 1.0) / B, 0.0)
    return w, B


def grpo_loss(logp, old, ref, adv_per_seq, mask, seq_len, eps_low=0.2,
              eps_high=0.2, beta=0.001, loss_denominator=0.0, aggregation="token"):
    """Masked GRPO loss L and g_t = dL/dlogp_t.

    aggregation "token": L = sum_t m_t l_t / M; "sequence": mean over
    completions of each completion's token mean. Returns (L, g [N],
    loss_tok [N], M) with M the token count (token) or completion count
    (sequence) used as denominator. Masked tokens have g_t = 0.
    """
    logp = _f64(logp)
    n = logp.shape[0]
    m = _f64(mask)
    A = broadcast_advantage(adv_per_seq, n, seq_len)
    if aggregation != "token":
        w, B = token_weights(mask, seq_len, aggregation, loss_denominator)
        lp = np.where(m > 0, logp, 0.0)
        od = np.where(m > 0, _f64(old), 0.0)
        rf = np.where(m > 0, _f64(ref), 0.0)
        loss_tok, dloss_tok, _, _ = token_terms(lp, od, rf, A, eps_low, eps_high, beta)
        L = float(np.sum(np.where(w > 0, w * loss_tok, 0.0)))
        return L, np.where(w > 0, w * dloss_tok, 0.0), np.where(m > 0, loss_tok, 0.0), B
    M = float(loss_denominator) if loss_denominator > 0 else float(m.sum())
    # Masked tokens contribute nothing; their logp (written as 0) never enters
    # the arithmetic, so their inputs may hold anything.
    lp = np.where(m > 0, logp, 0.0)
    od = np.where(m > 0, _f64(old), 0.0)
    rf = np.where(m > 0, _f64(ref), 0.0)
    loss_tok, dloss_tok, _, _ = token_terms(lp, od, rf, A, eps_low, eps_high, beta)
    if M == 0.0:
        return 0.0, np.zeros(n), np.where(m > 0, loss_tok, 0.0), M
    L = float(np.sum(np.where(m > 0, loss_tok, 0.0)) / M)
    g = np.where(m > 0, dloss_tok / M, 0.0)
    return L, g, loss_tok, M


def grad_hidden(hidden, W, ids, g, row_block: int = ROW_BLOCK, xf: Transform = IDENTITY):
    """dH_t = g_t * (W[y_t] - sum_v softmax(z_t)_v W_v), float64.

    ("GRPO with 7x longer context", section "Offloading activations for
    log-softmax": the backward re-runs the selective log-softmax and
    back-propagates g = dL/dlogp into the hidden states.) Rows with g_t = 0
    (masked rows) are exactly zero.
    """
    h = _f64(hidden)
    Wd = _f64(W)
    y = np.asarray(ids, dtype=np.int64)
    gd = _f64(g)
    n, d = h.shape
    dH = np.zeros((n, d), dtype=np.float64)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        rows = np.nonzero(gd[r0:r1] != 0.0)[0] + r0
        if rows.size == 0:
            continue
        z = logits_rows(h[rows], Wd)
        if xf.identity:
            p = np.exp(z - logsumexp_rows(z)[:, None])
            dH[rows] = gd[rows, None] * (Wd[y[rows]] - p @ Wd)
        else:
            # d logp_t / d z_v = (onehot_v(y_t) - softmax(z')_v) f'(z_v)
            zt, dz = xf.apply(z)
            jac = -np.exp(zt - logsumexp_rows(zt)[:, None])
            jac[np.arange(len(rows)), y[rows]] += 1.0
            dH[rows] = gd[rows, None] * ((jac * dz) @ Wd)
    return dH


def grad_weight(hidden, W, ids, g, row_block: int = ROW_BLOCK, xf: Transform = IDENTITY):
    """dW = dL/dW: dW_v = sum_t g_t (onehot_v(y_t) - softmax(z'_t)_v) f'(z_tv) h_t.

    The lm_head gradient (needed only when the head is trained; frozen under
    LoRA). Same Jacobian rows as grad_hidden, contracted with h instead of W.
    Returns float64 [V, D].
    """
    h = _f64(hidden)
    Wd = _f64(W)
    y = np.asarray(ids, dtype=np.int64)
    gd = _f64(g)
    dW = np.zeros_like(Wd)
    for r0 in range(0, h.shape[0], row_block):
        r1 = min(h.shape[0], r0 + row_block)
        rows = np.nonzero(gd[r0:r1] != 0.0)[0] + r0
        if rows.size == 0:
            continue
        z = logits_rows(h[rows], Wd)
        zt, dz = xf.apply(z) if not xf.identity else (z, np.ones_like(z))
        jac = -np.exp(zt - logsumexp_rows(zt)[:, None])
        jac[np.arange(len(rows)), y[rows]] += 1.0
        dW += ((gd[rows, None] * jac * dz).T) @ h[rows]
    return dW


def loss_fwd_bwd(hidden, W, ids, mask, old, ref, adv_per_seq, seq_len,
                 eps_low=0.2, eps_high=0.2, beta=0.001, loss_denominator=0.0,
                 xf: Transform = IDENTITY, aggregation="token"):
    """The whole path: logp, the loss, and the gradient to the hidden states.

    Returns a dict with L, logp (masked rows 0), lse, g, dH, M.
    """
    m = _f64(mask)
    logp, lse = selective_logp(hidden, W, ids, xf=xf)
    logp = np.where(m > 0, logp, 0.0)
    L, g, loss_tok, M = grpo_loss(logp, old, ref, adv_per_seq, mask, seq_len,
                                  eps_low, eps_high, beta, loss_denominator, aggregation)
    dH = grad_hidden(hidden, W, ids, g, xf=xf)
    return {"L": L, "logp": logp, "lse": lse, "g": g, "dH": dH, "M": M,
            "loss_tok": loss_tok}


def rows_fwd_bwd(hidden, W, ids, rows, old, ref, adv_per_seq, seq_len, M,
                 eps_low=0.2, eps_high=0.2, beta=0.001, xf: Transform = IDENTITY):
    """logp, g and dH for a chosen set of (unmasked) rows only.

    Given the loss denominator M, everything about a row depends on that row
    alone, so the values for sampled rows are exact, not estimates.
    """
    rows = np.asarray(rows, dtype=np.int64)
    h = _f64(hidden)[rows] if not hasattr(hidden, "detach") else _f64(hidden[rows])
    y = np.asarray(ids, dtype=np.int64)[rows]
    logp, lse = selective_logp(h, W, y, xf=xf)
    A = _f64(adv_per_seq)[rows // seq_len]
    _, dloss_tok, _, _ = token_terms(logp, _f64(old)[rows], _f64(ref)[rows], A,
                                     eps_low, eps_high, beta)
    g = dloss_tok / M
    dH = grad_hidden(h, W, y, g, xf=xf)
    return {"logp": logp, "lse": lse, "g": g, "dH": dH}
