"""The worked memory example of "GRPO with 7x longer context" (Unsloth docs),
section "Flattened sequence length chunking", Equations 1-3, and section
"Hidden states chunking" (fixture: tests/golden/grpo7x_memory_example.txt).

The page counts logit memory as elements / 1024^3 for the whole batch (Eq. 1),
for one sample at a time (Eq. 2), and for one sample's context split by the
multiplier max(4, context_length // 4096) (Eq. 3). Its printed logit values are
a constant 0.85 of what those formulas give, while its hidden-state values match
theirs; the reading taken here is the formulas' scaling, which the printed
values do follow. The library's chunked logit block is pinned to Eq. 3: at the
page's chunk it holds exactly Eq. 3's elements in fp16, per block, and does not
grow with the batch. Host-only calls; no GPU.
"""

import os

import pytest

import __graft_entry__

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "grpo7x_memory_example.txt")
GIB = 1024.0 ** 3
STORED = 1
RECOMPUTE = 16  # GRPO_FLAG_RECOMPUTE_LOGITS


@pytest.fixture(scope="module")
def ex():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (x.strip() for x in line.split("="))
                out[k] = float(v)
    return out


@pytest.fixture(scope="module")
def clp():
    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def multiplier(ex):
    return max(int(ex["multiplier_floor"]), int(ex["context_length"]) // int(ex["multiplier_divisor"]))


def test_hidden_state_example_matches_its_formula(ex):
    full = ex["hidden_batch_size"] * ex["hidden_context_length"] * ex["hidden_states_dim"] / GIB
    one = ex["hidden_context_length"] * ex["hidden_states_dim"] / GIB
    assert abs(full - ex["hidden_gb"]) < 0.05  # printed as "about 2"
    assert abs(one - ex["hidden_chunked_gb"]) < 0.0005
    assert abs(full / one - ex["hidden_batch_size"]) < 1e-12


def test_printed_logit_values_follow_the_equations_scaling(ex):
    b, T, V = ex["batch_size"], ex["context_length"], ex["vocab_dim"]
    m = multiplier(ex)
    assert m == 4  # max(4, 8192 // 4096)
    eq = [b * T * V / GIB, T * V / GIB, (T / m) * V / GIB]
    printed = [ex["eq1_logit_gb"], ex["eq2_logit_gb"], ex["eq3_logit_gb"]]
    # Eq. 1 -> 2 divides by the batch, Eq. 2 -> 3 by the multiplier; the printed
    # values (two or three digits) keep both ratios.
    assert abs(printed[0] / printed[1] - b) / b < 0.02
    assert abs(printed[1] / printed[2] - m) / m < 0.02
    # Against the formulas themselves they are off by one common factor (~0.85),
    # not by a different structure.
    factors = [p / e for p, e in zip(printed, eq)]
    assert max(factors) - min(factors) < 0.01
    assert 0.8 < factors[0] < 0.9


@pytest.mark.parametrize("hidden, blocks", [(4096, 2), (1536, 1)])
def test_stored_logit_block_is_eq3_elements_in_fp16(clp, ex, hidden, blocks):
    # The page's example as a call: b completions of T tokens, chunk = T / multiplier.
    b, T, V = int(ex["batch_size"]), int(ex["context_length"]), int(ex["vocab_dim"])
    rows = T // multiplier(ex)
    eq3_elements = rows * V

    def ws(n, chunk):
        return clp.grpo_workspace_size(n, hidden, V, T, clp.make_params(chunk_tokens=chunk,
                                                                        flags=STORED))
    # Halving the chunk frees exactly half of Eq. 3's elements at 2 bytes, plus
    # one fp32 maximum per 64 of them (1/32 more), per logit block (two blocks
    # when G is formed in a pass of its own, D > 2048), and the chunk's copy of
    # h (its rows x D in bf16: the row blocks that span a completion's end).
    half = eq3_elements // 2
    assert V % 64 == 0
    assert ws(b * T, rows) - ws(b * T, rows // 2) == (blocks * (2 * half + 4 * (half // 64)) +
                                                      (rows // 2) * hidden * 2)
    # Eq. 2's point: the block does not grow with the batch; only per-row
    # vectors do (a few hundred bytes per token).
    grow = ws(2 * b * T, rows) - ws(b * T, rows)
    assert 0 < grow < b * T * 400


def test_recompute_g_block_is_eq3_elements_in_bf16(clp, ex):
    b, T, V = int(ex["batch_size"]), int(ex["context_length"]), int(ex["vocab_dim"])
    rows = T // multiplier(ex)

    def ws(chunk):
        return clp.grpo_workspace_size(b * T, 4096, V, T,
                                       clp.make_params(chunk_tokens=chunk, vocab_block=V,
                                                       flags=RECOMPUTE))
    # Eq. 3's elements in bf16, and the chunk's copy of h (rows x D in bf16).
    assert ws(rows) - ws(rows // 2) == 2 * (rows // 2) * V + (rows // 2) * 4096 * 2
