"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and the host-only calls (workspace sizing, status strings,
argument checks that fail before any GPU work) behave. No compute call runs.
"""

import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clp():
    __graft_entry__.build()
    import chunked_log_prob_gb300 as m

    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "grpo_gb300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(grpo_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(clp):
    declared = _declared_functions()
    assert declared == sorted(clp.EXPORTED)
    lib = ctypes.CDLL(clp._binding.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_library_is_loaded_in_process(clp):
    maps = open("/proc/self/maps").read()
    assert "libgrpo_gb300.so" in maps


def test_status_strings(clp):
    for code in range(0, -10, -1):
        assert clp.status_string(code) != "unknown status"
    assert clp.status_string(-99) == "unknown status"


def test_default_params(clp):
    p = clp.make_params()
    assert abs(p.eps_low - 0.2) < 1e-7 and abs(p.eps_high - 0.2) < 1e-7
    assert abs(p.beta - 0.001) < 1e-9 and p.flags == 0


def test_workspace_independent_of_vocab_times_tokens(clp):
    # Recomputed backward: grows with N (a few fp32 per row) and with chunk x
    # vocab block, never N x V.
    p = clp.make_params(chunk_tokens=1024, vocab_block=8192, flags=16)
    sizes = [clp.grpo_workspace_size(n, 4096, 128256, 1, p) for n in (4096, 16384, 65536)]
    per_row = (sizes[2] - sizes[1]) / (65536 - 16384)
    assert per_row < 64 * 4 * 2 + 64  # split partials + a few fp32 per row
    # G block, fp32 dH accumulator, the chunk's copy of h (chunk x D in bf16)
    fixed = 1024 * 8192 * 2 + 1024 * 4096 * 4 + 1024 * 4096 * 2
    assert sizes[0] < fixed + 4096 * 300 + 65536
    assert sizes[2] < 65536 * 128256 * 4 / 100  # far below the N x V fp32 logits


def test_workspace_grows_with_chunk(clp):
    a = clp.grpo_workspace_size(16384, 4096, 128256, 1, clp.make_params(chunk_tokens=1024))
    b = clp.grpo_workspace_size(16384, 4096, 128256, 1, clp.make_params(chunk_tokens=4096))
    assert b > a


def test_single_vocab_block_needs_no_accumulator(clp):
    big = clp.grpo_workspace_size(1024, 4096, 4096, 1, clp.make_params(
        chunk_tokens=1024, vocab_block=4096, flags=16))
    small = clp.grpo_workspace_size(1024, 4096, 4096, 1, clp.make_params(
        chunk_tokens=1024, vocab_block=2048, flags=16))
    assert small - big > 1024 * 4096 * 4 - 1024 * 2048 * 2 - 4096


@pytest.mark.parametrize("n,d,v,want", [
    (100, 12, 50, -3),   # hidden % 8 != 0
    (-1, 16, 50, -1),    # negative N
    (10, 16, 0, -1),     # empty vocabulary
])
def test_workspace_size_rejects_bad_shapes(clp, n, d, v, want):
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_workspace_size(n, d, v)
    assert e.value.code == want


def test_bad_params_rejected(clp):
    p = clp.make_params()
    p.flags = 64  # not a defined flag bit
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_workspace_size(10, 16, 50, 1, p)
    assert e.value.code == -1
    for forms in (1 | 16, 1 | 32, 16 | 32, 1 | 16 | 32):  # two backward forms at once
        p.flags = forms
        with pytest.raises(clp.GrpoError) as e:
            clp.grpo_workspace_size(10, 16, 50, 1, p)
        assert e.value.code == -1


def test_automatic_backward_form_follows_the_budget(clp):
    # Flags 0 (the default) choose the backward form: the stored one when the
    # workspace budget leaves room for chunks that fill the SMs, the
    # recomputed one under a tight budget. The choice is made at a fixed SM
    # count, so the sizing here (no device) is the call's own.
    STORED, RECOMPUTE = 1, 16
    n, d, v, t = 16384, 4096, 128256, 4096

    def ws(flags, limit=0):
        return clp.grpo_workspace_size(n, d, v, t, clp.make_params(
            flags=flags, workspace_limit_bytes=limit))
    SINGLE_PASS = 32
    assert ws(0) == ws(STORED)
    assert ws(0, 8 << 30) == ws(STORED, 8 << 30)
    # Between about 0.3 and 1.5 GB the stored form's chunks are too small for
    # whole SM waves: the single pass, which holds one or two vocabulary blocks
    # of a larger chunk, is modelled faster.
    assert ws(0, 1 << 30) == ws(SINGLE_PASS, 1 << 30) <= 1 << 30
    # Below the stored form's smallest chunk (two logit blocks of 256 rows),
    # it does not fit at all.
    with pytest.raises(clp.GrpoError):
        ws(STORED, 128 << 20)
    assert ws(0, 128 << 20) <= 128 << 20


def test_automatic_form_at_the_qwen25_head_counts_the_tail_split(clp):
    # D <= 2048: the stored form's fused dH GEMM and the single pass with P on
    # chip both split the last round of their dH-type launches once a budget
    # leaves room for the split's slots (from 608 MiB). Measured at this shape
    # on GB300: 1 GB, stored 3.55-3.65 ms against the single pass's 4.36-4.38;
    # 0.5 GB (no split), the single pass 5.64-5.69 against 7.65-7.69.
    STORED, SINGLE_PASS = 1, 32
    n, d, v, t = 8192, 1536, 151936, 1024

    def ws(flags, limit=0):
        return clp.grpo_workspace_size(n, d, v, t, clp.make_params(
            flags=flags, workspace_limit_bytes=limit))
    assert ws(0) == ws(STORED)
    for limit in (1 << 30, 2 << 30):
        assert ws(0, limit) == ws(STORED, limit) <= limit
    for limit in (256 << 20, 512 << 20):
        assert ws(0, limit) == ws(SINGLE_PASS, limit) <= limit


def test_null_pointers_rejected_before_launch(clp):
    shape = clp.make_shape(10, 5, 16, 50)
    rc = clp.lib.grpo_loss_fwd_bwd(None, None, None, None, None, None, None, None, None, None,
                                   None, ctypes.byref(shape), None, None, 0, None)
    assert rc == -1
    rc = clp.lib.grpo_logp_fwd(None, None, None, None, None, ctypes.byref(shape), None, None, 0,
                               None)
    assert rc == -1


def test_sequence_length_must_divide_tokens(clp):
    shape = clp.make_shape(10, 3, 16, 50)
    buf = ctypes.create_string_buffer(4096)
    addr = (ctypes.addressof(buf) + 255) // 256 * 256
    rc = clp.lib.grpo_loss_fwd_bwd(addr, addr, addr, addr, addr, addr, addr, addr, None, addr,
                                   None, ctypes.byref(shape), None, addr, 1024, None)
    assert rc == -3


def test_misaligned_pointers_rejected(clp):
    shape = clp.make_shape(8, 8, 16, 50)
    buf = ctypes.create_string_buffer(8192)
    a = (ctypes.addressof(buf) + 255) // 256 * 256
    rc = clp.lib.grpo_logp_fwd(a + 8, a, a, a, None, ctypes.byref(shape), None, a, 4096, None)
    assert rc == -2
    rc = clp.lib.grpo_logp_fwd(a, a, a, a, None, ctypes.byref(shape), None, a + 16, 4096, None)
    assert rc == -2


def stored_block(chunk, V):
    """One stored-logit block: fp16 logits of chunk x V (V padded to 8) and the
    fp32 maximum of every 64-column box of each row."""
    return chunk * (-(-V // 8) * 8 * 2 + -(-V // 64) * 4)


# The stored form's tail-split partial slots (vocabularies of at least 128 K
# stages): two fp32 tiles of 256 rows x 512 hidden columns for each of the 76
# SM pairs the sizing assumes. Fixed: independent of N, the chunk and V.
TAIL_SPLIT_BYTES = 2 * 76 * 256 * 512 * 4


def H_COPY(chunk, hidden):  # noqa: N802
    """The chunk's copy of h (rows x D in bf16) for the row blocks whose active
    16-row segments are not consecutive rows."""
    return chunk * hidden * 2


def test_stored_logit_workspace_is_chunk_times_vocab(clp):
    # Stored-logit backward: two blocks of chunk x V (double-buffered when
    # there is more than one chunk), independent of N.
    p = clp.make_params(chunk_tokens=2048, flags=1)
    a = clp.grpo_workspace_size(16384, 4096, 128256, 1, p)
    b = clp.grpo_workspace_size(65536, 4096, 128256, 1, p)
    block = stored_block(2048, 128256) + TAIL_SPLIT_BYTES + H_COPY(2048, 4096)
    extra = TAIL_SPLIT_BYTES + H_COPY(2048, 4096)
    assert 2 * block - extra < a < 2 * block - extra + 16384 * 400
    one = clp.grpo_workspace_size(2048, 4096, 128256, 1, p)  # a single chunk: one block
    assert block < one < block + 2048 * 400
    assert (b - a) / (65536 - 16384) < 64 * 4 * 2 + 64
    # Automatic chunk without a device: bounded by 2 GiB of fp16 logits per
    # block (plus their box maxima, 1/32 of that).
    auto = clp.grpo_workspace_size(131072, 2880, 201088, 1, clp.make_params(flags=1))
    assert auto < 2 * (2 << 30) * (1 + 1 / 32) + TAIL_SPLIT_BYTES + 131072 * 400


def test_stored_logit_workspace_single_block_up_to_2048_hidden(clp):
    # D <= 2048: the dH GEMM forms G from the stored logits itself, so one
    # logit block serves every chunk (no double buffering); larger chunks
    # are allowed in exchange (4 GiB of logits instead of 2 x 2 GiB).
    p = clp.make_params(chunk_tokens=2048, flags=1)
    block = stored_block(2048, 151936)
    small = clp.grpo_workspace_size(32768, 2048, 151936, 1, p)
    extra = TAIL_SPLIT_BYTES + H_COPY(2048, 2048)
    assert block + extra < small < block + extra + 32768 * 400
    big = clp.grpo_workspace_size(32768, 2056, 151936, 1, p)
    extra = TAIL_SPLIT_BYTES + H_COPY(2048, 2056)
    assert 2 * block + extra < big < 2 * block + extra + 32768 * 400
    auto = clp.grpo_workspace_size(131072, 1536, 151936, 1, clp.make_params(flags=1))
    assert (2 << 30) < auto < ((4 << 30) * (1 + 1 / 32) + TAIL_SPLIT_BYTES + H_COPY(16384, 1536) +
                               131072 * 400)


@pytest.mark.parametrize("flags", [16, 1, 0])
def test_workspace_budget_caps_the_chunk(clp, flags):
    n, d, v = 65536, 4096, 128256
    free = clp.grpo_workspace_size(n, d, v, 1, clp.make_params(flags=flags))
    for limit in (free // 2, free // 4):
        got = clp.grpo_workspace_size(n, d, v, 1, clp.make_params(flags=flags,
                                                                 workspace_limit_bytes=limit))
        assert got <= limit
    # A generous budget changes nothing.
    same = clp.grpo_workspace_size(n, d, v, 1, clp.make_params(flags=flags,
                                                              workspace_limit_bytes=free * 4))
    assert same == free


def test_workspace_budget_too_small_is_an_error(clp):
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_workspace_size(65536, 4096, 128256, 1,
                                clp.make_params(workspace_limit_bytes=1 << 20))
    assert e.value.code == -4
    # An explicit chunk that does not fit the budget is refused too.
    with pytest.raises(clp.GrpoError) as e:
        clp.grpo_workspace_size(65536, 4096, 128256, 1,
                                clp.make_params(flags=1, chunk_tokens=16384,
                                                workspace_limit_bytes=1 << 30))
    assert e.value.code == -4


def test_sequence_mean_flag_is_accepted(clp):
    assert clp.grpo_workspace_size(1024, 64, 100, 256,
                                   clp.make_params(flags=clp._binding.FLAG_SEQUENCE_MEAN)) > 0


def test_launch_timing_without_launches(clp):
    # Host-only: switching the timing on and off and reading an empty record
    # makes no CUDA call.
    clp.grpo_launch_timing_enable(True)
    assert clp.grpo_launch_timing_read() == []
    clp.grpo_launch_timing_enable(False)
    assert clp.grpo_launch_timing_read() == []


def test_launch_timing_read_rejects_bad_arguments(clp):
    lib = clp.lib
    count = ctypes.c_int(-5)
    assert lib.grpo_launch_timing_read(None, 0, ctypes.byref(count)) == 0
    assert count.value == 0
    assert lib.grpo_launch_timing_read(None, 0, None) == -1
    assert lib.grpo_launch_timing_read(None, 4, ctypes.byref(count)) == -1
    buf = (clp._binding.GrpoKernelTime * 1)()
    assert lib.grpo_launch_timing_read(buf, -1, ctypes.byref(count)) == -1
    assert ctypes.sizeof(clp._binding.GrpoKernelTime) == 56
