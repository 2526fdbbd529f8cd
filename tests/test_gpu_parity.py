"""GPU parity: the CUDA path through the C-ABI against the fp64 oracle, element by
element on the same seeded inputs. Tolerances: relative L2 error per tensor <= 1e-5 (fp32)
or 2e-2 (bf16) on logits, IIR scan inputs, FIR inputs, K/V and sliced states; accepted
lengths, corrections, candidates, KV lengths and slice indices exact, except on rounds the
oracle flags as near-ties (counted). Discrete decisions are compared in the kernel's
precision: the oracle's acceptance on the library's fp32 logits; the oracle state is then sliced
at the library's (k, candidate) and compared."""
import numpy as np
import pytest
import torch

from synth import LayerSpec, gen_round, get_workload
from gpu_harness import Pair, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from lossless_speculative_verify_gb300.build import build
    build()


def _lockstep(pair, rounds, first_round=0, drafts=None):
    """Run rounds on both sides; anchor = previous correction. Every round checks the
    block outputs, the decisions in the kernel's precision and the sliced state. The
    oracle's own fp64 decisions must match too (fp32 and bf16 alike), except on sequences
    it flags as near-ties, which are counted. Returns the number of rounds with a flagged
    near-tie."""
    ties = 0
    anchor = None
    for r in range(first_round, first_round + rounds):
        rnd = gen_round(pair.wl, r, anchor=anchor)
        if drafts is not None:
            rnd["tokens"] = drafts(pair, rnd)
        out = pair.run_round(rnd)
        if out.tie.any():
            ties += 1
        assert pair.fp64_disagreements == 0, (r, out.gk, out.k, out.gc, out.corr, out.gcand, out.cand, out.tie)
        pair.compare_state()
        anchor = out.gc
    return ties


def identity_drafts(pair, rnd, wrong_at=None):
    """Drafts equal to the oracle's greedy chain (optionally wrong at one position)."""
    toks = rnd["tokens"].copy()
    B, C, T = toks.shape
    for b in range(B):
        for c in range(C):
            probe = pair.states[b].clone()
            for i in range(T - 1):
                nxt = int(np.argmax(pair.tgt.step(probe, int(toks[b, c, i]))))
                w = wrong_at if np.isscalar(wrong_at) or wrong_at is None else wrong_at[c]
                if w is not None and i == w:
                    nxt = (nxt + 1) % pair.wl.vocab
                toks[b, c, i + 1] = nxt
    return toks


def identity_drafts_per_seq(pair, rnd, wrong_at):
    """Drafts equal to the oracle's greedy chain, made wrong at draft wrong_at[b][c] + 1 of
    sequence b, candidate c (None: every draft right), so that candidate accepts exactly
    wrong_at[b][c] drafts (or gamma)."""
    toks = rnd["tokens"].copy()
    B, C, T = toks.shape
    for b in range(B):
        for c in range(C):
            probe = pair.states[b].clone()
            for i in range(T - 1):
                nxt = int(np.argmax(pair.tgt.step(probe, int(toks[b, c, i]))))
                if wrong_at[b][c] is not None and i == wrong_at[b][c]:
                    nxt = (nxt + 1) % pair.wl.vocab
                toks[b, c, i + 1] = nxt
    return toks


def _wide_geometry():
    """The 4 x 4-candidate geometry at width 4096 (gamma 12, [FIR-3, IIR-16, FIR-7, attention
    32 x 128]) in greedy mode with a short prefix."""
    return get_workload("d4096_l8_p32k_b4c4_bf16").replace(
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 7), LayerSpec("attn", 32)),
        mode="greedy", prefix_len=96)


@pytest.mark.parametrize("wrong_at,want_k,want_cand", [
    # committed k = 1 (FIR-7 tail mixes 5 old-tail rows and 2 block rows), 5, 11, 12; the
    # committed candidate is never candidate 0, so its K/V side rows are copied at k > 0
    ([[0, 0, 1, 0], [1, 5, 3, 2], [0, 2, 4, 11], [3, None, None, 0]], [1, 5, 11, 12], [2, 1, 3, 1]),
    # committed k = 0 (every candidate rejects its first draft), 6 (tail all block rows), 2, 12
    ([[0, 0, 0, 0], [6, 0, 6, 1], [0, 1, 2, 0], [None, 11, 12 - 1, None]], [0, 6, 2, 12], [0, 0, 2, 0]),
])
def test_forced_slices_wide_multi_candidate(wrong_at, want_k, want_cand):
    """State restoration at chosen block indices on the 4096-wide, gamma-12, 4 x 4-candidate
    geometry (Figure 1(d): the block index k, the last L-1 FIR inputs, s_k): each sequence's
    candidates accept the given numbers of drafts, the longest is committed, and the sliced
    state (FIR-3 and FIR-7 tails, the IIR state rebuilt over k+1 steps, the committed
    candidate's K/V rows, KV lengths) matches the oracle; one more round then runs from it."""
    wl = _wide_geometry()
    pair = Pair(wl)
    pair.import_synthetic(wl.prefix_len)
    rnd = gen_round(wl, 5)
    rnd["tokens"] = identity_drafts_per_seq(pair, rnd, wrong_at)
    kv0 = [s.kv_len for s in pair.states]
    out = pair.run_round(rnd)
    np.testing.assert_array_equal(out.k, want_k)          # the oracle's own fp64 decisions
    np.testing.assert_array_equal(out.cand, want_cand)
    for b in range(wl.batch):
        if out.tie[b]:       # a flagged near-tie may flip the library's argmax: the oracle
            continue         # then slices at the library's decision, compared below
        assert (out.gk[b], out.gcand[b], out.gc[b]) == (want_k[b], want_cand[b], out.corr[b]), b
    assert [s.kv_len for s in pair.states] == [k0 + int(k) + 1 for k0, k in zip(kv0, out.gk)]
    pair.compare_state()
    assert pair.ver.flags() == 0
    _lockstep(pair, 1, first_round=6)


def test_tiny_fp32_prefill_matches_oracle():
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    pair.prefill(250)                   # 3 full chunks of 64 and a ragged chunk of 58
    # 250 sequential fp32 IIR steps with |lambda| <= 0.99 accumulate rounding ~ eps/(1-|lambda|)
    pair.compare_state(tol=5e-5)


def test_tiny_fp32_rounds_greedy():
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    pair.import_synthetic(wl.prefix_len)
    assert _lockstep(pair, 6) <= 1
    # identity drafter: every draft accepted, bonus from the last position
    rnd = gen_round(wl, 100)
    rnd["tokens"] = identity_drafts(pair, rnd)
    out = pair.run_round(rnd)
    assert out.k[0] == wl.gamma and out.gk[0] == wl.gamma and out.gc[0] == out.corr[0]
    pair.compare_state()


@pytest.mark.parametrize("k_force", list(range(7)))
def test_slice_at_every_k(k_force):
    """State restoration at each block index (Lemma 3): FIR tail, IIR state, KV length."""
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    pair.import_synthetic(40)
    rnd = gen_round(wl, 7)
    rnd["tokens"] = identity_drafts(pair, rnd, wrong_at=k_force if k_force < wl.gamma else None)
    kv0 = pair.states[0].kv_len
    out = pair.run_round(rnd)
    assert out.k[0] == k_force and out.gk[0] == k_force and out.gc[0] == out.corr[0]
    assert pair.states[0].kv_len == kv0 + k_force + 1
    pair.compare_state()
    # decoding continues identically from the sliced state
    assert _lockstep(pair, 2, first_round=8) <= 1


def test_tiny_fp32_sampling_rounds():
    wl = get_workload("tiny_d64_fp32").replace(mode="sampling", q_alpha=0.5)
    pair = Pair(wl)
    pair.import_synthetic(64)
    assert _lockstep(pair, 10) <= 2


def test_sampling_identity_drafts_with_q_equal_p_accept_all():
    """With q = p (the target's own distribution), rejection sampling accepts every draft."""
    wl = get_workload("tiny_d64_fp32").replace(mode="sampling", gamma=4)
    pair = Pair(wl)
    pair.import_synthetic(32)
    rnd = gen_round(wl, 3)
    toks = identity_drafts(pair, rnd)
    probe = pair.states[0].clone()
    q = np.zeros_like(rnd["q"])
    for i in range(wl.gamma):
        lg = pair.tgt.step(probe, int(toks[0, 0, i]))
        p = np.exp(lg - lg.max())
        q[0, 0, i] = (p / p.sum()).astype(np.float32)
    rnd.update(tokens=toks, q=q)
    out = pair.run_round(rnd)
    assert out.k[0] == wl.gamma and out.gk[0] == wl.gamma


def test_multi_candidate_fp32():
    wl = get_workload("tiny_d64_fp32").replace(batch=2, n_cand=3, gamma=5)
    pair = Pair(wl)
    pair.import_synthetic(48)
    rnd = gen_round(wl, 1)
    rnd["tokens"] = identity_drafts(pair, rnd, wrong_at=[1, 4, 2])
    out = pair.run_round(rnd)
    assert list(out.cand) == [1, 1] and list(out.gcand) == [1, 1]
    np.testing.assert_array_equal(out.gk, [4, 4])
    pair.compare_state()
    assert _lockstep(pair, 3, first_round=2) <= 1


def _shared_prefixes(pair, rnd):
    """Candidates 1 and 2 copy candidate 0's first draft, candidate 2 also its second, so
    the accepted path keeps several candidates alive."""
    toks = rnd["tokens"].copy()
    toks[:, 1, 1] = toks[:, 0, 1]
    toks[:, 2, 1:3] = toks[:, 0, 1:3]
    return toks


@pytest.mark.parametrize("rule", ["recursive", "max_accept"])
def test_multi_candidate_sampling_fp32(rule):
    """Several candidates under sampling, both rules: committed k, correction and candidate
    and every candidate's words exact against the oracle (fp32, also its own fp64
    decisions), over rounds where candidates share drafts."""
    wl = get_workload("tiny_d64_fp32").replace(batch=2, n_cand=3, gamma=5, mode="sampling", q_alpha=0.5,
                                               cand_rule=rule)
    pair = Pair(wl)
    pair.import_synthetic(48)
    assert _lockstep(pair, 8, drafts=_shared_prefixes) <= 2


def test_multi_candidate_sampling_bf16():
    wl = get_workload("tiny_d64_fp32").replace(
        d=256, dtype="bf16", head_dim=128, batch=2, n_cand=4, gamma=6, mode="sampling",
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 7), LayerSpec("attn", 2)))
    pair = Pair(wl)
    pair.import_synthetic(300)
    _lockstep(pair, 4)


def test_multi_candidate_bf16_wide_block():
    """112 block rows (4 sequences x 4 candidates x 7), more than the in-projection
    epilogue's mixers take: the standalone FIR / IIR kernels run on 16 blocks, with
    decisions and the sliced state against the oracle."""
    wl = get_workload("tiny_d64_fp32").replace(
        d=256, dtype="bf16", head_dim=128, batch=4, n_cand=4, gamma=6, mode="sampling",
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 7), LayerSpec("attn", 2)))
    pair = Pair(wl)
    pair.import_synthetic(200)
    _lockstep(pair, 3)


@pytest.mark.parametrize("batch,n_cand", [(1, 1), (4, 4)], ids=["fused_mixers", "standalone_scans"])
def test_bf16_other_filter_lengths_and_poles(batch, n_cand):
    """FIR lengths 5 and 16 and an 8-pole IIR: the projection's generic FIR epilogue (the
    lengths 3 and 7 have instantiations of their own) and the modal scan at another pole
    count, fused in the in-projections at 7 rows and standalone at 112 rows."""
    wl = get_workload("tiny_d64_fp32").replace(
        d=256, dtype="bf16", head_dim=128, batch=batch, n_cand=n_cand, gamma=6, mode="sampling",
        layers=(LayerSpec("fir", 5), LayerSpec("iir", 8), LayerSpec("fir", 16), LayerSpec("attn", 2)))
    pair = Pair(wl)
    pair.import_synthetic(150)
    _lockstep(pair, 3)


def test_bf16_small_stack_sampling():
    wl = get_workload("d1024_l8_p8k_bf16").replace(d=256, head_dim=128, prefix_len=500,
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 3), LayerSpec("attn", 2)) * 2)
    pair = Pair(wl)
    pair.prefill(wl.prefix_len)          # chunks of 128 and a ragged tail of 116
    pair.compare_state(tol=TOL["bf16"])
    _lockstep(pair, 5)


def test_bf16_long_prefix_multi_tile_chunks():
    """A prefix long enough that each attention CTA covers several 128-key tiles, with a
    ragged last tile (40000 = 312 x 128 + 64)."""
    wl = get_workload("d1024_l8_p8k_bf16").replace(d=256, head_dim=128, prefix_len=40000,
        layers=(LayerSpec("fir", 3), LayerSpec("attn", 2)))
    pair = Pair(wl)
    pair.import_synthetic(wl.prefix_len)
    _lockstep(pair, 3)


def test_full_size_d1024_l8_p8k():
    """The bench workload at full size (d=1024, 8 layers, 8192 cached tokens, gamma 6,
    sampling), same kernels and launch shapes as the benchmark."""
    wl = get_workload("d1024_l8_p8k_bf16")
    pair = Pair(wl)
    pair.import_synthetic(wl.prefix_len)
    _lockstep(pair, 3)


def test_host_errors():
    from lossless_speculative_verify_gb300 import EvsError
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl, t_max=20)
    with pytest.raises(EvsError) as e:
        pair.ver.slice()
    assert e.value.status == 3                              # slice without a verify
    with pytest.raises(EvsError) as e:
        pair.ver.prefill(torch.zeros((1, 21), dtype=torch.int32, device="cuda"))
    assert e.value.status == 2                              # beyond t_max
    pair.ver.prefill(torch.full((1, 14), 65, dtype=torch.int32, device="cuda"))
    toks = torch.full((1, 1, 7), 65, dtype=torch.int32, device="cuda")
    with pytest.raises(EvsError) as e:
        pair.ver.verify(toks)                               # 14 + 7 > 20
    assert e.value.status == 2
    assert pair.ver.flags() == 0


def test_device_flag_on_bad_token_and_bad_k():
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    pair.import_synthetic(16)
    toks = torch.full((1, 1, 7), 65, dtype=torch.int32, device="cuda")
    toks[0, 0, 3] = 9999
    pair.ver.verify(toks)
    assert pair.ver.flags() & 8
    bad_k = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    pair.ver.slice(bad_k)
    assert pair.ver.flags() & 2


@pytest.mark.parametrize("vocab,gamma,mode", [(256, 6, "greedy"), (1024, 6, "sampling"), (2048, 31, "sampling"),
                                              (4096, 12, "greedy"), (4096, 9, "sampling")])
def test_vocabularies_and_largest_block_fp32(vocab, gamma, mode):
    """Every instance of the acceptance kernel (1, 4, 8 and 16 token ids per thread; 2 is
    the 512-entry vocabulary of the other cases) and the largest block, gamma 31 (32
    positions), against the oracle over consecutive rounds with two candidates."""
    wl = get_workload("tiny_d64_fp32").replace(vocab=vocab, gamma=gamma, mode=mode, batch=2, n_cand=2,
                                               q_alpha=0.5)
    pair = Pair(wl)
    pair.import_synthetic(40)
    _lockstep(pair, 3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rounds_from_the_empty_state(dtype):
    """Verify rounds straight from the empty state: no cached keys, so each query attends
    to the block's own keys only (the attention's prefix chunks are all empty)."""
    if dtype == "f32":
        wl = get_workload("tiny_d64_fp32").replace(prefix_len=0)
    else:
        wl = get_workload("d1024_l8_p8k_bf16").replace(d=256, head_dim=128, prefix_len=0, n_cand=2,
            layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 7), LayerSpec("attn", 2)))
    pair = Pair(wl)
    assert _lockstep(pair, 3) <= 3
