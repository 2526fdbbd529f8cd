"""fp64 CPU oracle for replay-free block verification (test infrastructure only).

This package is the plain, slow definition that the CUDA path is checked against. Only
the test-suite, the smoke check of ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it; the library never does, and it imports nothing from the
library. It shares no code with the CUDA path: the only common module is ``synth``,
which draws seeded random inputs and holds none of the method's arithmetic.

Sources, all from "EvSpark: Lossless Speculative Decoding for Hybrid DNA Foundation
Models" (summary page, English; the Chinese page is the same text):
  * Figure 1(c): the target verifies the old anchor and the drafts in one block; a
    correction becomes the next unconsumed anchor.
  * Figure 1(d): state returns to block index k: the readable KV prefix is shortened, the
    last L-1 outer-FIR inputs are selected (u2, u3 for k=3, L=3) and IIR state s_k is kept.
  * Interpretation, paragraph 1: one initial-state block forward plus a common
    state-slicing protocol restores FIR, IIR and KV state (Lemma 2, block-forward
    contract; Lemma 3, state restoration; Theorem 1, sequence-level exactness).
  * ReaDy summary, section 3.1 and appendix D.2: greedy acceptance stops at the first
    argmax mismatch; accepting every draft adds a target-sampled bonus token; rejection
    sampling preserves the target distribution.

Layer internals are not given on the pages; the readings used here (RMS norm without
gain, depthwise FIR on the in-projected inputs, diagonal complex modal IIR with real
readout, attention without positional encoding, untied LM head) are listed in the
design notes of the repository.

Modules: ``model`` (token-by-token decode and an independent block-form forward),
``accept`` (greedy and rejection-sampling acceptance), ``verify`` (one round: block of
steps, acceptance, snapshot at k; and one step of native decoding).
"""
from .model import Target, SeqState
from .accept import (softmax_t, greedy_accept, sampling_accept, inverse_cdf, residual,
                     select_candidate, multi_candidate_accept)
from .verify import (verify_round, prefill, RoundResult, block_pass, accept_block, commit, decode_step,
                     pick_next)

__all__ = ["Target", "SeqState", "softmax_t", "greedy_accept", "sampling_accept",
           "inverse_cdf", "residual", "select_candidate", "verify_round", "prefill",
           "RoundResult", "block_pass", "accept_block", "commit", "decode_step", "pick_next", "multi_candidate_accept"]
