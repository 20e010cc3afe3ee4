"""Oracle of the model-free n-gram (prompt lookup) drafter.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): pure Python over each
request's token list, in the order the method is stated.

What it follows: "Co-Designing AI Models Using Speculative Decoding for
Faster LLM Inference", Table 1 (suffix / n-gram drafting: string matching over
the token stream, no model, one lookup, best for workloads with high
repetition), and the model-free passage of "Speculative Decoding"
(glossary), section "Variants: Draft Models, EAGLE, Medusa, and Model-Free
Methods" (n-gram or prompt-lookup drafting proposes tokens by matching strings
that already appear in the context).

Readings (the pages give no algorithm):
  - for n = n_max down to n_min: the suffix is the context's last n tokens;
    its occurrence is the latest earlier window equal to it that ends before
    the context's last token (so at least one token follows it);
  - the first n with an occurrence wins; the proposal is the up to K tokens
    that follow that occurrence in the context (fewer when the context ends
    first); with no occurrence for any n, nothing is proposed (K_b = 0).

Parity: exact (integer work).  Pinned against Python's str.rfind over an
encoding of the tokens, a periodic stream's closed form and special cases
(tests/test_oracle_pins_ngram.py).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def propose(ctx: Sequence[int], K: int, n_min: int, n_max: int) -> Tuple[List[int], int]:
    """(proposed tokens, end index of the matched window or -1) for one request."""
    L = len(ctx)
    for n in range(n_max, n_min - 1, -1):
        if n <= 0 or n > L - 1:
            continue
        suffix = list(ctx[L - n:])
        for e in range(L - 2, n - 2, -1):  # window ctx[e-n+1 .. e], latest first
            if list(ctx[e - n + 1:e + 1]) == suffix:
                out = list(ctx[e + 1:min(e + 1 + K, L)])
                return out, e
    return [], -1


def propose_batch(contexts: Sequence[Sequence[int]], K: int, n_min: int, n_max: int):
    """drafts (B x K, -1 padded) and counts (B,) as lists."""
    drafts, counts = [], []
    for ctx in contexts:
        toks, _ = propose(ctx, K, n_min, n_max)
        counts.append(len(toks))
        drafts.append(toks + [-1] * (K - len(toks)))
    return drafts, counts
