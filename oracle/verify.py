"""Oracle for the bookkeeping of a speculative verify pass.  TEST
INFRASTRUCTURE ONLY.

The DeepSeek-V4.1-Flash field report (section 3B) runs a draft-and-verify
loop: each pass verifies several draft tokens in one batched forward
(verify rows = the last accepted token plus the drafts), accepts a prefix,
and reports tokens per pass (3.39 in its log); decode speed is accepted
tokens per pass divided by the pass time.  The 2 x RTX PRO 6000 post verifies
all candidates layer by layer in one batch, commits the accepted prefix and
rolls the rejected tail back.

Readings (the pages give no rule; greedy verification, the plainest):
  * row 0 holds the last accepted token, rows 1..D the drafts d_1..d_D; the
    target's prediction after row i is t_i;
  * draft d_(i+1) is accepted while it equals t_i, for i = 0, 1, ...; with a
    drafts accepted, rows 0..a are committed and the pass emits a + 1 tokens
    (the accepted drafts and t_a); rows a+1..D are rolled back;
  * the statistics are passes, emitted tokens and the count of each a.
"""
from __future__ import annotations


def accept(draft, target):
    """Accepted draft count a: the longest prefix with draft[i] == target[i]."""
    a = 0
    while a < len(draft) and draft[a] == target[a]:
        a += 1
    return a


class Stats:
    def __init__(self, max_draft: int):
        self.passes = 0
        self.tokens = 0
        self.hist = [0] * (max_draft + 1)

    def add(self, draft, target):
        """One pass: returns (a, emitted tokens, committed-row mask)."""
        a = accept(draft, target)
        self.passes += 1
        self.tokens += a + 1
        self.hist[a] += 1
        mask = [1 if r <= a else 0 for r in range(len(draft) + 1)]
        return a, draft[:a] + [target[a]], mask

    def tokens_per_pass(self) -> float:
        return self.tokens / self.passes if self.passes else 0.0
