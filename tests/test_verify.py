"""Bookkeeping of a speculative verify pass (field report, section 3B;
2 x RTX PRO 6000 post): the oracle on hand-worked passes, then the library's
host entry point against it.  No GPU."""
import numpy as np
import pytest

from oracle import verify as OV


def test_oracle_by_hand():
    st = OV.Stats(3)
    assert st.add([5, 6, 7], [5, 6, 9, 1]) == (2, [5, 6, 9], [1, 1, 1, 0])   # two drafts kept, t_2 emitted
    assert st.add([1, 2, 3], [3, 4, 5, 6]) == (0, [3], [1, 0, 0, 0])        # the first draft already wrong
    assert st.add([1, 2, 3], [1, 2, 3, 8]) == (3, [1, 2, 3, 8], [1, 1, 1, 1])  # every draft kept, plus t_3
    assert st.add([7, 2, 3], [7, 9, 3, 8]) == (1, [7, 9], [1, 1, 0, 0])     # a later match does not count
    assert (st.passes, st.tokens, st.hist) == (4, 3 + 1 + 4 + 2, [1, 1, 1, 1])
    assert st.tokens_per_pass() == 2.5
    assert OV.Stats(0).add([], [4]) == (0, [4], [1])                         # no drafts: one token


@pytest.mark.parametrize("seed,n_draft,p", [(1, 5, 0.7), (2, 4, 0.9), (3, 1, 0.5), (4, 15, 0.95), (5, 0, 0.5)])
def test_library_matches_oracle(seed, n_draft, p):
    from bit_quantised_expert_gb300 import _abi as A
    rng = np.random.default_rng(seed)
    st = A.bqe_verify_stats()
    ref = OV.Stats(A.VERIFY_MAX_DRAFT)
    for _ in range(300):
        target = rng.integers(0, 1000, size=n_draft + 1).astype(np.int32)
        draft = np.where(rng.random(n_draft) < p, target[:n_draft], rng.integers(1000, 2000, size=n_draft))
        draft = draft.astype(np.int32)
        a, emitted, mask = ref.add(draft.tolist(), target.tolist())
        em, mk = A.bqe_verify_pass(draft, target, st)
        assert em.tolist() == emitted and mk.tolist() == mask
    assert (st.passes, st.tokens, list(st.hist)) == (ref.passes, ref.tokens, ref.hist)


def test_library_rejects_bad_arguments():
    from bit_quantised_expert_gb300 import _abi as A
    with pytest.raises(A.BqeError):
        A.bqe_verify_pass(np.zeros(16, np.int32), np.zeros(17, np.int32))  # more drafts than allowed
