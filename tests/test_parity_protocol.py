"""The comparison the GPU parity tests use, checked on the CPU with planted results: a token
that differs from the oracle's passes only where the oracle's own margin at that step is
below the near-tie threshold, and a hidden state beyond tolerance always fails."""
import numpy as np
import pytest

import oracle as O

from _util import NEAR_TIE, TOL, compare_block


def _ref(B=2, n=3, bb=4):
    tokens = np.arange(1, B * n + 1, dtype=np.int64).reshape(B, n)
    return O.BlockResult(tokens=tokens, hidden_out=np.zeros((B, n, bb)), logit_gap=np.ones((B, n)),
                         kth_gap=np.ones((B, n)), selected=None, steps=[])


def test_identical_results_compare_every_step():
    ref = _ref()
    cmp = compare_block(ref.tokens.copy(), ref.hidden_out.astype(np.float32), ref, "bf16")
    assert cmp.steps_compared == 6 and cmp.tie_divergences == [] and cmp.max_hidden_err == 0.0


def test_a_different_token_at_a_clear_margin_fails():
    ref = _ref()
    tok = ref.tokens.copy()
    tok[0, 1] += 1
    with pytest.raises(AssertionError, match="token mismatch"):
        compare_block(tok, None, ref, "bf16")


@pytest.mark.parametrize("which", ["logit_gap", "kth_gap"])
def test_a_different_token_at_a_near_tie_is_counted_and_ends_that_sequence(which):
    ref = _ref()
    getattr(ref, which)[1, 1] = 0.5 * NEAR_TIE["bf16"]
    tok = ref.tokens.copy()
    tok[1, 1] += 7
    tok[1, 2] += 3  # after a divergence the sequences follow different tokens: not compared
    cmp = compare_block(tok, None, ref, "bf16")
    assert len(cmp.tie_divergences) == 1 and cmp.tie_divergences[0][:2] == (1, 1)
    assert cmp.steps_compared == 3 + 2


def test_a_margin_at_the_threshold_is_not_a_tie():
    ref = _ref()
    ref.logit_gap[0, 0] = NEAR_TIE["f32"]
    tok = ref.tokens.copy()
    tok[0, 0] += 1
    with pytest.raises(AssertionError):
        compare_block(tok, None, ref, "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_hidden_state_beyond_tolerance_fails(dtype):
    ref = _ref()
    hid = ref.hidden_out.copy()
    hid[1, 2, 3] = 1.5 * TOL[dtype]
    with pytest.raises(AssertionError, match="hidden state"):
        compare_block(ref.tokens.copy(), hid, ref, dtype)
    hid[1, 2, 3] = 0.5 * TOL[dtype]
    assert compare_block(ref.tokens.copy(), hid, ref, dtype).max_hidden_err == pytest.approx(0.5 * TOL[dtype])
