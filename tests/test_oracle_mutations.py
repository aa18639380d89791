"""The pins must catch plausible mistakes: each case plants one mistake in the
oracle (on the CPU, through monkeypatching) and checks that a pin test fails."""
import numpy as np
import pytest

from oracle import nsa as O
from oracle import dsa as D
import tests.test_oracle_pins as P


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_shifted_overlap_is_caught(monkeypatch):
    real = O.overlap_matrix

    def shifted(Nc, nb, l, d, lsel):       # block j fed by compressed blocks 4j-4..4j
        Om = real(Nc + 3, nb, l, d, lsel)
        return Om[3:]
    monkeypatch.setattr(O, "overlap_matrix", shifted)
    _fails(P.test_block_scores_one_hot_and_conservation)


def test_partial_block_visibility_is_caught(monkeypatch):
    def early(t, l, d, Nc):                # a block counted visible once it starts
        t = np.asarray(t, dtype=np.int64)
        return np.minimum(t // d + 1, Nc)
    monkeypatch.setattr(O, "num_visible_compressed", early)
    _fails(P.test_cmp_attention_causality_and_empty)


def test_dropped_position_embedding_is_caught(monkeypatch):
    real = O.compress
    monkeypatch.setattr(O, "compress", lambda X, PE, W, l, d: real(X, 0 * PE, W, l, d))
    _fails(P.test_compress_matches_torch_unfold_matmul)


def test_reversed_tie_break_is_caught(monkeypatch):
    def rev(S32, t, n, lsel):
        jt = t // lsel
        out = np.full(n, -1, dtype=np.int32)
        if jt + 1 <= n:
            out[: jt + 1] = np.arange(jt + 1)
            return out
        forced = np.array(sorted({0, jt, jt - 1}))
        cand = np.setdiff1d(np.arange(jt + 1), forced)
        order = np.lexsort((-cand, -S32[cand]))
        out[:] = np.sort(np.concatenate([forced, cand[order[: n - forced.size]]]))
        return out
    monkeypatch.setattr(O, "select_blocks", rev)
    _fails(P.test_select_blocks_brute_force, 1)


def test_wrong_scale_is_caught(monkeypatch):
    real = O._attend
    monkeypatch.setattr(O, "_attend", lambda q, K, V, keys, scale: real(q, K, V, keys, 2 * scale))
    _fails(P.test_selection_only_equals_full_attention_when_all_blocks_fit)


def test_window_off_by_one_is_caught(monkeypatch):
    real = O._attend

    def win(q, t, K, V, w, scale):         # (t-w-1, t]: one token too many
        return real(q, K, V, np.arange(max(0, t - w), t + 1), scale)
    monkeypatch.setattr(O, "win_attention", win)
    _fails(P.test_uniform_attention_gives_plain_means)


def test_missing_relu_is_caught(monkeypatch):
    monkeypatch.setattr(D, "dsa_indexer_scores", lambda qI, wI, kI: (kI @ qI.T) @ wI)
    _fails(P.test_dsa_indexer_brute_force)


# ---------------------------------------------------------------- backward oracle
from oracle import nsa_bwd as BW  # noqa: E402
import tests.test_oracle_backward as PB  # noqa: E402


@pytest.fixture(scope="module")
def bwd_case():
    return PB.make_case()


def test_dropped_softmax_correction_is_caught(monkeypatch, bwd_case):
    real = BW.attend_bwd

    def wrong(q, K, V, keys, scale, dO):    # dS = P dP: the "- dO . O" term dropped
        if keys.size == 0:
            return real(q, K, V, keys, scale, dO)
        Kk, Vk = K[keys], V[keys]
        s = (q @ Kk.T) * scale
        P = np.exp(s - s.max(axis=-1, keepdims=True))
        P /= P.sum(axis=-1, keepdims=True)
        dS = P * (dO @ Vk.T)
        return P @ Vk, scale * dS @ Kk, scale * dS.T @ q, P.T @ dO
    monkeypatch.setattr(BW, "attend_bwd", wrong)
    _fails(PB.check_finite_differences, bwd_case)


def test_unscaled_key_gradient_is_caught(monkeypatch, bwd_case):
    real = BW.attend_bwd

    def wrong(q, K, V, keys, scale, dO):
        O_, dq, dK, dV = real(q, K, V, keys, scale, dO)
        return O_, dq, dK / scale, dV
    monkeypatch.setattr(BW, "attend_bwd", wrong)
    _fails(PB.check_finite_differences, bwd_case)


def test_shifted_compression_scatter_is_caught(monkeypatch, bwd_case):
    def wrong(X, PE, W, l, d, dXc):         # block i's gradient lands one token late
        dX, dPE, dW = real(X, PE, W, l, d, dXc)
        return np.roll(dX, 1, axis=0), dPE, dW
    real = BW.compress_bwd
    monkeypatch.setattr(BW, "compress_bwd", wrong)
    _fails(PB.check_finite_differences, bwd_case)


def test_widened_topk_band_is_caught(monkeypatch):
    # a band 1000x too wide would let a wrong DSA top-k set pass the GPU check
    real = D.topk_alternatives
    monkeypatch.setattr(D, "topk_alternatives", lambda I32, k, rel_tol: real(I32, k, 1e3 * rel_tol))
    _fails(P.test_topk_alternatives_cases)


def test_topk_band_ignoring_need_is_caught(monkeypatch):
    # accepting any number of picks from the band admits sets of the wrong size
    real = D.topk_alternatives

    def loose(I32, k, rel_tol):
        gap, above, band, need = real(I32, k, rel_tol)
        return gap, above, np.union1d(band, np.arange(I32.shape[0])), need
    monkeypatch.setattr(D, "topk_alternatives", loose)
    _fails(P.test_topk_set_valid_rejects_planted_invalid_sets)


def test_selection_band_dropping_forced_blocks_is_caught(monkeypatch):
    real = O.selection_alternatives

    def no_forced(S32, t, n, lsel, rel_tol):
        gap, definite, band, need = real(S32, t, n, lsel, rel_tol)
        jt = t // lsel
        return gap, definite - {0, jt - 1}, band | {0, jt - 1, 3}, need
    monkeypatch.setattr(O, "selection_alternatives", no_forced)
    _fails(P.test_selection_set_valid_rejects_planted_invalid_rows)


def test_dropped_branch_in_the_combined_output_is_caught(monkeypatch):
    import tests.test_oracle_backward as BWT
    real = O.win_attention
    monkeypatch.setattr(O, "win_attention", lambda *a, **kw: 0.0 * real(*a, **kw))
    _fails(BWT.test_combined_output_matches_an_independent_formulation, BWT.make_case())


def test_selected_branch_scored_with_the_window_gate_is_caught(monkeypatch):
    # the selected branch's output replaced by the window's: what a gate or
    # branch mix-up in the combine would produce
    import tests.test_oracle_backward as BWT
    monkeypatch.setattr(O, "sel_attention", lambda q, t, K, V, idx, lsel, scale:
                        O.win_attention(q, t, K, V, BWT.PARAMS.w, scale))
    _fails(BWT.test_combined_output_matches_an_independent_formulation, BWT.make_case())
