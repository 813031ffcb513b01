"""Host logic of negl_prob calibration (CPU only): the selection rule."""
from block_sparse_attention_fwd_gb300.calibrate import Trial, select_negl


def _t(negl, rel, cos):
    return Trial(negl, 0.0, {"G_Q": rel, "G_K": rel / 2, "G_V": rel / 3},
                 {"G_Q": cos, "G_K": 1.0, "G_V": 1.0})


def test_largest_candidate_meeting_both_targets():
    trials = [_t(0.01, 0.02, 0.9999), _t(0.05, 0.06, 0.999), _t(0.1, 0.12, 0.995)]
    assert select_negl(trials, max_rel_l2=0.1, min_cos=0.99) == 0.05
    assert select_negl(trials, max_rel_l2=0.2, min_cos=0.99) == 0.1
    assert select_negl(trials, max_rel_l2=0.2, min_cos=0.999) == 0.05


def test_non_monotone_errors_are_all_checked():
    trials = [_t(0.01, 0.2, 0.99), _t(0.05, 0.05, 0.999), _t(0.1, 0.3, 0.9)]
    assert select_negl(trials, 0.1, 0.99) == 0.05


def test_no_candidate_means_dense():
    assert select_negl([_t(0.01, 0.5, 0.5)], 0.1, 0.99) == 0.0
    assert select_negl([], 0.1, 0.99) == 0.0


def test_worst_gradient_decides():
    t = Trial(0.05, 0.0, {"G_Q": 0.01, "G_K": 0.2, "G_V": 0.01},
              {"G_Q": 1.0, "G_K": 1.0, "G_V": 0.98})
    assert t.worst_rel_l2 == 0.2 and t.worst_cos == 0.98
    assert select_negl([t], 0.1, 0.9) == 0.0
