"""Host arithmetic of the decode loop's summary (CPU): the tutorial's measures from recorded counts
and times, checked by hand."""
import numpy as np
import pytest

from quantized_speculative_decoding_qspec_gb300 import decode as dec


def make_runs(accept_len, gamma, t_draft_ms, t_verify_ms, spec_wall_s, t_target_ms, target_wall_s, n_target_tok,
              tally=None):
    n = np.asarray(accept_len, dtype=np.int32)
    spec = {"accept_len": n, "t_draft_ms": np.asarray(t_draft_ms, float), "t_verify_ms": np.asarray(t_verify_ms, float),
            "wall_s": spec_wall_s}
    if tally is not None:
        spec["tally"] = np.asarray(tally, float)
    target = {"t_target_ms": np.asarray(t_target_ms, float), "wall_s": target_wall_s,
              "generated": [list(range(n_target_tok))] * n.shape[1]}
    return spec, target


def test_summary_by_hand():
    gamma = 3
    # 4 iterations x 2 sequences: accepted drafts per (iteration, sequence)
    n = [[3, 0], [1, 2], [3, 3], [0, 1]]
    spec, target = make_runs(n, gamma, t_draft_ms=[0.3, 0.3, 0.3, 0.3], t_verify_ms=[0.2, 0.2, 0.25, 0.2],
                             spec_wall_s=0.004, t_target_ms=[0.1, 0.1, 0.1], target_wall_s=0.010, n_target_tok=20)
    s = dec.summarize(spec, target, gamma)
    assert s["acceptance_rate"] == pytest.approx(13 / 8 / 3)                 # mean accepted / gamma
    ET = (4 + 1 + 2 + 3 + 4 + 4 + 1 + 2) / 8                                  # n + 1 tokens per iteration
    assert s["accepted_tokens_per_iteration"] == pytest.approx(ET)
    assert s["t_draft_ms_per_token"] == pytest.approx(0.1)
    assert s["t_verify_ms"] == pytest.approx(0.2)
    assert s["t_overhead_ms"] == pytest.approx(1.0 - (0.3 + 0.2))            # 1 ms per iteration of wall time
    assert s["speedup_model"] == pytest.approx(ET * 0.1 / 1.0)
    assert s["speedup_model_device_only"] == pytest.approx(ET * 0.1 / 0.5)
    assert s["spec_tokens_per_s"] == pytest.approx(2 * ET * 4 / 0.004)
    assert s["target_only_tokens_per_s"] == pytest.approx(2 * 20 / 0.010)
    assert s["speedup_measured"] == pytest.approx(s["spec_tokens_per_s"] / s["target_only_tokens_per_s"])
    assert "top1" not in s


def test_full_acceptance_gives_gamma_plus_one():
    gamma = 4
    spec, target = make_runs([[4, 4, 4]] * 5, gamma, [1.0] * 5, [1.0] * 5, 0.5, [1.0], 1.0, 10)
    s = dec.summarize(spec, target, gamma)
    assert s["acceptance_rate"] == 1.0 and s["accepted_tokens_per_iteration"] == gamma + 1


def test_top1_tally_ratios():
    # positions, agree, both high, agree there, both low, agree there, sum p1 verify, sum p1 draft
    tally = [200, 150, 120, 118, 50, 20, 160.0, 150.0]
    spec, target = make_runs([[1]], 3, [0.3], [0.2], 0.001, [0.1], 0.01, 5, tally=tally)
    t = dec.summarize(spec, target, 3)["top1"]
    assert t == {"positions": 200, "agreement": 0.75, "mean_p1_verify_mode": 0.8, "mean_p1_draft_mode": 0.75,
                 "both_high_share": 0.6, "agreement_both_high": pytest.approx(118 / 120),
                 "agreement_both_low": 0.4}
    empty = dec.summarize(*make_runs([[1]], 3, [0.3], [0.2], 0.001, [0.1], 0.01, 5, tally=[0] * 8), 3)["top1"]
    assert empty["agreement"] is None and empty["agreement_both_high"] is None
