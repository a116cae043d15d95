"""The CPU oracle against the facts the pages and mathematics fix (no GPU)."""
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_FAST, ids=lambda f: f.__name__)
def test_pin(check):
    check(oracle)


def test_sampling_exact_marginal():
    pins.check_sampling_exact_marginal(oracle)


def test_sampling_monte_carlo_recovers_target_distribution():
    pins.check_sampling_monte_carlo(oracle)


def test_expected_tokens_monte_carlo():
    pins.check_expected_tokens(oracle)
