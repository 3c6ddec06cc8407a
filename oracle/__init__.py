"""CPU oracle: test infrastructure only (tests, smoke check, bench baseline)."""
