"""Batch-invariant selected-token log-probabilities on GB300 (sm_103a)."""
