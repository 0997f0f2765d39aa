"""Test-side glue: the oracle's adapters for the library's packed tensors."""
from oracle.packed import expert_fn, f64, run_oracle  # noqa: F401
