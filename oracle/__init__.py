"""fp64 CPU oracle (test infrastructure only; see armt_oracle's docstring)."""
