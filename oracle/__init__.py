"""fp64 CPU oracle: test infrastructure only (see slp_oracle.py's header)."""
