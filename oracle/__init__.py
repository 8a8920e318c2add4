"""fp64 CPU oracle (test infrastructure only; see srft_oracle's header)."""
