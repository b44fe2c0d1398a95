"""CPU oracle (test infrastructure only; see qcf_oracle's header)."""
