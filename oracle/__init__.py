"""CPU oracle for the VSA forward: test infrastructure only (see vsa_oracle)."""
