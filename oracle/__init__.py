"""CPU reference oracle (test infrastructure only; see dspark_oracle.py)."""
