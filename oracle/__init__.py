"""Float64 CPU oracle (test infrastructure only; see moe_oracle.py)."""
