"""CPU oracle (test infrastructure only; see oracle/encoder.py)."""
