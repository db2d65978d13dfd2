"""CPU oracle for the KPool-DSA forward (test infrastructure only; see kpool_oracle)."""
