"""Plain CPU oracle of the ZeRO step (test infrastructure; see zero_oracle)."""
