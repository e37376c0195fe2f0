"""CPU oracle of the rotated 3-bit KV cache (test infrastructure only)."""
