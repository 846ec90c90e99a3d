"""CPU oracle (test infrastructure only; the library never imports it)."""
