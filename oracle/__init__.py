"""CPU oracle of the FlashMap block-draft step (test infrastructure only)."""
