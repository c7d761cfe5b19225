"""CPU oracle of the GPT-2 training step: test infrastructure, never on the product path."""
