"""B300-native GPT-2 training step (forward, backward, AdamW) behind a C ABI."""
