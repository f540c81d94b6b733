"""Frame-aligned block-sparse attention with a norm-bound softmax, for B300 (sm_103a)."""
