"""Sparsely-Gated Mixture-of-Experts layer forward pass for B300 (sm_103a)."""
