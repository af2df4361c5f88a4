"""GRPO / entropy / selective-log-softmax row pass over LM-head logits, for GB300 (sm_103a)."""
