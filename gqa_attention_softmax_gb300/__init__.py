"""GQA attention with a learned per-head softmax sink, native to GB300 (sm_103a)."""
