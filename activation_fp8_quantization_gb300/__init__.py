"""Fused SwiGLU + MoE top-k weight + FP8/FP4 activation cast for GB300 (sm_103a)."""
