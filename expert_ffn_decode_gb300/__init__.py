"""Routed MoE-FFN step (sigmoid router, top-k, Q4_0/Q4_1 SwiGLU experts) on GB300."""
