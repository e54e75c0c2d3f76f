"""StreamBP LM head on GB300: sequence-chunked, exact forward + backward of the
language-model head (SFT cross-entropy, GRPO/PPO-clip, two-pass DPO), computed by
hand-written sm_103a CUDA kernels behind a C-ABI library (``libsbp.so``).

``memory_efficient_exact_gb300.sbp`` is the Python binding (argument marshalling
only); importing it loads the library and fails loudly if it was not built.
"""
__all__ = ["sbp", "inputs"]
