"""GB300-native Qwen3-style speech-LLM decoder: C-ABI library + Python binding.

Importing the package is cheap; the CUDA library is loaded by
``speech_decoder_gb300.binding`` on first use.
"""
__all__ = ["synth"]
