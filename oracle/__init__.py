"""CPU oracle for the GPT-2 training step: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct numpy implementation of one mixed-precision
GPT-2 training step (forward, backward, AdamW), written from the method that
llm.c's "State of the Union [May 3, 2024]" describes. It shares no code with
the CUDA library. Only the test suite, the smoke check and the benchmark's CPU
baseline may import it; the library never does.
"""
from .gpt2_ref import *  # noqa: F401,F403
