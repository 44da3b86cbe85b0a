"""GB300 (sm_103a) GPT-2-style forward pass and next-token cross-entropy.

The compute path is the CUDA library built from ``csrc/`` (see ``build.py``);
``binding`` is its thin ctypes binding. Importing this package loads nothing:
call ``binding.load()`` (or construct ``binding.GPTModel``) once the library is built.
"""
from . import build as _build  # noqa: F401

__all__ = ["binding", "build"]
