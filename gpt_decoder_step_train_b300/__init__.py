"""One GPT-2 decoder training step (forward, backward, AdamW) on a B300.

The compute lives in a C-ABI shared library built from ``csrc/`` for sm_103a;
``binding`` loads it with ctypes and marshals arguments.  Importing this
package loads nothing: call ``binding.lib()`` (or use ``binding.GPT2``) to load
the library, which fails loudly when it has not been built.
"""
__all__ = ["binding", "synthetic"]
