"""Clef JointSchemaHead forward pass on GB300: a C-ABI CUDA library and its binding.

``binding`` exposes the C entry points (ctypes); ``head`` adds torch-allocated
device buffers around them; ``build`` compiles the library in-tree for sm_103a.
"""
from . import binding
from .binding import ClefError, Schema, load

__all__ = ["binding", "ClefError", "Schema", "load"]
