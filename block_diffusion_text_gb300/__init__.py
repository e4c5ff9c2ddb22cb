"""GB300-native block-diffusion denoising step.

The compute path is the C-ABI library built from ``csrc/`` (see ``dg.py`` for
the Python binding).  Importing this package loads nothing; ``dg.load()``
loads the library and fails loudly if it has not been built.
"""
