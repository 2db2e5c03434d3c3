"""libbeamnorm: the fused tensor-parallel all-reduce epilogue on one GB300.

Placeholder while the binding is written.
"""
