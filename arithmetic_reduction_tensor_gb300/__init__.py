"""Tensor-core and fixed-order sum reduction for GB300 (binding placeholder)."""
