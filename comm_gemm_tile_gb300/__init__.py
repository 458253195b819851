"""Placeholder; replaced by the binding module."""
