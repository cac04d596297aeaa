"""Exact tiled attention (forward + backward) for GB300 / sm_103a."""
