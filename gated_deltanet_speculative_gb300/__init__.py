"""GB300-native gated-DeltaNet speculative verify path (placeholder until the binding lands)."""
from . import synth  # noqa: F401
