"""GB300-native ring attention (context parallelism) hot path."""
from . import accounting  # noqa: F401
