"""GB300-native fused MLA decode query projection and assembly."""
__version__ = "0.1.0"
