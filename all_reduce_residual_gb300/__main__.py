"""python -m all_reduce_residual_gb300: build libarf.so for sm_103a."""
from .build import build

print(build(force=True))
