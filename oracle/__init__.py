"""fp64 CPU oracle for the per-layer DP-SGD clipping path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference arm may import this package.  The product
path (the CUDA library and its Python binding) never imports, links or calls
anything here, and nothing here imports the product path.
"""
from .dpclip_oracle import *  # noqa: F401,F403
from .dpclip_oracle import __all__  # noqa: F401
