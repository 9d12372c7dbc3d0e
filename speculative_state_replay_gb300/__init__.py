"""GB300 (sm_103a) ReplaySSM checkpointing selective-state-update.

The op lives in librssm.so (C ABI, include/rssm.h); `api` is its thin torch
binding and `workloads` the seeded synthetic decode inputs.  Importing the
package does not load the library; the first call does, and raises if the
library has not been built (there is no fallback path).
"""
from . import workloads  # noqa: F401

__all__ = ["api", "workloads"]
