"""GB300-native LoongTrain 2D-Attention ring step (head-parallel x context-parallel).

The compute runs in the C-ABI library ``libloong_attn.so`` built from
``csrc/``; this package only marshals arguments to it (see ``ops``).  Importing
the package does not load the library; the first call does, and raises if the
library is missing.
"""
from .inputs import WORKLOADS, Workload, make_inputs  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_inputs"]
