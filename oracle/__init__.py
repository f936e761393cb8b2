"""Test infrastructure: the FP64 CPU oracle.  See ``lbq_oracle`` for scope and rules."""
