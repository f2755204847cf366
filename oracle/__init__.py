"""CPU oracle of the USAF sparse MoE fine-tuning hot path (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this package. The
product library (sparse_moe_fine_gb300) never imports it and shares no code with it.
"""
from .usaf_oracle import *  # noqa: F401,F403
