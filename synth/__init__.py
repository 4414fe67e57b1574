"""Seeded synthetic workloads shared by the tests and the benchmark."""
from .workloads import *  # noqa: F401,F403
from .workloads import (ALL_CONFIGS, CHAIN_CONFIGS, ChainConfig, TreeConfig, TreeSampleConfig, make_chain_inputs,
                        make_tree_inputs, make_tree_sample_inputs, make_d2t, to_bf16_bits, bf16_bits_to_f32, rng)
