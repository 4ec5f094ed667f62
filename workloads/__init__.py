"""Seeded synthetic input generators shared by the tests, the benchmark and
the smoke check.  Holds no step of the verification method itself."""
from .philox import philox4x32_10, u32_to_unit_float, uniform_grid  # noqa: F401
from .configs import (SPECS, TOY_P, TOY_Q, as_f32, bf16_bits_to_f32,  # noqa: F401
                      bytes_all_rows, bytes_needed, categorical_draws,
                      f32_to_bf16_bits, make_device, make_geometric, make_host,
                      make_pair_batch, make_spec_host, make_toy)
from .trees import full_tree, make_tree_host, make_tree_pair  # noqa: F401,E402
