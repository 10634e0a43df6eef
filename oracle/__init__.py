"""CPU oracle for the collective datapath: test infrastructure, not product code.

This package states, as plainly as numpy allows, what every collective of the
datapath computes.  It exists so that the CUDA path can be checked against
something written independently of it.  Only the test-suite, the package
smoke check and the benchmark's CPU-baseline / reference arm may import it;
the library itself never calls it, and no code is shared between the two.
"""

from .collectives import (  # noqa: F401
    bf16_bits_to_f32,
    f32_to_bf16_rne,
    fold_sum,
    all_reduce,
    reduce_scatter,
    reduce_scatter_v,
    all_gather,
    all_to_all,
    all_gather_v,
    all_to_all_v,
)
