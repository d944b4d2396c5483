"""Seeded synthetic inputs for the FP8 indexer logits (decode and prefill).

This package is shared by the tests, the smoke check and the benchmark.  It
draws random numbers and lays them out in the library's input formats; it
contains none of the logits arithmetic.
"""
from .synth import (  # noqa: F401
    CONFIGS,
    DecodeCase,
    PagedPrefillCase,
    PrefillCase,
    decode_case,
    e4m3_codes,
    make_config,
    paged_prefill_case,
    prefill_case,
    prefill_windows,
)
