"""GB300-native batched verify step of greedy (lossless) speculative decoding.

The compute lives in libspecverify.so (hand-written CUDA for sm_103a, C ABI declared in
include/spec_verify.h); this package is its thin Python binding plus the seeded input
generators used by the tests and the benchmark.
"""
from ._binding import (KMAX, SpecError, lib, make_kv_desc, spec_accept, spec_accept_sample,
                       spec_accept_sample_workspace, spec_accept_stop, spec_accept_tree, spec_h_gather,
                       spec_h_scatter, spec_kv_append, spec_kv_compact, spec_kv_desc, spec_kv_write_rows,
                       spec_lmhead_argmax, spec_lmhead_argmax_static, spec_lmhead_logits, spec_lmhead_workspace,
                       spec_mtp_input, spec_mtp_input_workspace, spec_verify_attn, spec_verify_attn_tree,
                       spec_verify_attn_workspace, strerror, version)

__all__ = ["KMAX", "SpecError", "lib", "make_kv_desc", "spec_accept", "spec_accept_sample",
           "spec_accept_sample_workspace", "spec_accept_stop", "spec_accept_tree", "spec_h_gather", "spec_h_scatter",
           "spec_kv_append", "spec_kv_compact", "spec_kv_desc", "spec_kv_write_rows", "spec_lmhead_argmax",
           "spec_lmhead_argmax_static", "spec_lmhead_logits", "spec_lmhead_workspace", "spec_mtp_input",
           "spec_mtp_input_workspace", "spec_verify_attn", "spec_verify_attn_tree", "spec_verify_attn_workspace",
           "strerror", "version"]
