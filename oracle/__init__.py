"""CPU oracle for the DeepSeekMoE layer forward (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this package. It
shares no code with the CUDA library, which never imports it. See ``moe_oracle.c`` for the
definitions it follows and the citations.
"""
from .oracle import (OracleCfg, backward, balance_stats, build, expert_ffn, forward_tokens,
                     group_range, layer_forward, lib_path, permute, route, threads)

__all__ = ["OracleCfg", "backward", "balance_stats", "build", "expert_ffn", "forward_tokens",
           "group_range", "layer_forward", "lib_path", "permute", "route", "threads"]
