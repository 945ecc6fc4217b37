"""fp64 CPU oracle for the Megatron tensor-parallel transformer layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``, never by the library.  See
``oracle/layer.py`` for what it computes and which passages it follows.
"""
from . import decode, fp8, philox
from .layer import (LN_EPS, ReductionCounter, attention_head_bwd, attention_head_fwd,
                    causal_mask, f_allreduce, g_allreduce, gelu, gelu_grad, layer_bwd,
                    layer_bwd_partitioned, layer_flops, layer_fwd, layer_fwd_partitioned,
                    layernorm_bwd, layernorm_fwd, multihead_bwd, multihead_fwd,
                    shard_ranges, split_qkv_columns, gemm_partitioned,
                    layer_fwd_post_ln, layer_bwd_post_ln, layer_fwd_post_ln_partitioned)
