"""Float64 CPU oracle for the tensor-parallel MLP (test infrastructure only).

Only tests/, the package entry file's smoke() and the benchmark's CPU-baseline
leg may import this package. The CUDA library never does.
"""

from .tpmlp_oracle import (  # noqa: F401
    gelu,
    gelu_grad,
    shard_mlp,
    mlp,
    shard_partial,
    shard_partial_rows,
    tp_mlp,
    tp_mlp_rows,
    tp_mlp_backward,
    tp_mlp_backward_dx_rows,
    grad_A_cols,
    grad_B_rows,
    LN_EPS,
    layer_norm,
    block_mlp,
    block_mlp_rows,
    layer_norm_backward,
    block_mlp_backward,
    block_mlp_backward_dx_rows,
    split_rows,
    all_gather,
    reduce_scatter,
    tp_mlp_sp,
    tp_mlp_sp_backward,
    softmax_rows,
    attention_core,
    mha,
    shard_attention,
    attn_shard_partial,
    tp_attention,
    tp_attention_rows,
)
