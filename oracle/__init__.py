"""CPU oracle for the fused MLA decode query projection (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path never does.
"""

from .mlaqp_oracle import (  # noqa: F401
    E4M3_MAX,
    LATENT_DIM,
    MX_BLOCK,
    NOPE_DIM,
    V_HEAD_DIM,
    OUT_DIM,
    ROPE_DIM,
    algorithmic_bytes,
    assemble,
    bf16_to_f32,
    bf16_to_f64,
    decode_weight,
    e4m3_ordinal,
    e4m3_to_f64,
    e8m0_to_f64,
    f32_to_e4m3_satfinite,
    f64_to_bf16_rne,
    mla_query,
    mla_v_up,
    project,
    v_up_algorithmic_bytes,
    write_workspace,
)
