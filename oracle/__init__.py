"""CPU oracle for W4A16 RTN quantization and GEMM, the seeded
stochastic-rounding quantize mode, the INT8 weight-only (W8A16) scheme and
the FP4 weight-only schemes (MXFP4, NVFP4).  Test infrastructure only: see
``w4a16_oracle``, ``stochastic``, ``w8a16_oracle`` and ``fp4_oracle`` for what
they compute and which passages they follow."""

from .w4a16_oracle import (  # noqa: F401
    GROUP,
    TILE_BYTES,
    TILE_ROWS,
    QMAX,
    QMIN,
    act_bits_to_f32,
    bf16_bits_to_f32,
    dequantize,
    f16_bits_to_f32,
    from_tile_layout,
    gemm,
    gemm_swiglu,
    pack_codes,
    quantize,
    quantize_f32,
    scales_f32,
    swiglu,
    tiled_bytes,
    to_tile_layout,
    unpack_codes,
)
from .stochastic import (  # noqa: F401
    philox4x32_10,
    quantize_sr,
    quantize_sr_f32,
    stochastic_code,
    uniform_at,
    uniform_block,
)
from .w8a16_oracle import (  # noqa: F401
    Q8MAX,
    Q8MIN,
    dequantize8,
    from_tile_layout8,
    gemm8,
    quantize8,
    quantize8_f32,
    tiled8_bytes,
    to_tile_layout8,
)
from .fp4_oracle import (  # noqa: F401
    dequantize_mxfp4,
    dequantize_nvfp4,
    e2m1_decode,
    e2m1_encode,
    e4m3_decode,
    e4m3_encode,
    gemm_fp4,
    mx_exponent,
    pack_codes_fp4,
    quantize_mxfp4_f32,
    quantize_nvfp4_f32,
    unpack_codes_fp4,
)
