"""CPU oracle for W4A16 RTN quantization and GEMM.  Test infrastructure only:
see ``w4a16_oracle`` for what it computes and which passages it follows."""

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
    pack_codes,
    quantize,
    quantize_f32,
    scales_f32,
    tiled_bytes,
    to_tile_layout,
    unpack_codes,
)
